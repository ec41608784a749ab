"""Coefficients of the cubic that approximates 2^f on [-1/2, 1/2] for the attention
kernel's software exp2 (range reduction 2^x = 2^n * 2^f, n = round(x)).

Method: minimax polynomial under relative error, found with the Remez exchange
algorithm (equioscillation on degree + 2 reference points).  Run this file to
reproduce the constants used in spk_attn_tc.cu:

    python streaming_paged_kv_two_gb300/csrc/exp2_poly_coeffs.py
"""
import numpy as np

DEG = 3
A, B = -0.5, 0.5


def remez(deg=DEG, iters=30):
    n = deg + 2
    k = np.arange(n)
    x = 0.5 * (A + B) + 0.5 * (B - A) * np.cos(np.pi * k[::-1] / (n - 1))  # Chebyshev extrema
    grid = np.linspace(A, B, 200001)
    for _ in range(iters):
        # solve sum c_i x^i - 2^x = (-1)^j E 2^x   (relative error E)
        f = np.exp2(x)
        M = np.zeros((n, n))
        for i in range(deg + 1):
            M[:, i] = x ** i
        M[:, deg + 1] = ((-1.0) ** k) * f
        sol = np.linalg.solve(M, f)
        c, E = sol[:deg + 1], sol[deg + 1]
        err = (np.polyval(c[::-1], grid) - np.exp2(grid)) / np.exp2(grid)
        # new reference: extrema of the error, one per sign change segment
        sign = np.sign(err)
        idx = np.where(np.diff(sign) != 0)[0]
        bounds = np.concatenate([[0], idx + 1, [len(grid)]])
        ext = [b0 + np.argmax(np.abs(err[b0:b1])) for b0, b1 in zip(bounds[:-1], bounds[1:]) if b1 > b0]
        if len(ext) != n:
            break
        x = grid[ext]
    return c, np.max(np.abs(err))


if __name__ == "__main__":
    c, e = remez()
    np.set_printoptions(precision=10)
    print("coefficients c0..c3:", [float(np.float32(v)) for v in c])
    print("max relative error on [-1/2, 1/2]:", e)
