"""3-D rotary position embedding of q and k before they enter the cache, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title, section):

* "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction",
  "3D RoPE Position Encoding": a three-dimensional rotary embedding is applied to
  the query and key tensors of each frame before they are cached; the positions
  carry the global frame index.
* same page, FAQ "How is temporal information preserved in the KV cache?": the
  positions are baked into q and k before the append, so attention needs no
  position lookup.

The pages name the embedding but do not write it out.  The reading taken here is
the rotary embedding of Su et al., "RoFormer: Enhanced Transformer with Rotary
Position Embedding" (2021), applied per position axis:

* a token has an integer position per axis (t, h, w);
* the head dimension is taken as D/2 adjacent pairs (x[2i], x[2i+1]); the first
  sections[0] pairs follow axis t, the next sections[1] axis h, the next
  sections[2] axis w, and any pairs after those are left as they are;
* pair j of an axis section with n pairs turns by the angle
  position_axis * theta**(-j / n) (RoFormer's theta_j = base**(-2j/d) for the
  2n dimensions of that section);
* turning a pair by angle a is the plane rotation
  (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a).

V is not rotated.  Positions, sections and theta are inputs: the pages leave
them to the model.
"""
from __future__ import annotations

import numpy as np


def pair_angles(positions, sections, theta: float, head_dim: int) -> np.ndarray:
    """Rotation angle of every (token, pair): float64 [T, head_dim // 2].

    positions: integer [T, 3] (t, h, w per token).  Pairs beyond the sections
    get angle 0.
    """
    pos = np.asarray(positions, dtype=np.int64)
    T = pos.shape[0]
    npairs = head_dim // 2
    if sum(sections) > npairs or min(sections) < 0:
        raise ValueError("sections must be non-negative and fit in head_dim/2 pairs")
    ang = np.zeros((T, npairs), dtype=np.float64)
    first = 0
    for axis, n in enumerate(sections):
        for j in range(n):
            freq = float(theta) ** (-j / n)
            ang[:, first + j] = pos[:, axis].astype(np.float64) * freq
        first += n
    return ang


def rotate(x, positions, sections, theta: float) -> np.ndarray:
    """Rotary-embedded copy of x [T, H, D] (float64); every head turns alike."""
    x = np.asarray(x, dtype=np.float64)
    T, H, D = x.shape
    ang = pair_angles(positions, sections, theta, D)  # [T, D/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x0 = x[:, :, 0::2]
    x1 = x[:, :, 1::2]
    out = np.empty_like(x)
    out[:, :, 0::2] = x0 * c - x1 * s
    out[:, :, 1::2] = x0 * s + x1 * c
    return out
