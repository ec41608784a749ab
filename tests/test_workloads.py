"""The seeded input generator's rotary positions and sections have the stated shape
(they are inputs to both the oracle and the GPU path, so they carry no arithmetic of
the method)."""
from __future__ import annotations

import numpy as np
import pytest

import workloads as wl


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_frame_positions_cover_the_patch_grid(name):
    w = wl.CONFIGS[name]
    rows, cols = wl.patch_grid(w)
    assert rows * cols == w.patches_per_frame and rows <= cols
    pos = wl.frame_positions(w, 7, 10_000)
    assert pos.shape == (w.tokens_per_frame, 3) and pos.dtype == np.int32
    assert (pos[:, 0] == 10_007).all()
    P = w.patches_per_frame
    cells = {(int(h), int(x)) for h, x in pos[:P, 1:]}
    assert cells == {(h, x) for h in range(rows) for x in range(cols)}
    assert (pos[P:, 1:] == -1).all()


@pytest.mark.parametrize("D", [64, 128])
def test_rope_sections_fill_the_pairs(D):
    w = wl.CONFIGS["steady_state_10k"].replace(head_dim=D)
    t, h, x = wl.rope_sections(w)
    assert t + h + x == D // 2 and h == x and t >= h > 0
