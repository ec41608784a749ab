"""Seeded synthetic workloads for the streaming two-stream paged-KV attention path.

This module only describes workload shapes and draws seeded random inputs.  It
holds none of the method's arithmetic (no page bookkeeping, no attention), so
both the fp64 oracle and the GPU path can take their inputs from it.

The five workloads follow the shapes the pages describe for LingBot-Map's
streaming inference ("How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D
Reconstruction", sections "Physical Memory Layout" and "Initializing the Cache
Manager": 256 patch + 6 special tokens per frame, 16 heads of 64, 8 scale
frames, a 64-frame window, headroom of 16 pages).  The pages print no activation
statistics, so values are normal draws with a per-workload scale; batched4_d128 adds
a per-(stream, head) scale drawn from U[0.25, 2].

Values are drawn in float32 and, for bf16 workloads, rounded to bfloat16
(round-to-nearest-even) here, so that every consumer sees the same stored bits.
bf16 values are returned as uint16 bit patterns; `bf16_bits_to_f64` and
`bf16_bits_to_f32` widen them exactly.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_blocks: int          # L, transformer blocks (one pool each)
    num_streams: int         # B, independent streams batched in one launch
    num_heads: int           # H
    head_dim: int            # D
    page_size: int           # ps
    patches_per_frame: int   # P
    specials_per_frame: int  # S
    scale_frames: int        # sc
    sliding_window: int      # w
    frames: int              # frames streamed
    dtype: str               # "bf16" or "f32"
    value_scale: float       # std of q/k/v draws (ignored when per_head_scale)
    per_head_scale: bool = False   # scale q/k/v by U[0.25, 2] per (stream, head)
    shuffle_pages: bool = False    # random initial free-list order per stream
    measured_frames: int = 100     # the last frames of the stream are timed
    seed: int = 20260731
    headroom: int = 16

    @property
    def tokens_per_frame(self) -> int:
        return self.patches_per_frame + self.specials_per_frame

    @property
    def max_patch_pages(self) -> int:
        # scale + window + headroom, the sizing rule printed with the
        # manager's constructor example (max_num_frames=88 for 8 + 64 + 16)
        return self.scale_frames + self.sliding_window + self.headroom

    @property
    def max_special_pages(self) -> int:
        return -(-self.frames * self.specials_per_frame // self.page_size)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS = {w.name: w for w in (
    Workload("tiny_stream_f32", 1, 1, 4, 64, 16, 16, 2, 2, 4, 12, "f32", 1.0,
             measured_frames=12),
    Workload("lingbot_like_200", 24, 1, 16, 64, 256, 256, 6, 8, 64, 200, "bf16", 0.5),
    Workload("steady_state_10k", 24, 1, 16, 64, 256, 256, 6, 8, 64, 10000, "bf16", 0.5),
    Workload("high_res_999", 24, 1, 16, 64, 1024, 999, 6, 8, 32, 2000, "bf16", 1.0),
    Workload("batched4_d128", 12, 4, 8, 128, 256, 256, 6, 4, 128, 5000, "bf16", 1.0,
             per_head_scale=True, shuffle_pages=True),
)}


# ---------------------------------------------------------------- bf16 bits

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored values (uint16 bf16 bits or float32) to float64, exactly."""
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------- draws

_TAG_PATCH, _TAG_SPECIAL, _TAG_Q, _TAG_HEADSCALE, _TAG_ORDER = 0, 1, 2, 3, 4


def _rng(cfg: Workload, *key: int) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, *key])


def head_scales(cfg: Workload, stream: int) -> np.ndarray:
    """Per-head multiplier for one stream: U[0.25, 2] when per_head_scale, else value_scale."""
    if cfg.per_head_scale:
        return _rng(cfg, _TAG_HEADSCALE, stream).uniform(0.25, 2.0, size=cfg.num_heads).astype(np.float32)
    return np.full(cfg.num_heads, cfg.value_scale, dtype=np.float32)


def _finish(cfg: Workload, x: np.ndarray, stream: int) -> np.ndarray:
    x = x * head_scales(cfg, stream)[None, :, None]
    if cfg.dtype == "bf16":
        return f32_to_bf16_bits(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def frame_patch_kv(cfg: Workload, stream: int, block: int, frame: int):
    """(k, v) patch rows of one frame: each [P, H, D] in the stored dtype."""
    g = _rng(cfg, _TAG_PATCH, stream, block, frame)
    kv = g.standard_normal((2, cfg.patches_per_frame, cfg.num_heads, cfg.head_dim), dtype=np.float32)
    return _finish(cfg, kv[0], stream), _finish(cfg, kv[1], stream)


def frame_special_kv(cfg: Workload, stream: int, block: int, frame: int):
    """(k, v) special rows of one frame: each [S, H, D] in the stored dtype."""
    g = _rng(cfg, _TAG_SPECIAL, stream, block, frame)
    kv = g.standard_normal((2, cfg.specials_per_frame, cfg.num_heads, cfg.head_dim), dtype=np.float32)
    return _finish(cfg, kv[0], stream), _finish(cfg, kv[1], stream)


def frame_kv(cfg: Workload, stream: int, block: int, frame: int):
    """(k, v) of one frame, each [T, H, D]: rows 0..P-1 patch, rows P..T-1 special."""
    kp, vp = frame_patch_kv(cfg, stream, block, frame)
    ks, vs = frame_special_kv(cfg, stream, block, frame)
    return np.concatenate([kp, ks], axis=0), np.concatenate([vp, vs], axis=0)


def frame_q(cfg: Workload, stream: int, block: int, frame: int) -> np.ndarray:
    """Query rows of one frame, [T, H, D] in the stored dtype."""
    g = _rng(cfg, _TAG_Q, stream, block, frame)
    q = g.standard_normal((cfg.tokens_per_frame, cfg.num_heads, cfg.head_dim), dtype=np.float32)
    return _finish(cfg, q, stream)


def patch_grid(cfg: Workload):
    """(rows, cols) of the frame's patch grid: the most nearly square factorisation of P
    with rows <= cols (16 x 16 for 256 patches, 27 x 37 for 999)."""
    P = cfg.patches_per_frame
    rows = int(np.floor(np.sqrt(P)))
    while P % rows:
        rows -= 1
    return rows, P // rows


def frame_positions(cfg: Workload, frame: int, frame_offset: int = 0) -> np.ndarray:
    """Rotary positions (t, h, w) of a frame's T tokens, int32 [T, 3].

    t is the global frame index (frame + frame_offset) for every token; patch p sits
    at (p // cols, p % cols) of the patch grid; special tokens sit at (-1, -1), off
    the grid.
    """
    rows, cols = patch_grid(cfg)
    P, T = cfg.patches_per_frame, cfg.tokens_per_frame
    pos = np.empty((T, 3), dtype=np.int32)
    pos[:, 0] = frame + frame_offset
    p = np.arange(P)
    pos[:P, 1] = p // cols
    pos[:P, 2] = p % cols
    pos[P:, 1:] = -1
    return pos


def rope_sections(cfg: Workload):
    """Rotary pairs per axis (t, h, w): h and w a third of the D/2 pairs each, t the rest."""
    n = cfg.head_dim // 2
    return (n - 2 * (n // 3), n // 3, n // 3)


def page_orders(cfg: Workload):
    """Initial free-list orders as global page ids, or (None, None) for ascending.

    Stream s owns patch ids [s*MPP, (s+1)*MPP) and special ids
    [B*MPP + s*MSP, B*MPP + (s+1)*MSP).  With shuffle_pages each stream's ids
    are a seeded permutation of its own range.
    """
    if not cfg.shuffle_pages:
        return None, None
    mpp, msp, b = cfg.max_patch_pages, cfg.max_special_pages, cfg.num_streams
    patch = np.empty(b * mpp, dtype=np.int32)
    special = np.empty(b * msp, dtype=np.int32)
    for s in range(b):
        g = _rng(cfg, _TAG_ORDER, s)
        patch[s * mpp:(s + 1) * mpp] = s * mpp + g.permutation(mpp)
        special[s * msp:(s + 1) * msp] = b * mpp + s * msp + g.permutation(msp)
    return patch, special


def element_bytes(cfg: Workload) -> int:
    return 2 if cfg.dtype == "bf16" else 4


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("dataclasses", "np", "annotations")]
