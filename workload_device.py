"""Device-side glue for the seeded workloads (no method arithmetic).

The library configuration that describes a `workloads.Workload`, and host arrays of
its inputs moved to the GPU as torch tensors.  Shared by the benchmark and the GPU
tests; the oracle never imports it.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl
import streaming_paged_kv_two_gb300 as spk


def spk_config_for(w: wl.Workload, splits: int = 0, max_query_frames: int = 0):
    """spk_config (and the arrays it points into) for workload w."""
    po, so = wl.page_orders(w)
    return spk.make_config(
        num_blocks=w.num_blocks, num_streams=w.num_streams, num_heads=w.num_heads, head_dim=w.head_dim,
        page_size=w.page_size, patches_per_frame=w.patches_per_frame, specials_per_frame=w.specials_per_frame,
        scale_frames=w.scale_frames, sliding_window=w.sliding_window, max_patch_pages=w.max_patch_pages,
        max_special_pages=w.max_special_pages, dtype=spk.SPK_BF16 if w.dtype == "bf16" else spk.SPK_F32,
        splits_per_stream=splits, max_query_frames=max_query_frames,
        patch_page_order=None if po is None else po.tolist(),
        special_page_order=None if so is None else so.tolist())


def to_device(x: np.ndarray, dtype: str) -> torch.Tensor:
    """A host array of the workload's values (bf16 bit patterns or fp32) as a CUDA tensor."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
