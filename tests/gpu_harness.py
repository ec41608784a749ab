"""GPU-side test glue: device buffers from torch, inputs from `workloads`, calls through
the C ABI binding.  Imported only by GPU tests (and the smoke check)."""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl
import streaming_paged_kv_two_gb300 as spk
from workload_device import spk_config_for, to_device  # noqa: F401  (re-exported for the tests)

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-4


def to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return wl.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.double().cpu().numpy()


class Harness:
    """Pools, workspace and an spk cache on cuda:0 for one workload."""

    def __init__(self, w: wl.Workload, splits: int = 0, max_query_frames: int = 0):
        self.w = w
        self.cfg, self.keep = spk_config_for(w, splits, max_query_frames)
        pool_bytes, ws_bytes = spk.required_bytes(self.cfg)
        self.pools = [torch.empty(pool_bytes, dtype=torch.uint8, device="cuda") for _ in range(w.num_blocks)]
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        self.cache = spk.Cache(self.cfg, self.pools, self.keep)
        self.stream = torch.cuda.current_stream()
        self.tdtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self._hold = []

    def append(self, stream: int, block: int, k: np.ndarray, v: np.ndarray):
        kd, vd = to_device(k, self.w.dtype), to_device(v, self.w.dtype)
        self._hold.append((kd, vd))
        self.cache.append_frame(stream, block, kd, vd, self.stream)

    def append_device(self, stream: int, block: int, kd: torch.Tensor, vd: torch.Tensor):
        self.cache.append_frame(stream, block, kd, vd, self.stream)

    def plan(self):
        self.cache.plan(self.ws, self.stream)

    def plan_queries(self, query_frames: int):
        self.cache.plan_queries(query_frames, self.ws, self.stream)

    def run(self, block: int, q: np.ndarray) -> np.ndarray:
        qd = to_device(q, self.w.dtype)
        out = torch.empty_like(qd)
        self.cache.run_attention(block, qd, out, self.ws, self.stream)
        torch.cuda.synchronize()
        self._hold.clear()
        return to_f64(out)

    def status(self) -> int:
        return spk.read_device_status(self.ws, self.stream)

    def read_page(self, block: int, page: int) -> np.ndarray:
        w = self.w
        shape = (2, w.page_size, w.num_heads, w.head_dim)
        dst = torch.empty(shape, dtype=self.tdtype, device="cuda")
        self.cache.read_kv(block, page, dst, self.stream)
        if self.tdtype == torch.bfloat16:
            return dst.view(torch.int16).cpu().numpy().view(np.uint16)
        return dst.cpu().numpy()

    def close(self):
        self.cache.close()


def check_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    err = np.abs(got - want)
    if dtype == "bf16":
        assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, \
            f"{what}: max-abs {err.max():.3e} mean-abs {err.mean():.3e}"
    else:
        assert err.max() <= F32_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    return float(err.max()), float(err.mean())
