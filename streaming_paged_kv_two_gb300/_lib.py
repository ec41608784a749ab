"""ctypes binding of libspk (include/spk.h): argument marshalling only.

Every call maps one-to-one onto a C entry point; all work happens in the library
and its CUDA kernels.  Device buffers may be passed as integers (device
addresses) or as objects with a ``data_ptr()`` method (e.g. torch tensors); CUDA
streams as integers (cudaStream_t values) or objects with a ``cuda_stream``
attribute.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspk.so")

SPK_OK = 0
SPK_ERR_INVALID_ARG = 1
SPK_ERR_OUT_OF_PATCH_PAGES = 2
SPK_ERR_OUT_OF_SPECIAL_PAGES = 3
SPK_ERR_BAD_STATE = 4
SPK_ERR_CUDA = 5
SPK_ERR_DEVICE_TIMEOUT = 6
SPK_BF16 = 0
SPK_F32 = 1

STATUS_NAMES = {
    SPK_OK: "SPK_OK", SPK_ERR_INVALID_ARG: "SPK_ERR_INVALID_ARG",
    SPK_ERR_OUT_OF_PATCH_PAGES: "SPK_ERR_OUT_OF_PATCH_PAGES",
    SPK_ERR_OUT_OF_SPECIAL_PAGES: "SPK_ERR_OUT_OF_SPECIAL_PAGES",
    SPK_ERR_BAD_STATE: "SPK_ERR_BAD_STATE", SPK_ERR_CUDA: "SPK_ERR_CUDA",
    SPK_ERR_DEVICE_TIMEOUT: "SPK_ERR_DEVICE_TIMEOUT",
}


class SpkError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


class spk_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_blocks", "num_streams", "num_heads", "head_dim", "page_size", "patches_per_frame",
        "specials_per_frame", "scale_frames", "sliding_window", "max_patch_pages", "max_special_pages",
        "dtype", "splits_per_stream", "max_query_frames")] + [
        ("patch_page_order", ctypes.POINTER(ctypes.c_int32)),
        ("special_page_order", ctypes.POINTER(ctypes.c_int32))]


class spk_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "frame_count", "scale_pages", "live_pages", "free_pages", "special_tokens")]


class spk_rope(ctypes.Structure):
    _fields_ = [("sections", ctypes.c_int32 * 3), ("reserved", ctypes.c_int32), ("theta", ctypes.c_double)]


class spk_plan_info(ctypes.Structure):
    _fields_ = [("num_chunks", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("merge_needed", ctypes.c_int32), ("visible_tokens", ctypes.c_int64),
                ("split_scratch_bytes", ctypes.c_int64), ("static_scratch_capacity", ctypes.c_int64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libspk.so is not built ({LIB_PATH}); run python streaming_paged_kv_two_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    pi32 = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "spk_last_error": (ctypes.c_char_p, []),
        "spk_required_bytes": (I32, [ctypes.POINTER(spk_config), ctypes.POINTER(SZ), ctypes.POINTER(SZ)]),
        "spk_create_cache": (I32, [ctypes.POINTER(spk_config), ctypes.POINTER(P), ctypes.POINTER(P)]),
        "spk_destroy_cache": (I32, [P]),
        "spk_reset": (I32, [P]),
        "spk_append_frame": (I32, [P, I32, I32, P, P, P]),
        "spk_append_frame_rope": (I32, [P, I32, I32, P, P, P, P, P, ctypes.POINTER(spk_rope), P]),
        "spk_evict_frames": (I32, [P, I32]),
        "spk_plan": (I32, [P, P, P]),
        "spk_set_defer_eviction": (I32, [P, I32, I32]),
        "spk_rollback_frame": (I32, [P, I32]),
        "spk_plan_queries": (I32, [P, I32, P, P]),
        "spk_run_attention": (I32, [P, I32, P, P, P, P]),
        "spk_read_kv": (I32, [P, I32, I32, P, P]),
        "spk_get_plan_host": (I32, [P, pi32, ctypes.c_int32, pi32, pi32, pi32, pi32, pi32]),
        "spk_get_plan_info": (I32, [P, ctypes.POINTER(spk_plan_info)]),
        "spk_get_frame_targets": (I32, [P, I32, pi32, pi32, pi32]),
        "spk_get_stats": (I32, [P, I32, ctypes.POINTER(spk_stats)]),
        "spk_read_device_status": (I32, [P, P, pi32]),
        "spk_selftest_wait_timeout": (I32, [P, I64, P]),
        "spk_run_attention_static_scratch": (I32, [P, I32, P, P, P, P]),
        "spk_debug_dump_scores": (I32, [P, I32, P, P, P, P]),
        "spk_debug_trace_attention": (I32, [P, I32, P, P, P, P, ctypes.c_int32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def last_error() -> str:
    return lib.spk_last_error().decode()


def _check(rc: int):
    if rc != SPK_OK:
        raise SpkError(rc, last_error())


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def make_config(*, num_blocks, num_streams, num_heads, head_dim, page_size, patches_per_frame,
                specials_per_frame, scale_frames, sliding_window, max_patch_pages, max_special_pages,
                dtype=SPK_BF16, splits_per_stream=0, patch_page_order=None, special_page_order=None,
                max_query_frames=0):
    """Return (spk_config, keepalive) with the optional page orders as int32 host arrays."""
    c = spk_config(num_blocks, num_streams, num_heads, head_dim, page_size, patches_per_frame,
                   specials_per_frame, scale_frames, sliding_window, max_patch_pages, max_special_pages,
                   dtype, splits_per_stream, max_query_frames)
    keep = []
    for field, arr in (("patch_page_order", patch_page_order), ("special_page_order", special_page_order)):
        if arr is not None:
            buf = (ctypes.c_int32 * len(arr))(*[int(v) for v in arr])
            keep.append(buf)
            setattr(c, field, ctypes.cast(buf, ctypes.POINTER(ctypes.c_int32)))
    return c, keep


def required_bytes(cfg: spk_config):
    pool, ws = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.spk_required_bytes(ctypes.byref(cfg), ctypes.byref(pool), ctypes.byref(ws)))
    return pool.value, ws.value


def read_device_status(workspace, cuda_stream=None) -> int:
    """Returns the raw device status code (0 = no timeout); raises SpkError on a recorded timeout."""
    code = ctypes.c_int32()
    rc = lib.spk_read_device_status(_ptr(workspace), _stream(cuda_stream), ctypes.byref(code))
    if rc not in (SPK_OK, SPK_ERR_DEVICE_TIMEOUT):
        _check(rc)
    if rc == SPK_ERR_DEVICE_TIMEOUT:
        raise SpkError(rc, last_error())
    return code.value


def selftest_wait_timeout(workspace, limit_ns: int, cuda_stream=None):
    _check(lib.spk_selftest_wait_timeout(_ptr(workspace), int(limit_ns), _stream(cuda_stream)))


class Cache:
    """One spk_cache.  Methods are the C entry points with the cache argument bound."""

    def __init__(self, cfg: spk_config, pools=None, keepalive=None):
        self.cfg = cfg
        self._keep = keepalive
        self._h = ctypes.c_void_p()
        if pools is None:
            arr = None
        else:
            ptrs = [_ptr(p) for p in pools]
            arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        _check(lib.spk_create_cache(ctypes.byref(cfg), arr, ctypes.byref(self._h)))
        self.B = cfg.num_streams
        self.S = cfg.specials_per_frame

    def close(self):
        if self._h:
            lib.spk_destroy_cache(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        _check(lib.spk_reset(self._h))

    def append_frame(self, stream: int, block: int, k=None, v=None, cuda_stream=None):
        _check(lib.spk_append_frame(self._h, stream, block, _ptr(k), _ptr(v), _stream(cuda_stream)))

    def append_frame_rope(self, stream: int, block: int, k=None, v=None, q=None, q_out=None, positions=None,
                          sections=(0, 0, 0), theta: float = 10000.0, cuda_stream=None):
        """append_frame with q and k turned by the 3-D rotary embedding (k into the cache,
        q into q_out, which may be q itself).  positions: device int32 [T, 3]."""
        rope = spk_rope((ctypes.c_int32 * 3)(*sections), 0, float(theta))
        _check(lib.spk_append_frame_rope(self._h, stream, block, _ptr(k), _ptr(v), _ptr(q), _ptr(q_out),
                                         _ptr(positions), ctypes.byref(rope), _stream(cuda_stream)))

    def evict_frames(self, stream: int):
        _check(lib.spk_evict_frames(self._h, stream))

    def plan(self, workspace=None, cuda_stream=None):
        _check(lib.spk_plan(self._h, _ptr(workspace), _stream(cuda_stream)))

    def set_defer_eviction(self, stream: int, on: bool):
        _check(lib.spk_set_defer_eviction(self._h, stream, 1 if on else 0))

    def rollback_frame(self, stream: int):
        _check(lib.spk_rollback_frame(self._h, stream))

    def plan_queries(self, query_frames: int, workspace=None, cuda_stream=None):
        _check(lib.spk_plan_queries(self._h, int(query_frames), _ptr(workspace), _stream(cuda_stream)))

    def run_attention(self, block: int, q, out, workspace, cuda_stream=None):
        _check(lib.spk_run_attention(self._h, block, _ptr(q), _ptr(out), _ptr(workspace), _stream(cuda_stream)))

    def run_attention_static_scratch(self, block: int, q, out, workspace, cuda_stream=None):
        """spk_run_attention with the split partials in the library's static device array."""
        _check(lib.spk_run_attention_static_scratch(self._h, block, _ptr(q), _ptr(out), _ptr(workspace),
                                                    _stream(cuda_stream)))

    def debug_dump_scores(self, block: int, q, dst, workspace, cuda_stream=None):
        _check(lib.spk_debug_dump_scores(self._h, block, _ptr(q), _ptr(dst), _ptr(workspace), _stream(cuda_stream)))

    def debug_trace_attention(self, block: int, q, out, workspace, trace, capacity: int, cuda_stream=None):
        _check(lib.spk_debug_trace_attention(self._h, block, _ptr(q), _ptr(out), _ptr(workspace), _ptr(trace),
                                             int(capacity), _stream(cuda_stream)))

    def read_kv(self, block: int, page_id: int, dst, cuda_stream=None):
        _check(lib.spk_read_kv(self._h, block, page_id, _ptr(dst), _stream(cuda_stream)))

    def get_plan_host(self):
        nnz = ctypes.c_int32()
        B = self.B
        kv = (ctypes.c_int32 * (B + 1))()
        lpl = (ctypes.c_int32 * B)()
        npp = (ctypes.c_int32 * B)()
        qo = (ctypes.c_int32 * (B + 1))()
        _check(lib.spk_get_plan_host(self._h, None, 0, kv, lpl, npp, qo, ctypes.byref(nnz)))
        idx = (ctypes.c_int32 * max(nnz.value, 1))()
        _check(lib.spk_get_plan_host(self._h, idx, nnz.value, None, None, None, None, ctypes.byref(nnz)))
        return {"indices": list(idx[:nnz.value]), "kv_indptr": list(kv), "last_page_len": list(lpl),
                "num_patch_pages": list(npp), "qo_indptr": list(qo)}

    def get_plan_info(self) -> dict:
        info = spk_plan_info()
        _check(lib.spk_get_plan_info(self._h, ctypes.byref(info)))
        return {f: getattr(info, f) for f, _ in spk_plan_info._fields_}

    def get_frame_targets(self, stream: int):
        pp = ctypes.c_int32()
        sp = (ctypes.c_int32 * self.S)()
        ss = (ctypes.c_int32 * self.S)()
        _check(lib.spk_get_frame_targets(self._h, stream, ctypes.byref(pp), sp, ss))
        return pp.value, list(zip(list(sp), list(ss)))

    def get_stats(self, stream: int) -> dict:
        st = spk_stats()
        _check(lib.spk_get_stats(self._h, stream, ctypes.byref(st)))
        return {f: getattr(st, f) for f, _ in spk_stats._fields_}
