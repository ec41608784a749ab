"""Streaming two-stream paged-KV attention for GB300 (sm_103a).

The compute path is libspk.so (C ABI in include/spk.h): host C++ page
bookkeeping and planning, and hand-written CUDA kernels for append, tcgen05
paged attention and the log-sum-exp merge.  This package is its ctypes binding;
importing it fails loudly when the library has not been built.
"""
from ._lib import (  # noqa: F401
    Cache,
    LIB_PATH,
    SPK_BF16,
    SPK_ERR_BAD_STATE,
    SPK_ERR_CUDA,
    SPK_ERR_DEVICE_TIMEOUT,
    SPK_ERR_INVALID_ARG,
    SPK_ERR_OUT_OF_PATCH_PAGES,
    SPK_ERR_OUT_OF_SPECIAL_PAGES,
    SPK_F32,
    SPK_OK,
    SpkError,
    last_error,
    lib,
    make_config,
    read_device_status,
    required_bytes,
    selftest_wait_timeout,
)
