"""fp64 CPU oracle for streaming two-stream paged-KV attention.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
restatement of what the GPU path computes, written from the pages' description
of LingBot-Map's FlashInfer KV cache manager.  Only the test suite, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA library and imports nothing from it; both
take their inputs from ``workloads``.

Modules
-------
``paged_cache``  page bookkeeping of one stream (free / scale / live-window patch
                 deques, append-only special pages) and the per-frame plan
                 (visible page table, indptr, last_page_len).
``attention``    gather of the visible K/V into dense arrays and exact softmax
                 attention in float64, plus the log-sum-exp merge of partial
                 results.
``rope``         the 3-D rotary position embedding of q and k before caching.

Every function cites the passage it follows by page title and section.
Attention values themselves are pinned by closed forms, invariants and a
library routine (float64 SDPA) rather than by numbers printed on the pages,
which print none.
"""
from .paged_cache import (  # noqa: F401
    OutOfPatchPages,
    OutOfSpecialPages,
    RollbackUnavailable,
    StreamPages,
    default_page_ids,
    plan,
)
from .attention import attend, gather_visible, merge  # noqa: F401
from .rope import pair_angles, rotate  # noqa: F401
