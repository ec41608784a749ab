"""The allocation-free attention entry point (this file is collected last).

Some callers must not allocate device memory once they are running: a real-time
loop whose memory was fixed when it started, or a process in which another
allocator already owns all device memory.  spk_run_attention_static_scratch
serves them by keeping the split-KV partial results in a static device array
inside the library instead of the caller's workspace.  These tests call it
through the C ABI and check it against spk_run_attention on the same plan, within
the bf16 tolerance the parity tests use.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _stream_frames(h, w):
    for f in range(w.frames):
        for s in range(w.num_streams):
            h.append(s, 0, *wl.frame_kv(w, s, 0, f))
        for s in range(w.num_streams):
            h.cache.evict_frames(s)
        h.plan()
        for b in range(1, w.num_blocks):
            for s in range(w.num_streams):
                h.append(s, b, *wl.frame_kv(w, s, b, f))


def test_static_scratch_matches_workspace_path_twice_in_a_row():
    import gpu_harness as gh

    w = wl.Workload("no_alloc", num_blocks=2, num_streams=2, num_heads=4, head_dim=64, page_size=256,
                    patches_per_frame=256, specials_per_frame=6, scale_frames=2, sliding_window=3, frames=6,
                    dtype="bf16", value_scale=0.5, shuffle_pages=True)
    h = gh.Harness(w, splits=4)   # several KV splits, so the merge reads partials back from the scratch
    _stream_frames(h, w)
    assert h.cache.get_plan_info()["merge_needed"] == 1
    qs = [gh.to_device(np.concatenate([wl.frame_q(w, s, b, w.frames - 1) for s in range(w.num_streams)]), "bf16")
          for b in range(w.num_blocks)]
    refs = []
    for b in range(w.num_blocks):
        ref = torch.empty_like(qs[b])
        h.cache.run_attention(b, qs[b], ref, h.ws, h.stream)
        refs.append(ref)
    # two calls in a row: the second finds the array as the first left it
    for b in (0, 1):
        got = torch.empty_like(qs[b])
        h.cache.run_attention_static_scratch(b, qs[b], got, h.ws, h.stream)
        torch.cuda.synchronize()
        gh.check_close(gh.to_f64(got), gh.to_f64(refs[b]), "bf16", f"static scratch, block {b}")
    assert h.status() == 0
    h.close()


def test_static_scratch_rejects_plans_that_do_not_fit():
    import gpu_harness as gh
    import streaming_paged_kv_two_gb300 as spk

    # 32 splits x 16 heads x 1005 rows x 65 floats is far beyond the static array
    w = wl.Workload("no_alloc_big", num_blocks=1, num_streams=1, num_heads=16, head_dim=64, page_size=1024,
                    patches_per_frame=999, specials_per_frame=6, scale_frames=2, sliding_window=40, frames=40,
                    dtype="bf16", value_scale=1.0)
    h = gh.Harness(w, splits=32)
    _stream_frames(h, w)
    q = gh.to_device(wl.frame_q(w, 0, 0, w.frames - 1), "bf16")
    out = torch.empty_like(q)
    with pytest.raises(spk.SpkError) as e:
        h.cache.run_attention_static_scratch(0, q, out, h.ws, h.stream)
    assert e.value.code == spk.SPK_ERR_INVALID_ARG and "static array" in str(e.value)
    h.close()
