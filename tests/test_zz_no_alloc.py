"""The allocation-free attention entry point (this file is collected last).

Some callers must not allocate device memory once they are running: a real-time
loop whose memory was fixed when it started, or a process in which another
allocator already owns all device memory.  spk_run_attention_static_scratch
serves them by keeping the split-KV partial results in a static device array
inside the library instead of the caller's workspace.  These tests call it
through the C ABI and check that

* its output is bit for bit the output of spk_run_attention on the same plan (the
  same kernels run on the same inputs; only the address of the partials differs),
  and within the parity bar of the fp64 oracle;
* this holds for the bf16 and the fp32 kernels, with several KV splits (the merge
  reads the partials back from the array) and with one split (no partials);
* it holds on repeated calls of the same block, and when another cache's call ran
  on the array in between (every call overwrites what the previous one left);
* once the library is set up, a call changes the device's free memory by nothing;
* a plan whose partials do not fit is refused before anything runs.
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


def _workload(dtype: str, seed_name: str):
    return wl.Workload(seed_name, num_blocks=2, num_streams=2, num_heads=4, head_dim=64, page_size=256,
                       patches_per_frame=256, specials_per_frame=6, scale_frames=2, sliding_window=3, frames=6,
                       dtype=dtype, value_scale=0.5, shuffle_pages=True)


def _oracle_out(w, block):
    import oracle  # noqa: F401
    from oracle_cases import make_streams, oracle_attention, step
    streams = make_streams(w)
    for _ in range(w.frames):
        step(streams)
    out, _ = oracle_attention(w, streams, block, w.frames - 1)
    return out


@pytest.mark.parametrize("dtype,splits", [("bf16", 4), ("bf16", 1), ("f32", 3), ("f32", 1)])
def test_static_scratch_is_bit_exact_with_the_workspace_path(dtype, splits):
    import gpu_harness as gh

    w = _workload(dtype, f"no_alloc_{dtype}")
    h = gh.Harness(w, splits=splits)
    _stream_frames(h, w)
    info = h.cache.get_plan_info()
    assert info["merge_needed"] == (1 if splits > 1 else 0)
    assert info["split_scratch_bytes"] <= info["static_scratch_capacity"]
    assert (info["split_scratch_bytes"] > 0) == (splits > 1)

    # a second cache whose calls also go through the static array, between ours
    w2 = _workload(dtype, f"no_alloc_other_{dtype}").replace(num_heads=2, frames=4)
    h2 = gh.Harness(w2, splits=5)
    _stream_frames(h2, w2)
    q2 = gh.to_device(np.concatenate([wl.frame_q(w2, s, 0, w2.frames - 1) for s in range(w2.num_streams)]), dtype)
    o2 = torch.empty_like(q2)

    qs = [gh.to_device(np.concatenate([wl.frame_q(w, s, b, w.frames - 1) for s in range(w.num_streams)]), dtype)
          for b in range(w.num_blocks)]
    refs = [torch.empty_like(q) for q in qs]
    gots = [[torch.empty_like(q) for _ in range(3)] for q in qs]
    for b in range(w.num_blocks):
        h.cache.run_attention(b, qs[b], refs[b], h.ws, h.stream)
    # every call on one stream: block 0 twice, the other cache, block 0 again, then block 1
    h.cache.run_attention_static_scratch(0, qs[0], gots[0][0], h.ws, h.stream)
    h.cache.run_attention_static_scratch(0, qs[0], gots[0][1], h.ws, h.stream)
    h2.cache.run_attention_static_scratch(0, q2, o2, h2.ws, h.stream)
    h.cache.run_attention_static_scratch(0, qs[0], gots[0][2], h.ws, h.stream)
    for i in range(3):
        h.cache.run_attention_static_scratch(1, qs[1], gots[1][i], h.ws, h.stream)
    torch.cuda.synchronize()
    for b in range(w.num_blocks):
        want = gh.to_f64(refs[b])
        gh.check_close(want, _oracle_out(w, b), dtype, f"workspace path, block {b}")
        for i, got in enumerate(gots[b]):
            assert torch.equal(got.view(torch.int32) if dtype == "f32" else got.view(torch.int16),
                               refs[b].view(torch.int32) if dtype == "f32" else refs[b].view(torch.int16)), \
                f"static scratch call {i} of block {b} differs from spk_run_attention"
    # the other cache's result through the array is right too
    ref2 = torch.empty_like(q2)
    h2.cache.run_attention(0, q2, ref2, h2.ws, h2.stream)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16) if dtype == "bf16" else o2.view(torch.int32),
                       ref2.view(torch.int16) if dtype == "bf16" else ref2.view(torch.int32))
    assert h.status() == 0 and h2.status() == 0
    h2.close()
    h.close()


def test_static_scratch_call_reserves_no_device_memory():
    import gpu_harness as gh

    w = _workload("bf16", "no_alloc_mem")
    h = gh.Harness(w, splits=4)
    _stream_frames(h, w)
    q = gh.to_device(np.concatenate([wl.frame_q(w, s, 1, w.frames - 1) for s in range(w.num_streams)]), "bf16")
    out = torch.empty_like(q)
    h.cache.run_attention_static_scratch(1, q, out, h.ws, h.stream)  # kernels loaded, array in use
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        h.cache.run_attention_static_scratch(1, q, out, h.ws, h.stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes across static-scratch calls"
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
    info = h.cache.get_plan_info()
    assert info["split_scratch_bytes"] > info["static_scratch_capacity"]
    q = gh.to_device(wl.frame_q(w, 0, 0, w.frames - 1), "bf16")
    out = torch.full_like(q, 7.0)
    with pytest.raises(spk.SpkError) as e:
        h.cache.run_attention_static_scratch(0, q, out, h.ws, h.stream)
    assert e.value.code == spk.SPK_ERR_INVALID_ARG and "static array" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a refused call must launch nothing"
    h.close()
