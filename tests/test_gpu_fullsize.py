"""Full-size parity: the four bf16 workloads streamed to their measured frame, in the
launch configuration bench.py times (planner's own split choice), blocks 0 and L-1
compared with the fp64 oracle over all query rows and heads; and the LingBot-like stream
stored in fp32 through the fp32 accuracy path (max-abs 1e-4).

Frames whose patch pages are no longer visible at a checked frame receive a fixed
filler for their patch rows (their specials are always the real draws): attention
must not see them, and a wrong eviction would pull the filler into the softmax and
fail the comparison.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import oracle  # noqa: E402
import workloads as wl  # noqa: E402
from oracle_cases import frame_fetcher, make_streams  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _patch_visible_at(w, frame, at):
    """True when frame's patch page is visible after `at` frames (window rules)."""
    return frame < min(at, w.scale_frames) or max(w.scale_frames, at - w.sliding_window) <= frame < at


FULLSIZE = {name: wl.CONFIGS[name] for name in ("lingbot_like_200", "steady_state_10k", "high_res_999",
                                               "batched4_d128")}
FULLSIZE["lingbot_like_200_f32"] = wl.CONFIGS["lingbot_like_200"].replace(name="lingbot_like_200_f32", dtype="f32")


@pytest.mark.parametrize("name", sorted(FULLSIZE))
def test_fullsize_parity(name):
    import gpu_harness as gh

    w = FULLSIZE[name]
    dt = w.dtype
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    B, L, P = w.num_streams, w.num_blocks, w.patches_per_frame
    blocks = [0, L - 1]
    checks = sorted({w.frames // 2, w.frames})
    h = gh.Harness(w)
    streams = make_streams(w)
    rng = np.random.default_rng(12345)
    filler = rng.standard_normal((P, w.num_heads, w.head_dim), dtype=np.float32)
    filler = gh.to_device(wl.f32_to_bf16_bits(filler) if dt == "bf16" else filler, dt)
    bufs = {}
    for s in range(B):
        for b in blocks:
            kd = torch.empty((w.tokens_per_frame, w.num_heads, w.head_dim), dtype=tdt, device="cuda")
            vd = torch.empty_like(kd)
            bufs[(s, b)] = (kd, vd)
    fetch_cache = {}
    for f in range(w.frames):
        at_next_check = min(c for c in checks if c > f)
        for s in range(B):
            for b in blocks:
                kd, vd = bufs[(s, b)]
                if _patch_visible_at(w, f, at_next_check) or any(_patch_visible_at(w, f, c) for c in checks if c > f):
                    kp, vp = wl.frame_patch_kv(w, s, b, f)
                    kd[:P].copy_(gh.to_device(kp, dt))
                    vd[:P].copy_(gh.to_device(vp, dt))
                else:
                    kd[:P].copy_(filler)
                    vd[:P].copy_(filler)
                ks, vs = wl.frame_special_kv(w, s, b, f)
                kd[P:].copy_(gh.to_device(ks, dt))
                vd[P:].copy_(gh.to_device(vs, dt))
                if b == 0:
                    h.append_device(s, 0, kd, vd)
                    streams[s].append()
            for b in blocks[1:]:
                h.append_device(s, b, *bufs[(s, b)])
        for s in range(B):
            h.cache.evict_frames(s)
            streams[s].evict()
        if f + 1 in checks:
            h.plan()
            for b in blocks:
                q = np.concatenate([wl.frame_q(w, s, b, f) for s in range(B)])
                got = h.run(b, q)
                want = []
                for s in range(B):
                    fetch = frame_fetcher(w, s, b, fetch_cache.setdefault((s, b), {}))
                    k, v = oracle.gather_visible(streams[s].visible_sources(), fetch)
                    qs = wl.to_f64(q[s * w.tokens_per_frame:(s + 1) * w.tokens_per_frame], dt)
                    want.append(oracle.attend(qs, k, v)[0])
                mx, mn = gh.check_close(got, np.concatenate(want), dt, f"{w.name} frame {f} block {b}")
                print(f"{w.name} frames={f + 1} block={b}: max-abs {mx:.3e} mean-abs {mn:.3e} "
                      f"plan={h.cache.get_plan_info()}")
    assert h.status() == 0
    h.close()
