"""GPU cases that force the online softmax's rare paths, checked against the oracle.

The attention kernel keeps a running max per query row and moves it (rescaling the O
it has accumulated so far) only when a score exceeds it by more than a threshold.  With
ordinary N(0, 1) data that hardly ever happens after the first keys, so these cases
build inputs where it must, using the closed forms the pages' attention fixes ("How
LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction", "Attention Kernel
Execution": exact softmax attention over the visible keys):

* one key that dominates every row's logits (20+ log2 units above the rest), placed in
  the last chunk of a split that is not the first, so O is already filled when the
  running max jumps: the output is (close to) that key's V row;
* every visible key equal: the output is the mean of the visible V rows;
* a dominant key that only the tail rows (the few rows past the last full 128-row tile)
  see as dominant;
* a frame whose K/V hold Inf and NaN, appended and rolled back: its slots now lie past
  the tail special page's valid length, are loaded with the chunk and must not reach
  the output.

Each case runs through spk_debug_trace_attention, whose counters report how many times
a main-tile warp and the tail warps rescaled an accumulated O; the cases that force a
jump require them to be non-zero, and every output is compared element by element with
the fp64 oracle over the same (modified) data.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import workloads as wl  # noqa: E402
from oracle_cases import frame_fetcher, make_streams  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _gh():
    import gpu_harness
    return gpu_harness


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (round to nearest even), as the workloads store them."""
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _workload(D: int, P: int):
    # 9 frames, 2 scale frames, window 3: visible chunks = 5 patch pages x 2 + 1 special chunk;
    # with 3 forced splits the splits cover chunks [0, 3), [3, 7), [7, 11)
    return wl.Workload(f"paths_d{D}_p{P}", num_blocks=1, num_streams=1, num_heads=2, head_dim=D, page_size=256,
                       patches_per_frame=P, specials_per_frame=6, scale_frames=2, sliding_window=3, frames=9,
                       dtype="bf16", value_scale=0.5)


class _Data:
    """Every frame's k/v (float32 before rounding) and the final frame's q, with edits."""

    def __init__(self, w):
        self.w = w
        self.k, self.v = {}, {}
        for f in range(w.frames):
            k, v = wl.frame_kv(w, 0, 0, f)
            self.k[f] = wl.to_f64(k, "bf16").astype(np.float32)
            self.v[f] = wl.to_f64(v, "bf16").astype(np.float32)
        self.q = wl.to_f64(wl.frame_q(w, 0, 0, w.frames - 1), "bf16").astype(np.float32)

    def bits(self, x):
        return _bf16_round(x)

    def fetcher(self):
        cache = {}
        P = self.w.patches_per_frame
        for f in self.k:
            cache[("p", f)] = (wl.to_f64(self.bits(self.k[f][:P]), "bf16"), wl.to_f64(self.bits(self.v[f][:P]), "bf16"))
            cache[("s", f)] = (wl.to_f64(self.bits(self.k[f][P:]), "bf16"), wl.to_f64(self.bits(self.v[f][P:]), "bf16"))
        return frame_fetcher(self.w, 0, 0, cache)


def _run(w, data: _Data, splits: int = 3):
    gh = _gh()
    h = gh.Harness(w, splits=splits)
    st = make_streams(w)[0]
    for f in range(w.frames):
        h.append(0, 0, data.bits(data.k[f]), data.bits(data.v[f]))
        st.append()
        h.cache.evict_frames(0)
        st.evict()
    h.plan()
    qd = gh.to_device(data.bits(data.q), "bf16")
    out = torch.empty_like(qd)
    cap = 16
    buf = torch.zeros(20 * cap + 2, dtype=torch.int64, device="cuda")
    h.cache.debug_trace_attention(0, qd, out, h.ws, buf, cap, h.stream)
    torch.cuda.synchronize()
    got = gh.to_f64(out)
    counters = buf[20 * cap:].cpu().tolist()
    want, _ = oracle.attend(wl.to_f64(data.bits(data.q), "bf16"), *oracle.gather_visible(st.visible_sources(),
                                                                                        data.fetcher()))
    assert h.status() == 0
    info = h.cache.get_plan_info()
    h.close()
    return got, want, counters, info


def _unit(D, seed):
    u = np.random.default_rng(seed).standard_normal(D)
    return (u / np.linalg.norm(u)).astype(np.float32)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("P", [256, 250])   # T = 262 (two tiles and a 6-row tail) and T = 256 (no tail)
def test_dominant_key_late_in_a_split_moves_the_running_max(D, P):
    gh = _gh()
    w = _workload(D, P)
    data = _Data(w)
    H = w.num_heads
    alpha, beta = 4.0, 48.0 if D == 64 else 68.0   # alpha * beta / sqrt(D) * log2(e) > 30
    u = np.stack([_unit(D, 100 + h) for h in range(H)])          # [H, D]
    data.q += alpha * u[None]                                    # every row leans towards u
    # frame 7 is the middle page of the window: its first chunk is the last chunk of split 1
    data.k[7][100] = beta * u
    data.v[7][100] = 3.0 * _unit(D, 7)[None]
    got, want, counters, info = _run(w, data)
    assert info["num_splits"] == 3 and info["merge_needed"] == 1
    gh.check_close(got, want, "bf16", f"dominant key D={D} T={w.tokens_per_frame}")
    assert counters[0] > 0, "no main-tile warp rescaled an accumulated O"
    if w.tokens_per_frame % 128:
        assert counters[1] > 0, "the tail warps never rescaled an accumulated O"
    # the closed form: every row's output is (nearly) the dominant key's V row
    np.testing.assert_allclose(want, np.broadcast_to(wl.to_f64(data.bits(data.v[7][100]), "bf16"), want.shape),
                               atol=2e-2)  # the other keys keep a weight below 2^-16 each


@pytest.mark.parametrize("D", [64, 128])
def test_equal_keys_give_the_mean_of_v(D):
    gh = _gh()
    w = _workload(D, 256)
    data = _Data(w)
    kconst = np.random.default_rng(5).standard_normal((w.num_heads, D)).astype(np.float32)
    for f in data.k:
        data.k[f][:] = kconst[None]
    got, want, _, _ = _run(w, data)
    gh.check_close(got, want, "bf16", f"equal keys D={D}")
    st = make_streams(w)[0]
    for _ in range(w.frames):
        st.append()
        st.evict()
    _, vv = oracle.gather_visible(st.visible_sources(), data.fetcher())
    mean_v = vv.mean(axis=0)                                     # [H, D]
    np.testing.assert_allclose(got, np.broadcast_to(mean_v[None], got.shape), atol=2e-2)
    assert np.abs(got - mean_v[None]).mean() <= 2e-3


@pytest.mark.parametrize("D", [64, 128])
def test_jump_seen_by_the_tail_rows_only(D):
    gh = _gh()
    w = _workload(D, 256)
    data = _Data(w)
    T, H = w.tokens_per_frame, w.num_heads
    u = np.stack([_unit(D, 200 + h) for h in range(H)])
    data.q[256:] += 4.0 * u[None]                                # only the 6 tail rows lean towards u
    data.k[8][200] = (48.0 if D == 64 else 68.0) * u             # the newest window page, late in the last split
    data.v[8][200] = 3.0 * _unit(D, 9)[None]
    got, want, counters, _ = _run(w, data)
    gh.check_close(got, want, "bf16", f"tail-only jump D={D}")
    assert counters[1] > 0, "the tail warps never rescaled an accumulated O"
    np.testing.assert_allclose(want[256:], np.broadcast_to(wl.to_f64(data.bits(data.v[8][200]), "bf16"),
                                                           want[256:].shape), atol=2e-2)  # the other keys keep a weight below 2^-16 each
    assert T == 262


@pytest.mark.parametrize("D", [64, 128])
def test_non_finite_values_in_rolled_back_slots_do_not_reach_the_output(D):
    gh = _gh()
    w = _workload(D, 256).replace(frames=6)
    h = gh.Harness(w, splits=2)
    st = make_streams(w)[0]
    data = _Data(w)
    for f in range(w.frames):
        h.append(0, 0, data.bits(data.k[f]), data.bits(data.v[f]))
        st.append()
        h.cache.evict_frames(0)
        st.evict()
    # a candidate frame full of Inf / NaN, rolled back: its special slots stay in the tail
    # special page past the valid length (and are loaded with that chunk), its patch page is free
    h.cache.set_defer_eviction(0, True)
    bad_k = np.full((w.tokens_per_frame, w.num_heads, D), np.inf, dtype=np.float32)
    bad_v = np.full_like(bad_k, np.nan)
    bad_v[::2] = -np.inf
    h.append(0, 0, data.bits(bad_k), data.bits(bad_v))
    h.cache.rollback_frame(0)
    h.cache.set_defer_eviction(0, False)
    h.plan()
    qd = gh.to_device(data.bits(data.q), "bf16")
    out = torch.empty_like(qd)
    h.cache.run_attention(0, qd, out, h.ws, h.stream)
    torch.cuda.synchronize()
    got = gh.to_f64(out)
    assert np.isfinite(got).all(), "a rolled-back frame's non-finite values reached the output"
    want, _ = oracle.attend(wl.to_f64(data.bits(data.q), "bf16"),
                            *oracle.gather_visible(st.visible_sources(), data.fetcher()))
    gh.check_close(got, want, "bf16", f"after rollback of a non-finite frame D={D}")
    assert h.status() == 0
    h.close()
