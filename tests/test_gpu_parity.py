"""GPU parity of the C-ABI path against the fp64 oracle (small and ragged cases).

Every case streams frames through append -> evict -> plan -> per-block
append/run_attention exactly as the library's users do, and compares each block's
output with the oracle's dense float64 attention over the visible keys:
bf16 within max-abs 2e-2 and mean-abs 2e-3, fp32 within max-abs 1e-4.
Pool contents are compared bit for bit through read_kv.
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


def _h():
    import gpu_harness
    return gpu_harness


def small(**kw):
    base = dict(name="small", num_blocks=2, num_streams=1, num_heads=2, head_dim=64, page_size=256,
                patches_per_frame=256, specials_per_frame=6, scale_frames=2, sliding_window=3,
                frames=9, dtype="bf16", value_scale=0.5)
    base.update(kw)
    return wl.Workload(**base)


def stream_and_check(w: wl.Workload, splits: int = 0, check=lambda f: True, blocks=None):
    """Stream w.frames frames; compare every checked frame's output with the oracle."""
    gh = _h()
    h = gh.Harness(w, splits)
    streams = make_streams(w)
    blocks = list(range(w.num_blocks)) if blocks is None else blocks
    fetch_cache = {}
    worst = (0.0, 0.0)
    T = w.tokens_per_frame
    for f in range(w.frames):
        for s in range(w.num_streams):
            k, v = wl.frame_kv(w, s, 0, f)
            h.append(s, 0, k, v)
            streams[s].append()
        for s in range(w.num_streams):
            h.cache.evict_frames(s)
            streams[s].evict()
        h.plan()
        for b in blocks:
            if b > 0:
                for s in range(w.num_streams):
                    k, v = wl.frame_kv(w, s, b, f)
                    h.append(s, b, k, v)
            q = np.concatenate([wl.frame_q(w, s, b, f) for s in range(w.num_streams)])
            got = h.run(b, q)
            if not check(f):
                continue
            fetchers = [frame_fetcher(w, s, b, fetch_cache.setdefault((s, b), {})) for s in range(w.num_streams)]
            qs = [wl.to_f64(q[s * T:(s + 1) * T], w.dtype) for s in range(w.num_streams)]
            want = np.concatenate([
                oracle.attend(qs[s], *oracle.gather_visible(streams[s].visible_sources(), fetchers[s]))[0]
                for s in range(w.num_streams)])
            mx, mn = gh.check_close(got, want, w.dtype, f"{w.name} frame {f} block {b}")
            worst = (max(worst[0], mx), max(worst[1], mn))
    assert h.status() == 0
    h.close()
    return worst


# ------------------------------------------------------------------ device status

def test_selftest_wait_timeout_is_reported_and_context_survives():
    import streaming_paged_kv_two_gb300 as spk
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    spk.selftest_wait_timeout(ws, 2_000_000, torch.cuda.current_stream())
    with pytest.raises(spk.SpkError) as e:
        spk.read_device_status(ws, torch.cuda.current_stream())
    assert e.value.code == spk.SPK_ERR_DEVICE_TIMEOUT
    assert spk.read_device_status(ws, torch.cuda.current_stream()) == 0   # cleared
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1024 * 1023 / 2                               # context still usable


# ------------------------------------------------------------------ append / read_kv

@pytest.mark.parametrize("w", [
    small(frames=7),
    small(frames=7, dtype="f32", head_dim=128),
    small(frames=9, page_size=256, patches_per_frame=200, specials_per_frame=57, scale_frames=1, sliding_window=2),
    small(frames=6, num_streams=2, shuffle_pages=True, head_dim=128),
], ids=["bf16_d64", "f32_d128", "pad_and_straddle", "two_streams_shuffled"])
def test_append_is_bit_exact(w):
    gh = _h()
    h = gh.Harness(w)
    streams = make_streams(w)
    for f in range(w.frames):
        frame_data = {}
        for s in range(w.num_streams):
            for b in range(w.num_blocks):
                k, v = wl.frame_kv(w, s, b, f)
                frame_data[(s, b)] = (k, v)
            k, v = frame_data[(s, 0)]
            h.append(s, 0, k, v)
            pid, targets = streams[s].append()
            assert h.cache.get_frame_targets(s) == (pid, targets)
        for s in range(w.num_streams):
            for b in range(1, w.num_blocks):
                h.append(s, b, *frame_data[(s, b)])
            h.cache.evict_frames(s)
            streams[s].evict()
        torch.cuda.synchronize()
        # every page written this frame holds exactly the frame's rows
        for s, st in enumerate(streams):
            pid, targets = h.cache.get_frame_targets(s)
            for b in range(w.num_blocks):
                k, v = frame_data[(s, b)]
                page = h.read_page(b, pid)
                P = w.patches_per_frame
                assert np.array_equal(page[0, :P], k[:P]) and np.array_equal(page[1, :P], v[:P])
                for j, (sp, slot) in enumerate(targets):
                    spage = h.read_page(b, sp)
                    assert np.array_equal(spage[0, slot], k[P + j]) and np.array_equal(spage[1, slot], v[P + j])
    # and every visible slot still holds what the oracle says was written there
    for s, st in enumerate(streams):
        for b in range(w.num_blocks):
            for page, slots in st.contents.items():
                if page not in st.visible_pages():
                    continue
                got = h.read_page(b, page)
                for slot, (frame, row) in slots.items():
                    k, v = wl.frame_kv(w, s, b, frame)
                    assert np.array_equal(got[0, slot], k[row]) and np.array_equal(got[1, slot], v[row])
    h.close()


# ------------------------------------------------------------------ raw scores

@pytest.mark.parametrize("D", [64, 128])
def test_tensor_core_scores_match(D):
    """S = Q K^T of each CTA's first chunk, straight from TMEM, against numpy."""
    gh = _h()
    w = small(frames=1, head_dim=D, num_blocks=1)
    h = gh.Harness(w, splits=3)          # chunks: patch 0..127, patch 128..255, specials 0..5
    k, v = wl.frame_kv(w, 0, 0, 0)
    h.append(0, 0, k, v)
    h.cache.evict_frames(0)
    h.plan()
    info = h.cache.get_plan_info()
    assert info["num_splits"] == 3 and info["num_chunks"] == 3
    T, H = w.tokens_per_frame, w.num_heads
    groups = info["num_ctas"] // (3 * H)
    q = wl.frame_q(w, 0, 0, 0)
    qd = gh.to_device(q, "bf16")
    dst = torch.zeros((info["num_ctas"], 2, 128, 128), dtype=torch.float32, device="cuda")
    h.cache.debug_dump_scores(0, qd, dst, h.ws, h.stream)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().astype(np.float64)
    qf = wl.to_f64(q, "bf16")
    kf = wl.to_f64(k, "bf16")
    chunk_keys = [kf[0:128], kf[128:256], np.concatenate([kf[256:262], np.zeros((122, H, D))])]
    # main tiles: the 6 trailing rows belong to the tail (not dumped)
    main_rows = 256
    checked = 0
    for split in range(3):
        for head in range(H):
            for group in range(groups):
                for t in range(2):
                    r0 = group * 256 + t * 128
                    if r0 >= main_rows:
                        continue
                    cta = (split * H + head) * groups + group
                    qt = np.zeros((128, D))
                    rows = qf[r0:min(main_rows, r0 + 128), head]
                    qt[:len(rows)] = rows
                    want = qt @ chunk_keys[split][:, head].T
                    np.testing.assert_allclose(got[cta, t], want, atol=2e-3, rtol=1e-4,
                                               err_msg=f"split {split} head {head} group {group} tile {t}")
                    checked += 1
    assert checked == 3 * H * 2
    h.close()


def test_trace_mode_gives_the_same_output_and_ordered_events():
    """spk_debug_trace_attention: same output as spk_run_attention; CTA 0's recorded
    clocks are filled for every chunk and ordered along the pipeline."""
    gh = _h()
    w = small(frames=6, num_blocks=1)
    h = gh.Harness(w, splits=2)
    for f in range(w.frames):
        h.append(0, 0, *wl.frame_kv(w, 0, 0, f))
        h.cache.evict_frames(0)
    h.plan()
    q = gh.to_device(wl.frame_q(w, 0, 0, w.frames - 1), "bf16")
    ref = torch.empty_like(q)
    h.cache.run_attention(0, q, ref, h.ws, h.stream)
    out = torch.empty_like(q)
    cap = 64
    buf = torch.zeros(20 * cap + 2, dtype=torch.int64, device="cuda")  # event clocks + two rescale counters
    h.cache.debug_trace_attention(0, q, out, h.ws, buf, cap, h.stream)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    t = buf[:20 * cap].view(20, cap).cpu().numpy()
    n = int((t[0] != 0).sum())                 # chunks CTA 0 loaded
    assert n >= 1
    tma, s0_seen, p0_arrive, p0_seen = t[0, :n], t[11, :n], t[12, :n], t[3, :n]
    assert (s0_seen > tma).all() and (p0_arrive >= s0_seen).all() and (p0_seen >= p0_arrive).all()
    assert h.status() == 0
    h.close()


# ------------------------------------------------------------------ attention parity

CASES = {
    "tiny_stream_f32": (wl.CONFIGS["tiny_stream_f32"], 0),
    "tiny_stream_bf16": (wl.CONFIGS["tiny_stream_f32"].replace(dtype="bf16", name="tiny_stream_bf16"), 0),
    "t262_d64": (small(), 0),
    "t262_d64_split1": (small(), 1),
    "t262_d64_split5": (small(), 5),
    "t262_d128_two_streams": (small(head_dim=128, num_streams=2, shuffle_pages=True, frames=7), 0),
    "t129_pad": (small(patches_per_frame=123, page_size=128, frames=8), 3),
    "t1005_ps1024": (small(patches_per_frame=999, page_size=1024, frames=5, value_scale=1.0, num_heads=2), 0),
    "specials_straddle": (small(patches_per_frame=200, specials_per_frame=57, frames=8), 2),
    "specials_only": (small(scale_frames=0, sliding_window=0, frames=6), 0),
    "window1_no_scale": (small(scale_frames=0, sliding_window=1, frames=5), 0),
    "f32_d128_streams": (small(dtype="f32", head_dim=128, num_streams=2, frames=5, value_scale=1.0), 3),
    "per_head_scale_d128": (small(head_dim=128, per_head_scale=True, num_streams=2, frames=5, shuffle_pages=True), 0),
    "t1_row": (small(patches_per_frame=1, specials_per_frame=1, page_size=16, frames=12), 0),
    "t136_tail8": (small(patches_per_frame=130, page_size=256, frames=6), 2),
    "t144_rem16_main": (small(patches_per_frame=138, page_size=256, frames=6), 2),
    "t150_rem22_main": (small(patches_per_frame=144, page_size=256, frames=6), 0),
    "t6_tail_only": (small(patches_per_frame=3, specials_per_frame=3, page_size=16, frames=10), 2),
    # more than 16 splits per stream: the merge combines its groups of 16 splits online
    "t262_d64_split24": (small(sliding_window=12, frames=16), 24),
    "f32_split20": (small(dtype="f32", sliding_window=12, frames=14, value_scale=1.0), 20),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_stream_parity(name):
    w, splits = CASES[name]
    worst = stream_and_check(w, splits)
    print(f"{name}: worst max-abs {worst[0]:.3e} mean-abs {worst[1]:.3e}")


# ------------------------------------------------------------------ several frames of queries

def queries_and_check(w: wl.Workload, plans: dict, splits: int = 0):
    """Stream w.frames frames; after frame f (all blocks appended), when f is in plans,
    plan plans[f] frames of queries and compare every block's output, whose rows are
    the last plans[f] frames' queries of each stream, with the oracle."""
    gh = _h()
    h = gh.Harness(w, splits, max_query_frames=max(plans.values()))
    streams = make_streams(w)
    fetch_cache = {}
    for f in range(w.frames):
        for s in range(w.num_streams):
            h.append(s, 0, *wl.frame_kv(w, s, 0, f))
            streams[s].append()
        for s in range(w.num_streams):
            h.cache.evict_frames(s)
            streams[s].evict()
        h.plan()
        for b in range(1, w.num_blocks):
            for s in range(w.num_streams):
                h.append(s, b, *wl.frame_kv(w, s, b, f))
        if f not in plans:
            continue
        qf = plans[f]
        h.plan_queries(qf)
        for b in range(w.num_blocks):
            qs = [np.concatenate([wl.frame_q(w, s, b, g) for g in range(f - qf + 1, f + 1)])
                  for s in range(w.num_streams)]
            got = h.run(b, np.concatenate(qs))
            fetchers = [frame_fetcher(w, s, b, fetch_cache.setdefault((s, b), {})) for s in range(w.num_streams)]
            want = np.concatenate([
                oracle.attend(wl.to_f64(qs[s], w.dtype), *oracle.gather_visible(streams[s].visible_sources(),
                                                                                 fetchers[s]))[0]
                for s in range(w.num_streams)])
            gh.check_close(got, want, w.dtype, f"{w.name} frame {f} block {b}, {qf} query frames")
    assert h.status() == 0
    h.close()


@pytest.mark.parametrize("name,w,plans,splits", [
    # scale phase: the first frames, full attention over all of them (8 x 262 = 2096 rows)
    ("scale_phase_d64", small(scale_frames=8, sliding_window=4, frames=8), {7: 8}, 0),
    ("scale_phase_d64_split3", small(scale_frames=4, sliding_window=2, frames=4), {3: 4}, 3),
    ("midstream_d128_two_streams", small(head_dim=128, num_streams=2, shuffle_pages=True, frames=7), {6: 3}, 2),
    ("midstream_f32", small(dtype="f32", frames=6, value_scale=1.0), {2: 2, 5: 3}, 2),
    ("tail_only_d64", small(patches_per_frame=2, specials_per_frame=1, page_size=16, frames=5), {4: 2}, 0),
    ("t130_x2_tail_d64", small(patches_per_frame=124, frames=4), {3: 2}, 2),
])
def test_multi_frame_query_parity(name, w, plans, splits):
    queries_and_check(w.replace(name=name), plans, splits)


# ------------------------------------------------------------------ deferred eviction and rollback

def test_rolled_back_frame_is_not_visible():
    """Key-frame selection: a candidate frame is appended with eviction deferred, attended,
    rolled back and replaced by another frame; attention then sees the replacement and
    the frame the deferral kept in the window, never the candidate."""
    gh = _h()
    w = small(frames=9, scale_frames=1, sliding_window=2, num_blocks=2)
    h = gh.Harness(w, splits=2)
    streams = make_streams(w)
    st = streams[0]
    T = w.tokens_per_frame
    caches = {}

    def check(f, data_frame, alias):
        for b in range(w.num_blocks):
            q = wl.frame_q(w, 0, b, data_frame)
            got = h.run(b, q)
            base = frame_fetcher(w, 0, b, caches.setdefault((b, data_frame != f), {}))
            fetch = lambda frame, rows: base(alias.get(frame, frame), rows)   # noqa: E731
            want = oracle.attend(wl.to_f64(q, w.dtype), *oracle.gather_visible(st.visible_sources(), fetch))[0]
            gh.check_close(got, want, w.dtype, f"frame {f} block {b} (data of frame {data_frame})")

    def append_all(f, data_frame, defer=None):
        h.append(0, 0, *wl.frame_kv(w, 0, 0, data_frame))
        st.append()
        if defer is not None:
            h.cache.set_defer_eviction(0, defer)
            st.set_defer(defer)
        h.cache.evict_frames(0)
        st.evict()
        h.plan()
        for b in range(1, w.num_blocks):
            h.append(0, b, *wl.frame_kv(w, 0, b, data_frame))

    for f in range(w.frames):
        if f in (4, 7):
            cand = 1000 + f
            h.cache.set_defer_eviction(0, True)
            st.set_defer(True)
            append_all(f, cand)
            check(f, cand, {f: cand})              # the candidate is visible while pending
            h.cache.rollback_frame(0)
            st.rollback()
            append_all(f, f, defer=False)          # the replacement; deferral ends with its eviction
        else:
            append_all(f, f)
        check(f, f, {})
    assert h.status() == 0
    h.close()


# ------------------------------------------------------------------ state errors on a real cache

def test_run_attention_state_errors():
    import streaming_paged_kv_two_gb300 as spk
    gh = _h()
    w = small(frames=3, num_blocks=3)
    h = gh.Harness(w)
    q = gh.to_device(wl.frame_q(w, 0, 0, 0), "bf16")
    out = torch.empty_like(q)
    k, v = wl.frame_kv(w, 0, 0, 0)
    h.append(0, 0, k, v)
    h.cache.evict_frames(0)
    with pytest.raises(spk.SpkError) as e:
        h.cache.run_attention(0, q, out, h.ws, h.stream)        # no plan yet
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    h.plan()
    with pytest.raises(spk.SpkError) as e:
        h.cache.run_attention(1, q, out, h.ws, h.stream)        # block 1 not appended
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    other = torch.zeros_like(h.ws)
    with pytest.raises(spk.SpkError) as e:
        h.cache.run_attention(0, q, out, other, h.stream)       # not the planned workspace
    assert e.value.code == spk.SPK_ERR_INVALID_ARG
    h.cache.run_attention(0, q, out, h.ws, h.stream)
    h.append(0, 0, k, v)                                        # new frame: plan is stale
    with pytest.raises(spk.SpkError) as e:
        h.cache.run_attention(0, q, out, h.ws, h.stream)
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    torch.cuda.synchronize()
    assert h.status() == 0
    h.close()


# ------------------------------------------------------------------ rotary append

def _rotated_close(got: np.ndarray, want: np.ndarray, x: np.ndarray, dtype: str, what: str):
    """got (device result, f64) against the fp64 rotation want of x.

    The kernel's fp32 angle reduction, sin/cos and rotation stay within 2e-6 of the
    pair's norm; bf16 then adds at most half an ulp of the stored value.  fp32 stores
    keep that 2e-6 bound alone.
    """
    norm = np.repeat(np.hypot(x[..., 0::2], x[..., 1::2]), 2, axis=-1)
    slack = 2e-6 * norm + 1e-30
    if dtype == "bf16":
        mag = np.abs(want) + slack
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 1e-38))) - 8)
        bound = half_ulp + slack
        exact = wl.bf16_bits_to_f64(wl.f32_to_bf16_bits(want.astype(np.float32)))
        assert np.mean(got == exact) > 0.99, f"{what}: {np.mean(got != exact):.4f} not nearest"
    else:
        bound = slack
    err = np.abs(got - want)
    assert (err <= bound).all(), f"{what}: worst excess {np.max(err - bound):.3e}"


def _rope_fetcher(w, block, sections, theta, offset, cache):
    base = frame_fetcher(w, 0, block, cache)

    def fetch(frame, rows):
        k, v = base(frame, rows)
        pos = wl.frame_positions(w, frame, offset)[np.asarray(rows)]
        return oracle.rotate(k, pos, sections, theta), v
    return fetch


ROPE_APPEND_CASES = {
    "bf16_d64_late_frames": (small(frames=5, num_heads=4), (12, 10, 10), 10000.0, 9990),
    "bf16_d128_pad_straddle": (small(frames=4, head_dim=128, patches_per_frame=200, specials_per_frame=57,
                                     scale_frames=1, sliding_window=2), (22, 21, 21), 10000.0, 123456),
    "f32_d128_partial_sections": (small(frames=4, dtype="f32", head_dim=128), (8, 4, 4), 100.0, 0),
    "bf16_d64_no_sections": (small(frames=3), (0, 0, 0), 10000.0, 7),
}


@pytest.mark.parametrize("name", sorted(ROPE_APPEND_CASES))
def test_rope_append_rotates_k_and_q(name):
    w, sections, theta, offset = ROPE_APPEND_CASES[name]
    gh = _h()
    h = gh.Harness(w)
    P, rot = w.patches_per_frame, 2 * sum(sections)
    for f in range(w.frames):
        pos = wl.frame_positions(w, f, offset)
        posd = torch.from_numpy(pos).cuda()
        for b in range(w.num_blocks):
            k, v = wl.frame_kv(w, 0, b, f)
            q = wl.frame_q(w, 0, b, f)
            kd, vd, qd = (gh.to_device(x, w.dtype) for x in (k, v, q))
            q_out = torch.empty_like(qd) if b == 0 else qd      # block 1 rotates q in place
            h.cache.append_frame_rope(0, b, kd, vd, qd, q_out, posd, sections, theta, h.stream)
            torch.cuda.synchronize()
            pid, targets = h.cache.get_frame_targets(0)
            page = h.read_page(b, pid)
            sk = np.concatenate([page[0, :P]] + [h.read_page(b, sp)[0, slot][None] for sp, slot in targets])
            sv = np.concatenate([page[1, :P]] + [h.read_page(b, sp)[1, slot][None] for sp, slot in targets])
            assert np.array_equal(sv, v), "V is stored unchanged"
            # pairs past the sections are copied bit for bit
            assert np.array_equal(sk[..., rot:], k[..., rot:])
            got_q = gh.to_f64(q_out)
            for got, x, label in ((wl.to_f64(sk, w.dtype), wl.to_f64(k, w.dtype), "k"),
                                  (got_q, wl.to_f64(q, w.dtype), "q")):
                want = oracle.rotate(x, pos, sections, theta)
                if rot == 0:
                    assert np.array_equal(got, x), label
                else:
                    _rotated_close(got, want, x, w.dtype, f"{name} frame {f} block {b} {label}")
        h.cache.evict_frames(0)
    assert h.status() == 0
    h.close()


def test_rope_append_argument_errors_launch_nothing():
    """Misaligned or missing device pointers are refused on the host (SPK_ERR_INVALID_ARG)
    before any bookkeeping changes or any kernel runs."""
    import streaming_paged_kv_two_gb300 as spk
    w = small(frames=2)
    gh = _h()
    h = gh.Harness(w)
    k, v = wl.frame_kv(w, 0, 0, 0)
    q = wl.frame_q(w, 0, 0, 0)
    kd, vd, qd = (gh.to_device(x, w.dtype) for x in (k, v, q))
    posd = torch.from_numpy(wl.frame_positions(w, 0)).cuda()
    sections = wl.rope_sections(w)
    before = h.cache.get_stats(0)
    bad = [dict(positions=posd.data_ptr() + 2), dict(positions=None), dict(q_out=None),
           dict(q=qd.data_ptr() + 8, q_out=qd.data_ptr() + 8)]
    for b in bad:
        args = dict(k=kd, v=vd, q=qd, q_out=qd, positions=posd)
        args.update(b)
        with pytest.raises(spk.SpkError) as e:
            h.cache.append_frame_rope(0, 0, args["k"], args["v"], args["q"], args["q_out"], args["positions"],
                                      sections, 10000.0, h.stream)
        assert e.value.code == spk.SPK_ERR_INVALID_ARG
        assert h.cache.get_stats(0) == before
    h.cache.append_frame_rope(0, 0, kd, vd, qd, qd, posd, sections, 10000.0, h.stream)
    torch.cuda.synchronize()
    assert h.cache.get_stats(0)["frame_count"] == before["frame_count"] + 1
    assert h.status() == 0
    h.close()


@pytest.mark.parametrize("w,offset", [
    (small(frames=6, num_heads=4), 2000),
    (small(frames=5, head_dim=128, patches_per_frame=200, specials_per_frame=57, scale_frames=1,
           sliding_window=2), 0),
], ids=["bf16_d64", "bf16_d128_pad_straddle"])
def test_rope_stream_attention_parity(w, offset):
    """Append with the rotary embedding, attend with the rotated queries: the oracle's
    attention over its own fp64 rotations of q and of every visible key."""
    gh = _h()
    h = gh.Harness(w)
    streams = make_streams(w)
    sections, theta = wl.rope_sections(w), 10000.0
    fetch_cache = {}
    for f in range(w.frames):
        pos = wl.frame_positions(w, f, offset)
        posd = torch.from_numpy(pos).cuda()
        hold = []
        for b in range(w.num_blocks):
            k, v = wl.frame_kv(w, 0, b, f)
            q = wl.frame_q(w, 0, b, f)
            kd, vd, qd = (gh.to_device(x, w.dtype) for x in (k, v, q))
            hold.append((kd, vd, qd))
            if b == 0:
                h.cache.append_frame_rope(0, 0, kd, vd, qd, qd, posd, sections, theta, h.stream)
                streams[0].append()
                h.cache.evict_frames(0)
                streams[0].evict()
                h.plan()
            else:
                h.cache.append_frame_rope(0, b, kd, vd, qd, qd, posd, sections, theta, h.stream)
            out = torch.empty_like(qd)
            h.cache.run_attention(b, qd, out, h.ws, h.stream)
            torch.cuda.synchronize()
            fetch = _rope_fetcher(w, b, sections, theta, offset, fetch_cache.setdefault(b, {}))
            rq = oracle.rotate(wl.to_f64(q, w.dtype), pos, sections, theta)
            want = oracle.attend(rq, *oracle.gather_visible(streams[0].visible_sources(), fetch))[0]
            gh.check_close(gh.to_f64(out), want, w.dtype, f"rope frame {f} block {b}")
    assert h.status() == 0
    h.close()
