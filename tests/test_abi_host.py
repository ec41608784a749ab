"""Host-side tests of libspk (no GPU): exported symbols, configuration checks,
bookkeeping-only caches against the oracle (bit-exact page tables, indptr,
last_page_len, patch-page counts, frame targets and statistics), and error codes."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wl
from oracle_cases import make_streams

spk = pytest.importorskip("streaming_paged_kv_two_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def cfg_for(w: wl.Workload, **over):
    po, so = wl.page_orders(w)
    args = dict(num_blocks=w.num_blocks, num_streams=w.num_streams, num_heads=w.num_heads, head_dim=w.head_dim,
                page_size=w.page_size, patches_per_frame=w.patches_per_frame,
                specials_per_frame=w.specials_per_frame, scale_frames=w.scale_frames,
                sliding_window=w.sliding_window, max_patch_pages=w.max_patch_pages,
                max_special_pages=w.max_special_pages,
                dtype=spk.SPK_BF16 if w.dtype == "bf16" else spk.SPK_F32,
                patch_page_order=None if po is None else po.tolist(),
                special_page_order=None if so is None else so.tolist())
    args.update(over)
    return spk.make_config(**args)


def test_every_declared_symbol_is_exported():
    inc = os.path.join(ROOT, "include")
    header = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    declared = set(re.findall(r"^\s*(?:int|const char\*)\s+(spk_\w+)\s*\(", header, re.M))
    assert len(declared) >= 15
    for name in sorted(declared):
        assert hasattr(spk.lib, name), name
        assert ctypes.cast(getattr(spk.lib, name), ctypes.c_void_p).value


def test_required_bytes_matches_layout():
    w = wl.CONFIGS["steady_state_10k"]
    cfg, keep = cfg_for(w)
    pool, ws = spk.required_bytes(cfg)
    pages = w.num_streams * (w.max_patch_pages + w.max_special_pages)
    assert pool == pages * 2 * w.page_size * w.num_heads * w.head_dim * 2
    assert ws % 256 == 0 and ws > 0


@pytest.mark.parametrize("over,needle", [
    (dict(head_dim=32), "head_dim"),
    (dict(page_size=100, patches_per_frame=101), "page_size"),
    (dict(specials_per_frame=0), "specials"),
    (dict(num_heads=0), "num_heads"),
    (dict(dtype=7), "dtype"),
    (dict(max_special_pages=0), "max pages"),
])
def test_invalid_configs_are_rejected(over, needle):
    cfg, keep = cfg_for(wl.CONFIGS["lingbot_like_200"], **over)
    with pytest.raises(spk.SpkError) as e:
        spk.required_bytes(cfg)
    assert e.value.code == spk.SPK_ERR_INVALID_ARG
    assert needle in str(e.value)


def test_bad_page_order_is_rejected():
    w = wl.CONFIGS["batched4_d128"]
    po, so = wl.page_orders(w)
    po = po.copy()
    po[3] = po[4]  # duplicate id
    cfg, keep = cfg_for(w, patch_page_order=po.tolist())
    with pytest.raises(spk.SpkError) as e:
        spk.Cache(cfg, None, keep)
    assert e.value.code == spk.SPK_ERR_INVALID_ARG
    po2, _ = wl.page_orders(w)
    po2 = po2.copy()
    po2[0], po2[w.max_patch_pages] = po2[w.max_patch_pages], po2[0]  # ids swapped across streams
    cfg, keep = cfg_for(w, patch_page_order=po2.tolist())
    with pytest.raises(spk.SpkError):
        spk.Cache(cfg, None, keep)


def _compare_stream_run(w: wl.Workload, frames: int, every: int = 1):
    cfg, keep = cfg_for(w)
    cache = spk.Cache(cfg, None, keep)
    streams = make_streams(w)
    T = w.tokens_per_frame
    for f in range(1, frames + 1):
        for s, st in enumerate(streams):
            pid, targets = st.append()
            cache.append_frame(s, 0)
            got_pid, got_targets = cache.get_frame_targets(s)
            assert got_pid == pid and got_targets == targets, (f, s)
        for s, st in enumerate(streams):
            st.evict()
            cache.evict_frames(s)
        if f % every == 0 or f == frames:
            cache.plan()
            want = oracle.plan(streams, T)
            got = cache.get_plan_host()
            assert got == want, f
            for s, st in enumerate(streams):
                assert cache.get_stats(s) == st.stats()
            info = cache.get_plan_info()
            cpp = lambda n: -(-n // 128)
            chunks = 0
            for s, st in enumerate(streams):
                chunks += st.num_patch_pages() * cpp(w.patches_per_frame)
                ns = len(st.special_pages)
                chunks += (ns - 1) * cpp(w.page_size) + cpp(st.last_page_len())
            assert info["num_chunks"] == chunks
            assert info["visible_tokens"] == sum(len(st.visible_sources()) for st in streams) if f % (every * 10) == 0 else True
    cache.close()


@pytest.mark.parametrize("name", ["tiny_stream_f32", "lingbot_like_200", "high_res_999", "batched4_d128"])
def test_bookkeeping_matches_oracle_workloads(name):
    w = wl.CONFIGS[name]
    _compare_stream_run(w, w.frames, every=1 if w.frames <= 2000 else 7)


def test_bookkeeping_matches_oracle_steady_state():
    w = wl.CONFIGS["steady_state_10k"]
    _compare_stream_run(w, w.frames, every=13)


@pytest.mark.parametrize("over", [
    dict(scale_frames=0, sliding_window=0),
    dict(scale_frames=0, sliding_window=1),
    dict(page_size=128, patches_per_frame=128, specials_per_frame=64),
    dict(page_size=256, patches_per_frame=199, specials_per_frame=57),
    dict(num_streams=3, shuffle_pages=True),
])
def test_bookkeeping_matches_oracle_edge_cases(over):
    base = wl.CONFIGS["lingbot_like_200"].replace(frames=150, num_blocks=2, **over)
    _compare_stream_run(base, base.frames)


def test_golden_stats_through_the_library():
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "cache_stats_after_42_frames.json")))
    s = g["setup"]
    cfg, keep = spk.make_config(num_blocks=1, num_streams=1, num_heads=16, head_dim=64, page_size=s["page_size"],
                                patches_per_frame=s["patches_per_frame"], specials_per_frame=s["specials_per_frame"],
                                scale_frames=s["scale_frames"], sliding_window=s["sliding_window"],
                                max_patch_pages=s["max_patch_pages"], max_special_pages=s["max_special_pages"])
    cache = spk.Cache(cfg, None, keep)
    for _ in range(s["frames"]):
        cache.append_frame(0, 0)
        cache.evict_frames(0)
    assert cache.get_stats(0) == g["expected"]


def test_visible_page_order_through_the_library():
    """The library's plan against the hand-worked page tables of the golden fixture (scale -> window
    oldest first -> specials in opening order, streams in index order)."""
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "visible_page_order.json")))
    for case in ("single_stream", "two_streams"):
        s = g[case]["setup"]
        cfg, keep = spk.make_config(num_blocks=1, num_streams=s["num_streams"], num_heads=2, head_dim=64,
                                    page_size=s["page_size"], patches_per_frame=s["patches_per_frame"],
                                    specials_per_frame=s["specials_per_frame"], scale_frames=s["scale_frames"],
                                    sliding_window=s["sliding_window"], max_patch_pages=s["max_patch_pages"],
                                    max_special_pages=s["max_special_pages"])
        cache = spk.Cache(cfg, None, keep)
        for want in g[case]["after_frame"]:
            for b in range(s["num_streams"]):
                cache.append_frame(b, 0)
            for b in range(s["num_streams"]):
                cache.evict_frames(b)
            cache.plan()
            got = cache.get_plan_host()
            want = {k: v for k, v in want.items() if k != "frame"}
            assert got == want, (case, got, want)


def _dry(w=None, **over):
    w = w or wl.CONFIGS["lingbot_like_200"].replace(num_blocks=3)
    cfg, keep = cfg_for(w, **over)
    return spk.Cache(cfg, None, keep)


def test_out_of_special_pages_changes_nothing():
    c = _dry(max_special_pages=1)   # 256 slots: 42 frames of 6 fit, the 43rd needs a second page
    for _ in range(42):
        c.append_frame(0, 0); c.evict_frames(0)
    before = c.get_stats(0)
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 0)
    assert e.value.code == spk.SPK_ERR_OUT_OF_SPECIAL_PAGES
    assert c.get_stats(0) == before


def test_out_of_patch_pages_changes_nothing():
    c = _dry(max_patch_pages=5)
    for _ in range(5):
        c.append_frame(0, 0)      # no eviction
    before = c.get_stats(0)
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 0)
    assert e.value.code == spk.SPK_ERR_OUT_OF_PATCH_PAGES
    assert c.get_stats(0) == before


def test_block_order_errors():
    c = _dry()
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 2)      # block 2 before any block 0
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    c.append_frame(0, 0)
    c.append_frame(0, 2)
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 2)      # twice in one frame
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 3)      # out of range
    assert e.value.code == spk.SPK_ERR_INVALID_ARG
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(1, 0)      # stream out of range
    assert e.value.code == spk.SPK_ERR_INVALID_ARG


def test_plan_needs_a_frame_and_dry_cache_has_no_device_calls():
    c = _dry()
    with pytest.raises(spk.SpkError) as e:
        c.plan()
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    with pytest.raises(spk.SpkError) as e:
        c.get_plan_host()
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    c.append_frame(0, 0)
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 1, k=16, v=16)   # dry cache takes no device pointers
    assert e.value.code == spk.SPK_ERR_INVALID_ARG
    c.plan()
    with pytest.raises(spk.SpkError) as e:
        c.run_attention(0, 16, 16, 256)
    assert e.value.code == spk.SPK_ERR_INVALID_ARG


def test_reset_restores_initial_order():
    w = wl.CONFIGS["batched4_d128"].replace(frames=300)
    cfg, keep = cfg_for(w)
    c = spk.Cache(cfg, None, keep)
    first = []
    for rnd in range(2):
        got = []
        for f in range(40):
            for s in range(w.num_streams):
                c.append_frame(s, 0)
                got.append(c.get_frame_targets(s))
                c.evict_frames(s)
        if rnd == 0:
            first = got
            c.reset()
            assert c.get_stats(0) == dict(frame_count=0, scale_pages=0, live_pages=0,
                                          free_pages=w.max_patch_pages, special_tokens=0)
        else:
            assert got == first


def test_split_choice_is_valid():
    w = wl.CONFIGS["steady_state_10k"].replace(frames=2000)
    cfg, keep = cfg_for(w)
    c = spk.Cache(cfg, None, keep)
    for f in range(300):
        c.append_frame(0, 0); c.evict_frames(0)
        c.plan()
        info = c.get_plan_info()
        assert 1 <= info["num_splits"] <= min(32, info["num_chunks"])
        assert info["num_ctas"] == info["num_splits"] * 16   # one CTA per (split, head): 2 tiles + 6-row tail
    for k in (1, 5, 32, 1000):
        cfg, keep = cfg_for(w, splits_per_stream=k)
        c = spk.Cache(cfg, None, keep)
        for f in range(100):
            c.append_frame(0, 0); c.evict_frames(0)
        c.plan()
        info = c.get_plan_info()
        assert info["num_splits"] == min(k, 32, info["num_chunks"])
        assert info["merge_needed"] == (1 if info["num_splits"] > 1 else 0)


# ------------------------------------------------------------------ several frames of queries

def test_plan_queries_tables_and_errors():
    """Scale-phase prefill plan ("Frame Processing Loop", num_frames > 1): the visible
    table is that of spk_plan, the query rows per stream are query_frames * T."""
    w = wl.CONFIGS["steady_state_10k"].replace(frames=64)
    cfg, keep = cfg_for(w, max_query_frames=8)
    c = spk.Cache(cfg, None, keep)
    T = w.tokens_per_frame
    with pytest.raises(spk.SpkError) as e:
        c.plan_queries(1)                       # no frame yet
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    for f in range(8):
        c.append_frame(0, 0); c.evict_frames(0)
    c.plan()
    one = c.get_plan_host()
    for qf in (1, 2, 8):
        c.plan_queries(qf)
        got = c.get_plan_host()
        for key in ("indices", "kv_indptr", "last_page_len", "num_patch_pages"):
            assert np.array_equal(got[key], one[key]), key
        assert list(got["qo_indptr"]) == [0, qf * T]
        info = c.get_plan_info()
        rows = qf * T
        main, rem = divmod(rows, 128)
        if rem > 8:                             # more than the D = 64 tail holds: another 128-row tile
            main += 1
        groups = max(1, -(-main // 2))          # two main tiles per CTA
        assert info["num_ctas"] == info["num_splits"] * w.num_heads * groups
    for bad in (0, 9):
        with pytest.raises(spk.SpkError) as e:
            c.plan_queries(bad)
        assert e.value.code == spk.SPK_ERR_INVALID_ARG
    cfg1, keep1 = cfg_for(w)                    # max_query_frames = 0: one frame per call
    c1 = spk.Cache(cfg1, None, keep1)
    c1.append_frame(0, 0); c1.append_frame(0, 0)
    with pytest.raises(spk.SpkError) as e:
        c1.plan_queries(2)
    assert e.value.code == spk.SPK_ERR_INVALID_ARG
    c2 = spk.Cache(cfg, None, keep)
    c2.append_frame(0, 0)
    with pytest.raises(spk.SpkError) as e:
        c2.plan_queries(2)                      # only one frame held
    assert e.value.code == spk.SPK_ERR_BAD_STATE


def test_max_query_frames_sizes_the_workspace():
    w = wl.CONFIGS["steady_state_10k"]
    ws = [spk.required_bytes(cfg_for(w, max_query_frames=q)[0])[1] for q in (0, 1, 8)]
    assert ws[0] == ws[1] < ws[2]
    with pytest.raises(spk.SpkError) as e:
        spk.required_bytes(cfg_for(w, max_query_frames=65)[0])
    assert e.value.code == spk.SPK_ERR_INVALID_ARG and "max_query_frames" in str(e.value)


# ------------------------------------------------------------------ deferred eviction and rollback

def _op_sequence_matches_oracle(w: wl.Workload, ops: int, seed: int):
    """Seeded random append / evict / defer / rollback / plan sequence: the library's
    tables, statistics and frame targets equal the oracle's after every step."""
    cfg, keep = cfg_for(w)
    cache = spk.Cache(cfg, None, keep)
    streams = make_streams(w)
    rng = np.random.default_rng(seed)
    T = w.tokens_per_frame
    rolled = 0
    for i in range(ops):
        s = int(rng.integers(w.num_streams))
        st = streams[s]
        r = rng.random()
        if r < 0.45:
            try:
                want = st.append()
            except (oracle.OutOfPatchPages, oracle.OutOfSpecialPages):
                with pytest.raises(spk.SpkError):
                    cache.append_frame(s, 0)
                continue
            cache.append_frame(s, 0)
            assert cache.get_frame_targets(s) == want, i
        elif r < 0.65:
            st.evict()
            cache.evict_frames(s)
        elif r < 0.75:
            on = bool(rng.integers(2))
            st.set_defer(on)
            cache.set_defer_eviction(s, on)
        else:
            try:
                st.rollback()
            except oracle.RollbackUnavailable:
                with pytest.raises(spk.SpkError) as e:
                    cache.rollback_frame(s)
                assert e.value.code == spk.SPK_ERR_BAD_STATE
                continue
            cache.rollback_frame(s)
            rolled += 1
        assert cache.get_stats(s) == st.stats(), i
        if all(x.frame_count for x in streams):
            cache.plan()
            assert cache.get_plan_host() == oracle.plan(streams, T), i
    cache.close()
    assert rolled > 0


@pytest.mark.parametrize("over,seed", [
    (dict(), 1),
    (dict(scale_frames=2, sliding_window=3), 2),
    (dict(scale_frames=0, sliding_window=0), 3),
    (dict(page_size=16, patches_per_frame=16, specials_per_frame=6, sliding_window=2, scale_frames=1), 4),
    (dict(num_streams=3, shuffle_pages=True, sliding_window=4, scale_frames=2), 5),
])
def test_rollback_and_deferral_match_oracle(over, seed):
    w = wl.CONFIGS["lingbot_like_200"].replace(frames=120, num_blocks=2, **over)
    _op_sequence_matches_oracle(w, 600, seed)


def test_rollback_restores_block_marks_and_targets():
    c = _dry()                                   # 3 blocks
    c.set_defer_eviction(0, True)
    c.append_frame(0, 0); c.append_frame(0, 1); c.append_frame(0, 2)
    prev = c.get_frame_targets(0)
    c.append_frame(0, 0)                         # new frame: only block 0 so far
    new = c.get_frame_targets(0)
    c.rollback_frame(0)
    assert c.get_frame_targets(0) == prev
    with pytest.raises(spk.SpkError) as e:
        c.append_frame(0, 1)                     # block 1 of the restored frame was already appended
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    with pytest.raises(spk.SpkError) as e:
        c.rollback_frame(0)                      # one rollback per append
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    c.append_frame(0, 0)
    assert c.get_frame_targets(0) == new         # the same targets again
    c.reset()
    with pytest.raises(spk.SpkError) as e:
        c.rollback_frame(0)
    assert e.value.code == spk.SPK_ERR_BAD_STATE


# ---------------------------------------------------------------- rotary append (host checks)

def _rope_call(cache, sections=(4, 2, 2), theta=10000.0, reserved=0, stream=0, block=0, **ptrs):
    rope = spk._lib.spk_rope((ctypes.c_int32 * 3)(*sections), reserved, theta)
    return spk.lib.spk_append_frame_rope(cache._h, stream, block, ptrs.get("k"), ptrs.get("v"), ptrs.get("q"),
                                         ptrs.get("q_out"), ptrs.get("positions"), ctypes.byref(rope), None)


@pytest.mark.parametrize("bad,needle", [
    (dict(sections=(-1, 2, 2)), "negative"),
    (dict(sections=(20, 10, 3)), "head_dim/2"),
    (dict(theta=0.0), "theta"),
    (dict(theta=float("nan")), "theta"),
    (dict(theta=float("inf")), "theta"),
    (dict(reserved=1), "reserved"),
    (dict(q=4096), "NULL"),
    (dict(positions=4096), "NULL"),
])
def test_rope_append_rejects_bad_arguments_and_changes_nothing(bad, needle):
    w = wl.CONFIGS["lingbot_like_200"]          # D = 64: 32 pairs
    cfg, keep = cfg_for(w)
    cache = spk.Cache(cfg, None, keep)
    cache.append_frame_rope(0, 0, sections=(12, 10, 10))
    cache.append_frame_rope(0, 1, sections=(12, 10, 10))
    before = (cache.get_stats(0), cache.get_frame_targets(0))
    rc = _rope_call(cache, **bad)
    assert rc == spk.SPK_ERR_INVALID_ARG
    assert needle in spk.last_error()
    assert (cache.get_stats(0), cache.get_frame_targets(0)) == before
    with pytest.raises(spk.SpkError):
        cache.append_frame_rope(0, 0, sections=(-1, 0, 0))
    assert (cache.get_stats(0), cache.get_frame_targets(0)) == before
    cache.close()


def test_rope_append_keeps_the_bookkeeping_of_append():
    w = wl.CONFIGS["high_res_999"]
    cfg, keep = cfg_for(w)
    a = spk.Cache(cfg, None, keep)
    b = spk.Cache(cfg, None, keep)
    for f in range(120):
        for blk in range(3):
            a.append_frame(0, blk)
            b.append_frame_rope(0, blk, sections=wl.rope_sections(w), theta=500.0)
        assert a.get_frame_targets(0) == b.get_frame_targets(0)
        a.evict_frames(0)
        b.evict_frames(0)
        assert a.get_stats(0) == b.get_stats(0)
    a.plan()
    b.plan()
    assert a.get_plan_host() == b.get_plan_host()
    with pytest.raises(spk.SpkError) as e:
        b.append_frame_rope(0, 1, sections=(0, 0, 0))   # block 1 twice in one frame
    assert e.value.code == spk.SPK_ERR_BAD_STATE
    a.close()
    b.close()


def test_package_refuses_to_import_without_the_library(tmp_path):
    """No CPU fallback: a copy of the binding without libspk.so fails at import."""
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "streaming_paged_kv_two_gb300")
    dst = tmp_path / "streaming_paged_kv_two_gb300"
    dst.mkdir()
    for f in ("__init__.py", "_lib.py"):
        shutil.copy(os.path.join(pkg, f), dst / f)
    r = subprocess.run([sys.executable, "-c", "import streaming_paged_kv_two_gb300"], cwd=tmp_path,
                       env={**os.environ, "PYTHONPATH": str(tmp_path)}, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libspk.so is not built" in r.stderr
