"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

* the cache-statistics example the pages print (golden fixture);
* the visible page order (scale -> window -> specials, the window oldest first, the
  specials in the order they were opened, streams in index order) of two small
  streams worked by hand, frame by frame (golden fixture);
* closed forms of the visible set (patch pages, special tokens, last page length);
* bookkeeping invariants (page conservation, no duplicate ids, specials never leave);
* brute force: dense attention over the whole frame history, sliced by the window
  rules, computed with float64 scaled_dot_product_attention from PyTorch;
* invariance under permutation of physical page ids;
* closed forms of attention (equal keys, one dominant key, V scaling, key shift);
* the log-sum-exp merge equals attention over the union, and lse equals a library
  logsumexp of the logits;
* deferred eviction and rollback: a rolled-back frame leaves the bookkeeping
  exactly as before its append (and the next append takes the same targets);
  deferred evictions, once committed, give the visible frames of a stream that
  never deferred;
* rotary embedding: angles and rotated values of a hand-worked token (closed-form
  cos/sin of angles derived by hand from the RoFormer frequencies), pair norms kept,
  rotations compose additively in position, scores depend only on the position
  difference, zero positions and empty sections leave x unchanged;
* planted mistakes in the oracle are caught by at least one of the pins above.
"""
from __future__ import annotations

import contextlib
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import oracle.attention as oatt
import oracle.paged_cache as opc
import oracle.rope as orope
import workloads as wl
from oracle_cases import make_streams, step

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(**kw):
    base = dict(name="small", num_blocks=1, num_streams=1, num_heads=2, head_dim=16, page_size=8,
                patches_per_frame=8, specials_per_frame=3, scale_frames=2, sliding_window=3,
                frames=12, dtype="f32", value_scale=1.0)
    base.update(kw)
    return wl.Workload(**base)


SMALL_VARIANTS = [
    _small(),
    _small(page_size=16, patches_per_frame=11, specials_per_frame=5),   # pad slots on patch pages
    _small(page_size=4, patches_per_frame=4, specials_per_frame=6),     # specials straddle 2+ pages
    _small(scale_frames=0, sliding_window=1),
    _small(scale_frames=0, sliding_window=0),                            # specials only
    _small(scale_frames=5, sliding_window=0, frames=9),
    _small(num_streams=2, shuffle_pages=True, frames=10),
    _small(num_heads=3, head_dim=8, frames=7, specials_per_frame=1, page_size=2, patches_per_frame=2),
]


# ---------------------------------------------------------------- pin helpers

def pin_golden_stats():
    with open(os.path.join(GOLDEN, "cache_stats_after_42_frames.json")) as fh:
        g = json.load(fh)
    s = g["setup"]
    st = oracle.StreamPages(patches_per_frame=s["patches_per_frame"], specials_per_frame=s["specials_per_frame"],
                            page_size=s["page_size"], scale_frames=s["scale_frames"],
                            sliding_window=s["sliding_window"],
                            patch_ids=range(s["max_patch_pages"]),
                            special_ids=range(s["max_patch_pages"], s["max_patch_pages"] + s["max_special_pages"]))
    for _ in range(s["frames"]):
        st.append()
        st.evict()
    assert st.stats() == g["expected"], st.stats()


def pin_page_order():
    """Visible page tables of the hand-worked streams in tests/golden/visible_page_order.json."""
    with open(os.path.join(GOLDEN, "visible_page_order.json")) as fh:
        g = json.load(fh)
    for case in ("single_stream", "two_streams"):
        s = g[case]["setup"]
        B, mpp, msp = s["num_streams"], s["max_patch_pages"], s["max_special_pages"]
        streams = []
        for b in range(B):
            pids, sids = oracle.default_page_ids(B, mpp, msp, b)
            streams.append(oracle.StreamPages(patches_per_frame=s["patches_per_frame"],
                                              specials_per_frame=s["specials_per_frame"], page_size=s["page_size"],
                                              scale_frames=s["scale_frames"], sliding_window=s["sliding_window"],
                                              patch_ids=pids, special_ids=sids))
        T = s["patches_per_frame"] + s["specials_per_frame"]
        for want in g[case]["after_frame"]:
            step(streams)
            p = oracle.plan(streams, T)
            for key in ("indices", "kv_indptr", "last_page_len", "num_patch_pages", "qo_indptr"):
                assert p[key] == want[key], f"{case} frame {want['frame']}: {key} {p[key]} != {want[key]}"


def closed_form(cfg, f):
    sc, w, P, S, ps = cfg.scale_frames, cfg.sliding_window, cfg.patches_per_frame, cfg.specials_per_frame, cfg.page_size
    n_patch = min(f, sc) + min(max(f - sc, 0), w)
    st = f * S
    ns = -(-st // ps)
    lpl = st - (ns - 1) * ps
    return n_patch, st, ns, lpl, n_patch * P + st


def pin_closed_forms(cfg, frames=None, check_sources_every=1):
    streams = make_streams(cfg)
    frames = cfg.frames if frames is None else frames
    seen_special = [[] for _ in streams]
    for f in range(1, frames + 1):
        step(streams)
        n_patch, st_tok, ns, lpl, n_vis = closed_form(cfg, f)
        p = oracle.plan(streams, cfg.tokens_per_frame)
        for s, st in enumerate(streams):
            assert p["num_patch_pages"][s] == n_patch
            assert st.special_tokens == st_tok
            assert len(st.special_pages) == ns
            assert p["last_page_len"][s] == lpl and 1 <= lpl <= cfg.page_size
            assert p["kv_indptr"][s + 1] - p["kv_indptr"][s] == n_patch + ns
            # invariants: page conservation, no duplicates, specials only grow
            assert len(st.free) + len(st.scale) + len(st.live) == cfg.max_patch_pages
            ids = list(st.free) + st.scale + list(st.live)
            assert len(set(ids)) == len(ids)
            assert st.special_pages[:len(seen_special[s])] == seen_special[s]
            seen_special[s] = list(st.special_pages)
            if f % check_sources_every == 0:
                assert len(st.visible_sources()) == n_vis
        assert p["qo_indptr"] == [i * cfg.tokens_per_frame for i in range(len(streams) + 1)]


def history_keys(cfg, hist_k, hist_v, f):
    """Brute-force visible set from the dense history: window rules applied to frames."""
    sc, w, P = cfg.scale_frames, cfg.sliding_window, cfg.patches_per_frame
    patch_frames = list(range(min(f, sc))) + list(range(max(sc, f - w), f))
    k = [hist_k[i][:P] for i in patch_frames] + [hist_k[i][P:] for i in range(f)]
    v = [hist_v[i][:P] for i in patch_frames] + [hist_v[i][P:] for i in range(f)]
    return np.concatenate(k), np.concatenate(v)


def sdpa64(q, k, v):
    """float64 scaled_dot_product_attention from PyTorch: q [T,H,D], k/v [N,H,D]."""
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]
    kt = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))[None]
    vt = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
    return o[0].numpy().transpose(1, 0, 2)


def pin_brute_force(cfg, seed=0):
    rng = np.random.default_rng(seed)
    T, H, D = cfg.tokens_per_frame, cfg.num_heads, cfg.head_dim
    streams = make_streams(cfg)
    hist = [([], []) for _ in streams]
    stores = [dict() for _ in streams]
    for f in range(1, cfg.frames + 1):
        for s, st in enumerate(streams):
            k = rng.standard_normal((T, H, D)); v = rng.standard_normal((T, H, D))
            hist[s][0].append(k); hist[s][1].append(v)
            stores[s][f - 1] = (k, v)
        step(streams)
        for s, st in enumerate(streams):
            q = rng.standard_normal((T, H, D))
            store = stores[s]
            kv, vv = oracle.gather_visible(st.visible_sources(),
                                           lambda fr, rows, store=store: (store[fr][0][rows], store[fr][1][rows]))
            o, _ = oracle.attend(q, kv, vv)
            kb, vb = history_keys(cfg, hist[s][0], hist[s][1], f)
            ref = sdpa64(q, kb, vb)
            np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def pin_permutation(seed=1):
    base = _small(frames=11, page_size=4, patches_per_frame=3, specials_per_frame=3, num_streams=2)
    perm = base.replace(shuffle_pages=True)
    rng = np.random.default_rng(seed)
    T, H, D = base.tokens_per_frame, base.num_heads, base.head_dim
    sa, sb = make_streams(base), make_streams(perm)
    po, so = wl.page_orders(perm)
    mpp, msp, B = base.max_patch_pages, base.max_special_pages, base.num_streams
    # ascending id -> permuted id (k-th id of a stream's list maps to the k-th of the other)
    idmap = {}
    for s in range(B):
        pa, spa = oracle.default_page_ids(B, mpp, msp, s)
        idmap.update(zip(pa, po[s * mpp:(s + 1) * mpp].tolist()))
        idmap.update(zip(spa, so[s * msp:(s + 1) * msp].tolist()))
    store = [dict() for _ in range(B)]
    for f in range(perm.frames):
        for s in range(B):
            store[s][f] = (rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D)))
        step(sa); step(sb)
        pa_, pb_ = oracle.plan(sa, T), oracle.plan(sb, T)
        assert pb_["indices"] == [idmap[i] for i in pa_["indices"]]
        for key in ("kv_indptr", "last_page_len", "num_patch_pages", "qo_indptr"):
            assert pa_[key] == pb_[key]
        q = rng.standard_normal((T, H, D))
        for s in range(B):
            fetch = lambda fr, rows, s=s: (store[s][fr][0][rows], store[s][fr][1][rows])
            oa, _ = oracle.attend(q, *oracle.gather_visible(sa[s].visible_sources(), fetch))
            ob, _ = oracle.attend(q, *oracle.gather_visible(sb[s].visible_sources(), fetch))
            np.testing.assert_allclose(oa, ob, rtol=0, atol=1e-12)


def pin_attention_closed_forms(seed=2):
    rng = np.random.default_rng(seed)
    T, N, H, D = 5, 37, 3, 16
    q = rng.standard_normal((T, H, D))
    v = rng.standard_normal((N, H, D))
    # equal keys -> mean of V
    k = np.broadcast_to(rng.standard_normal((1, H, D)), (N, H, D)).copy()
    o, lse = oracle.attend(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), (T, H, D)), atol=1e-12)
    # lse of equal keys: logit + log N
    logit = np.einsum("thd,hd->th", q, k[0]) / math.sqrt(D)
    np.testing.assert_allclose(lse, logit + math.log(N), atol=1e-12)
    # one dominant key -> its V row (keys small, one key along q_row with a huge logit)
    k = 0.01 * rng.standard_normal((N, H, D))
    j = 17
    for h in range(H):
        k[j, h] = 400.0 * q[0, h] / np.linalg.norm(q[0, h]) * math.sqrt(D) / np.linalg.norm(q[0, h])
    o, _ = oracle.attend(q[:1], k, v)
    np.testing.assert_allclose(o[0], v[j], atol=1e-9)
    # random keys: V scaling and shifting every key by one vector (logit shift per row)
    k = rng.standard_normal((N, H, D))
    o, lse = oracle.attend(q, k, v)
    o2, _ = oracle.attend(q, k, 3.5 * v)
    np.testing.assert_allclose(o2, 3.5 * o, atol=1e-12)
    u = rng.standard_normal((1, H, D))
    o3, _ = oracle.attend(q, k + u, v)
    np.testing.assert_allclose(o3, o, atol=1e-12)
    # lse against a library logsumexp of the scaled logits
    logits = np.einsum("thd,nhd->thn", q, k) / math.sqrt(D)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(logits, axis=2), atol=1e-12)
    # single frame, no scale frames: plain self-attention (library routine)
    np.testing.assert_allclose(o, sdpa64(q, k, v), atol=1e-12)


def pin_merge(seed=3):
    rng = np.random.default_rng(seed)
    T, N, H, D = 7, 50, 2, 8
    q, k, v = (rng.standard_normal(s) for s in ((T, H, D), (N, H, D), (N, H, D)))
    full_o, full_l = oracle.attend(q, k, v)
    for cuts in ([1], [25], [49], [3, 30], [10, 11, 40]):
        edges = [0, *cuts, N]
        parts = [oracle.attend(q, k[a:b], v[a:b]) for a, b in zip(edges[:-1], edges[1:])]
        o, l = oracle.merge(parts)
        np.testing.assert_allclose(o, full_o, atol=1e-12)
        np.testing.assert_allclose(l, full_l, atol=1e-12)
    o, l = oracle.merge([(full_o, full_l)])
    np.testing.assert_allclose(o, full_o, atol=1e-14)


def _state(st):
    return (list(st.free), list(st.scale), list(st.live), list(st.special_free), list(st.special_pages),
            st.special_tokens, st.frame_count, st.visible_sources() if st.frame_count else [])


def pin_rollback(cfg):
    """Rollback restores the pre-append state; committed deferrals match plain eviction."""
    st = make_streams(cfg)[0]
    ref = make_streams(cfg)[0]
    st.set_defer(True)
    for f in range(cfg.frames - 1):
        before = _state(st)
        first = st.append()
        st.evict()                              # deferred: a no-op
        st.rollback()
        assert _state(st) == before, f"rollback at frame {f} did not restore the state"
        assert st.append() == first, "the re-append must take the rolled-back targets"
        if f % 3 == 2:                          # commit the deferred evictions every third frame
            st.set_defer(False)
            st.evict()
            st.set_defer(True)
        ref.append()
        ref.evict()
        if f % 3 == 2:
            assert st.visible_sources() == ref.visible_sources(), f"frame {f}: deferred != plain eviction"
            total = len(st.free) + len(st.scale) + len(st.live)
            assert total == st.num_patch_ids and len(set(st.free) | set(st.scale) | set(st.live)) == total
    try:
        st.rollback(); st.rollback()            # one rollback per append
        raise AssertionError("a second rollback must be refused")
    except oracle.RollbackUnavailable:
        pass


def pin_rope_worked_example():
    """D = 8 (4 pairs), sections (2, 1, 0), theta = 100, token at (t, h, w) = (3, 5, 7).

    By hand: pair 0 is axis t, j = 0, frequency 1 -> angle 3; pair 1 is axis t,
    j = 1 of 2, frequency 100**(-1/2) = 0.1 -> angle 0.3; pair 2 is axis h, j = 0 ->
    angle 5; pair 3 lies past the sections -> not turned.
    """
    x = np.array([1.0, 0.0, 0.0, 1.0, 2.0, 0.0, 3.0, 4.0]).reshape(1, 1, 8)
    pos = np.array([[3, 5, 7]])
    ang = orope.pair_angles(pos, (2, 1, 0), 100.0, 8)
    np.testing.assert_allclose(ang[0], [3.0, 0.3, 5.0, 0.0], rtol=0, atol=1e-15)
    want = [math.cos(3.0), math.sin(3.0),          # (1, 0) turned by 3
            -math.sin(0.3), math.cos(0.3),         # (0, 1) turned by 0.3
            2 * math.cos(5.0), 2 * math.sin(5.0),  # (2, 0) turned by 5
            3.0, 4.0]
    np.testing.assert_allclose(orope.rotate(x, pos, (2, 1, 0), 100.0)[0, 0], want, rtol=0, atol=1e-14)


def pin_rope_properties(seed=5):
    """Rotations: pair norms kept, additive in position, scores relative, identity at 0."""
    rng = np.random.default_rng(seed)
    T, H, D = 7, 3, 16
    sections, theta = (3, 2, 2), 10000.0   # 7 of 8 pairs turned
    x = rng.standard_normal((T, H, D))
    p1 = rng.integers(-50, 10000, size=(T, 3))
    p2 = rng.integers(-50, 50, size=(T, 3))
    y = orope.rotate(x, p1, sections, theta)
    np.testing.assert_allclose(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]),
                               rtol=1e-12, atol=0)
    np.testing.assert_array_equal(y[..., 14:], x[..., 14:])  # the pair past the sections
    np.testing.assert_allclose(orope.rotate(y, p2, sections, theta), orope.rotate(x, p1 + p2, sections, theta),
                               rtol=0, atol=1e-9)
    np.testing.assert_array_equal(orope.rotate(x, np.zeros((T, 3), dtype=np.int64), sections, theta), x)
    np.testing.assert_array_equal(orope.rotate(x, p1, (0, 0, 0), theta), x)
    # q_i . k_j depends on the position difference only: shift every position alike
    q, k = x, rng.standard_normal((T, H, D))
    pq, pk = p2, rng.integers(-50, 50, size=(T, 3))
    shift = np.array([[1234, -7, 19]])
    s0 = np.einsum("ihd,jhd->hij", orope.rotate(q, pq, sections, theta), orope.rotate(k, pk, sections, theta))
    s1 = np.einsum("ihd,jhd->hij", orope.rotate(q, pq + shift, sections, theta),
                   orope.rotate(k, pk + shift, sections, theta))
    np.testing.assert_allclose(s1, s0, rtol=0, atol=1e-9)


PINS = {
    "golden_stats": pin_golden_stats,
    "page_order": pin_page_order,
    "closed_forms": lambda: [pin_closed_forms(c) for c in SMALL_VARIANTS],
    "brute_force": lambda: [pin_brute_force(c, i) for i, c in enumerate(SMALL_VARIANTS)],
    "permutation": pin_permutation,
    "attention_closed_forms": pin_attention_closed_forms,
    "merge": pin_merge,
    "rollback": lambda: [pin_rollback(c) for c in SMALL_VARIANTS if c.num_streams == 1],
    "rope_worked_example": pin_rope_worked_example,
    "rope_properties": pin_rope_properties,
}


# ---------------------------------------------------------------- tests

def test_golden_stats_example():
    pin_golden_stats()


def test_visible_page_order_worked_by_hand():
    pin_page_order()


@pytest.mark.parametrize("idx", range(len(SMALL_VARIANTS)))
def test_closed_forms_small(idx):
    pin_closed_forms(SMALL_VARIANTS[idx])


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_closed_forms_workloads(name):
    cfg = wl.CONFIGS[name]
    # every frame of every workload; the dense source list is checked on a stride
    pin_closed_forms(cfg, check_sources_every=max(1, cfg.frames // 20))


@pytest.mark.parametrize("idx", range(len(SMALL_VARIANTS)))
def test_brute_force_history(idx):
    pin_brute_force(SMALL_VARIANTS[idx], idx)


def test_brute_force_config1_shape():
    pin_brute_force(wl.CONFIGS["tiny_stream_f32"], 99)


def test_permutation_invariance():
    pin_permutation()


def test_attention_closed_forms():
    pin_attention_closed_forms()


def test_lse_merge():
    pin_merge()


def test_rope_worked_example():
    pin_rope_worked_example()


def test_rope_properties():
    pin_rope_properties()


def test_rollback_and_deferred_eviction():
    for c in SMALL_VARIANTS:
        if c.num_streams == 1:
            pin_rollback(c)


def test_rollback_needs_the_page_still_held():
    st = make_streams(_small(scale_frames=0, sliding_window=0, frames=4))[0]
    st.append()
    st.evict()                                  # w = 0 and no deferral: the page is already free
    with pytest.raises(oracle.RollbackUnavailable):
        st.rollback()
    st2 = make_streams(_small(frames=4))[0]
    with pytest.raises(oracle.RollbackUnavailable):
        st2.rollback()                          # nothing appended


def test_append_failure_changes_nothing():
    cfg = _small(frames=2)   # max_special_pages = ceil(2*3/8) = 1: the third frame needs a second page
    st = make_streams(cfg)[0]
    for _ in range(2):
        st.append(); st.evict()
    before = (list(st.free), list(st.scale), list(st.live), list(st.special_pages), st.special_tokens, st.frame_count)
    with pytest.raises(oracle.OutOfSpecialPages):
        st.append()
    after = (list(st.free), list(st.scale), list(st.live), list(st.special_pages), st.special_tokens, st.frame_count)
    assert before == after
    cfg = _small(frames=40, scale_frames=2, sliding_window=3, headroom=0)
    st = make_streams(cfg)[0]
    for _ in range(5):
        st.append()          # no eviction: 2 scale + 3 live fill all 5 patch pages
    with pytest.raises(oracle.OutOfPatchPages):
        st.append()


# ---------------------------------------------------------------- planted mistakes

@contextlib.contextmanager
def _patched(obj, name, value):
    old = getattr(obj, name)
    setattr(obj, name, value)
    try:
        yield
    finally:
        setattr(obj, name, old)


def _evict_keep_one_less(self):
    while len(self.live) > max(self.w - 1, 0):
        self.free.append(self.live.popleft())


def _evict_lifo(self):
    while len(self.live) > self.w:
        self.free.append(self.live.pop())


def _evict_scale_too(self):
    while len(self.live) > self.w:
        self.free.append(self.live.popleft())
    if len(self.scale) > 1 and self.frame_count > self.sc + self.w:
        self.free.append(self.scale.pop(0))


def _lpl_off_by_one(self):
    n = len(self.special_pages)
    return (self.special_tokens - (n - 1) * self.ps) % self.ps


def _attend_no_scale(q, k, v):
    return _ORIG_ATTEND(q * math.sqrt(q.shape[2]), k, v)


def _attend_k_for_v(q, k, v):
    return _ORIG_ATTEND(q, k, k)


def _attend_causal_drop_last(q, k, v):
    return _ORIG_ATTEND(q, k[:-1], v[:-1])


def _merge_wrong_sign(parts):
    lses = np.stack([l for _, l in parts]); outs = np.stack([o for o, _ in parts])
    m = lses.max(axis=0); w = np.exp(m - lses); total = w.sum(axis=0)
    return (w[..., None] * outs).sum(axis=0) / total[..., None], m + np.log(total)


_ORIG_ATTEND = oatt.attend


def _sources_skip_pad_wrong(self):
    out = []
    for pid in self.scale + list(self.live):
        page = self.contents[pid]
        out.extend(page[t] for t in range(self.P - 1))
    n = len(self.special_pages)
    for i, sp in enumerate(self.special_pages):
        count = self.ps if i < n - 1 else self.last_page_len()
        out.extend(self.contents[sp][t] for t in range(count))
    return out


def _rollback_page_to_back(self):
    pid, in_scale, opened, targets = self.undo
    (self.scale if in_scale else self.live).pop()
    self.free.append(pid)
    for sp, slot in targets:
        del self.contents[sp][slot]
    for sp in reversed(opened):
        self.special_pages.pop()
        self.special_free.appendleft(sp)
    self.special_tokens -= self.S
    self.frame_count -= 1
    self.undo = None


def _rollback_keeps_special_pages(self):
    pid, in_scale, opened, targets = self.undo
    (self.scale if in_scale else self.live).pop()
    self.free.appendleft(pid)
    for sp, slot in targets:
        del self.contents[sp][slot]
    self.special_tokens -= self.S
    self.frame_count -= 1
    self.undo = None


def _pages_specials_first(self):
    return list(self.special_pages) + list(self.scale) + list(self.live)


def _pages_window_reversed(self):
    return list(self.scale) + list(reversed(self.live)) + list(self.special_pages)


def _pages_scale_after_window(self):
    return list(self.live) + list(self.scale) + list(self.special_pages)


def _pages_specials_reversed(self):
    return list(self.scale) + list(self.live) + list(reversed(self.special_pages))


def _pages_window_by_id(self):
    return list(self.scale) + sorted(self.live) + list(self.special_pages)


def _plan_streams_reversed(streams, tokens_per_frame):
    p = _ORIG_PLAN(list(reversed(streams)), tokens_per_frame)
    return p


_ORIG_PLAN = opc.plan


_ORIG_PAIR_ANGLES = orope.pair_angles


def _rotate_backwards(x, positions, sections, theta):
    return _ORIG_ROTATE(x, -np.asarray(positions), sections, theta)


def _rotate_half_split(x, positions, sections, theta):
    # pairs (x[i], x[i + D/2]) instead of adjacent pairs
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[2]
    perm = np.empty(D, dtype=np.int64)
    perm[0::2] = np.arange(D // 2)
    perm[1::2] = np.arange(D // 2) + D // 2
    out = np.empty_like(x)
    out[..., perm] = _ORIG_ROTATE(x[..., perm], positions, sections, theta)
    return out


def _angles_full_dim_exponent(positions, sections, theta, head_dim):
    # theta**(-2j/n) instead of theta**(-j/n)
    return _ORIG_PAIR_ANGLES(positions, sections, float(theta) ** 2, head_dim)


def _angles_axis_swapped(positions, sections, theta, head_dim):
    return _ORIG_PAIR_ANGLES(np.asarray(positions)[:, [1, 0, 2]], sections, theta, head_dim)


_ORIG_ROTATE = orope.rotate


MUTATIONS = {
    "specials_listed_first": (opc.StreamPages, "visible_pages", _pages_specials_first),
    "window_listed_newest_first": (opc.StreamPages, "visible_pages", _pages_window_reversed),
    "scale_listed_after_window": (opc.StreamPages, "visible_pages", _pages_scale_after_window),
    "special_pages_reversed": (opc.StreamPages, "visible_pages", _pages_specials_reversed),
    "window_sorted_by_page_id": (opc.StreamPages, "visible_pages", _pages_window_by_id),
    "streams_planned_in_reverse": (opc, "plan", _plan_streams_reversed),
    "rope_turns_backwards": (orope, "rotate", _rotate_backwards),
    "rope_half_split_pairs": (orope, "rotate", _rotate_half_split),
    "rope_frequency_exponent_doubled": (orope, "pair_angles", _angles_full_dim_exponent),
    "rope_axes_swapped": (orope, "pair_angles", _angles_axis_swapped),
    "rollback_page_to_back_of_free_list": (opc.StreamPages, "rollback", _rollback_page_to_back),
    "rollback_keeps_opened_special_pages": (opc.StreamPages, "rollback", _rollback_keeps_special_pages),
    "window_excludes_current_frame": (opc.StreamPages, "evict", _evict_keep_one_less),
    "lifo_eviction": (opc.StreamPages, "evict", _evict_lifo),
    "scale_pages_evicted": (opc.StreamPages, "evict", _evict_scale_too),
    "last_page_len_zero_when_full": (opc.StreamPages, "last_page_len", _lpl_off_by_one),
    "patch_page_short_by_one": (opc.StreamPages, "visible_sources", _sources_skip_pad_wrong),
    "missing_softmax_scale": (oatt, "attend", _attend_no_scale),
    "k_used_as_v": (oatt, "attend", _attend_k_for_v),
    "last_key_dropped": (oatt, "attend", _attend_causal_drop_last),
    "merge_weight_sign": (oatt, "merge", _merge_wrong_sign),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    obj, attr, fn = MUTATIONS[name]
    monkeypatch.setattr(obj, attr, fn)
    # the package re-exports attend/merge/plan: patch those too
    if obj is oatt or obj is opc:
        monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for pin_name, pin in PINS.items():
        try:
            pin()
        except (AssertionError, KeyError, IndexError, ValueError, RuntimeError):
            caught.append(pin_name)
    assert caught, f"no pin caught the planted mistake {name}"
