"""Helpers that drive the oracle over a workload (test-side glue, no method arithmetic)."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl


def make_streams(cfg: wl.Workload):
    """One oracle StreamPages per stream, with the workload's initial page orders."""
    patch_order, special_order = wl.page_orders(cfg)
    mpp, msp, b = cfg.max_patch_pages, cfg.max_special_pages, cfg.num_streams
    streams = []
    for s in range(b):
        if patch_order is None:
            pids, sids = oracle.default_page_ids(b, mpp, msp, s)
        else:
            pids = patch_order[s * mpp:(s + 1) * mpp].tolist()
            sids = special_order[s * msp:(s + 1) * msp].tolist()
        streams.append(oracle.StreamPages(
            patches_per_frame=cfg.patches_per_frame, specials_per_frame=cfg.specials_per_frame,
            page_size=cfg.page_size, scale_frames=cfg.scale_frames,
            sliding_window=cfg.sliding_window, patch_ids=pids, special_ids=sids))
    return streams


def step(streams):
    """Append one frame to every stream, then evict (the order the forward pass uses)."""
    targets = [st.append() for st in streams]
    for st in streams:
        st.evict()
    return targets


def frame_fetcher(cfg: wl.Workload, stream: int, block: int, cache=None):
    """fetch(frame, rows) for oracle.gather_visible, drawing frames from the workload."""
    cache = {} if cache is None else cache
    P = cfg.patches_per_frame

    def fetch(frame, rows):
        rows = np.asarray(rows)
        out_k, out_v = [], []
        if (rows < P).any():
            key = ("p", frame)
            if key not in cache:
                kp, vp = wl.frame_patch_kv(cfg, stream, block, frame)
                cache[key] = (wl.to_f64(kp, cfg.dtype), wl.to_f64(vp, cfg.dtype))
        if (rows >= P).any():
            key = ("s", frame)
            if key not in cache:
                ks, vs = wl.frame_special_kv(cfg, stream, block, frame)
                cache[key] = (wl.to_f64(ks, cfg.dtype), wl.to_f64(vs, cfg.dtype))
        for r in rows:
            if r < P:
                k, v = cache[("p", frame)]
                out_k.append(k[r]); out_v.append(v[r])
            else:
                k, v = cache[("s", frame)]
                out_k.append(k[r - P]); out_v.append(v[r - P])
        return np.stack(out_k), np.stack(out_v)

    return fetch


def oracle_attention(cfg: wl.Workload, streams, block: int, frame: int, q_per_stream=None, fetchers=None):
    """Oracle output [B*T, H, D] and lse [B*T, H] for the current plan of every stream."""
    outs, lses = [], []
    for s, st in enumerate(streams):
        fetch = fetchers[s] if fetchers is not None else frame_fetcher(cfg, s, block)
        k, v = oracle.gather_visible(st.visible_sources(), fetch)
        if q_per_stream is None:
            q = wl.to_f64(wl.frame_q(cfg, s, block, frame), cfg.dtype)
        else:
            q = q_per_stream[s]
        o, l = oracle.attend(q, k, v)
        outs.append(o); lses.append(l)
    return np.concatenate(outs), np.concatenate(lses)
