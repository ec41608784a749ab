"""Dense fp64 attention over the gathered visible K/V, and the log-sum-exp merge.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title, section):

* "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction",
  "Attention Kernel Execution": the accuracy-check path copies every visible key
  and value out of the pages into contiguous arrays and applies plain scaled
  dot-product attention to them.  This module is that definition in float64:
  gather, then for every head
  softmax(Q K^T / sqrt(D)) V, non-causal, over all visible keys including the
  current frame's own.
* "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction",
  "Frame Processing Loop": in streaming mode the frame's queries attend against
  the cached K/V through the planned page table.

The pages do not state the softmax scale; 1/sqrt(D) is the scaled dot-product
attention the accuracy path calls.  The log-sum-exp merge is not on the pages;
it is the exact recombination of softmax attention over disjoint key sets.
"""
from __future__ import annotations

import numpy as np


def gather_visible(sources, fetch):
    """Dense K and V [N, H, D] (float64) for the visible keys.

    sources: (frame, row) per visible key in page-table order.
    fetch(frame, rows) -> (k_rows, v_rows), each [len(rows), H, D] float64.
    """
    ks, vs = [], []
    i, n = 0, len(sources)
    while i < n:
        frame = sources[i][0]
        j = i
        while j < n and sources[j][0] == frame:
            j += 1
        k, v = fetch(frame, [r for _, r in sources[i:j]])
        ks.append(np.asarray(k, dtype=np.float64))
        vs.append(np.asarray(v, dtype=np.float64))
        i = j
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


def attend(q, k, v):
    """Exact attention of q [T, H, D] over k, v [N, H, D], all float64.

    Returns (out [T, H, D], lse [T, H]) with lse the natural-log sum of the
    scaled logits' exponentials, per row and head.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    t, h, d = q.shape
    out = np.empty((t, h, d))
    lse = np.empty((t, h))
    scale = 1.0 / np.sqrt(d)
    for hh in range(h):
        logits = (q[:, hh, :] @ k[:, hh, :].T) * scale     # [T, N]
        m = logits.max(axis=1, keepdims=True)
        p = np.exp(logits - m)
        l = p.sum(axis=1, keepdims=True)
        out[:, hh, :] = (p @ v[:, hh, :]) / l
        lse[:, hh] = (m + np.log(l))[:, 0]
    return out, lse


def merge(parts):
    """Combine attention results over disjoint key sets.

    parts: list of (out_j [T, H, D], lse_j [T, H]).  With M = max_j lse_j and
    w_j = exp(lse_j - M): out = sum_j w_j out_j / sum_j w_j and
    lse = M + log(sum_j w_j).
    """
    lses = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])   # [J, T, H]
    outs = np.stack([np.asarray(o, dtype=np.float64) for o, _ in parts])   # [J, T, H, D]
    m = lses.max(axis=0)
    w = np.exp(lses - m)
    total = w.sum(axis=0)
    out = (w[..., None] * outs).sum(axis=0) / total[..., None]
    return out, m + np.log(total)
