"""Page bookkeeping of the two-stream paged KV cache, restated in plain Python.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title, section):

* "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction",
  "Patch Stream and Special Stream": patch pages 0..max_patch_pages-1, the first
  scale_frames frames kept for good, the next sliding_window frames form the
  recyclable live window; special pages max_patch_pages..max_num_pages-1 are
  append-only and never evicted.
* same page, "Page Table Planning and Reuse": the planned table lists the scale
  pages first, then the live-window pages, then the special pages, and
  paged_kv_last_page_len counts the tokens held by the last (possibly partial) page.
* "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback in
  Streaming Inference", "Two-Stream Design": one frame per patch page; special
  tokens pack contiguously across special pages, a new page taken from the free
  special pages when the tail page is full.
* "How FlashInfer KV Cache Attention Accelerates Streaming 3D Reconstruction
  Over SDPA", "FlashInferAttention Forward Pass": append, then evict, then
  attend — so the window counts the current frame.
* "How Paged KV Cache Attention Achieves Stable Inference in Ling-Bot-Map",
  "Sliding-Window Eviction Strategy": eviction moves page ids to the free list,
  no data is copied.
* "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback in
  Streaming Inference", "Inspecting Cache Statistics": the statistics dict
  (frame_count, scale_pages, live_pages, free_pages, special_tokens).
* "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction",
  "Scale Frames vs Sliding Window" and "Summary": deferred eviction, so that a
  frame can be rolled back (key-frame selection) without losing cache contents.

Readings where the pages are silent: the free lists are FIFO (allocate from the
front, recycle to the back); the initial order is ascending unless an explicit
order is given; an append that cannot get every page it needs changes nothing;
last_page_len is in [1, page_size], never 0; with several streams, stream s owns
patch ids [s*MPP, (s+1)*MPP) and special ids [B*MPP + s*MSP, B*MPP + (s+1)*MSP).
Deferred eviction and rollback (the pages name the feature only): while deferral is
on, evict() keeps the live window as it is; rollback() removes the newest frame and
returns the bookkeeping to its state just before that frame's append -- its patch
page goes back to the front of the free list, the special pages it opened to the
front of the free special list, its special tokens are dropped.  One rollback per
append; it needs the frame's patch page still held (not already evicted).
"""
from __future__ import annotations

from collections import deque


class OutOfPatchPages(RuntimeError):
    pass


class OutOfSpecialPages(RuntimeError):
    pass


class RollbackUnavailable(RuntimeError):
    pass


def default_page_ids(num_streams: int, max_patch_pages: int, max_special_pages: int, stream: int):
    """Ascending patch and special page ids owned by one stream."""
    b, mpp, msp = num_streams, max_patch_pages, max_special_pages
    patch = list(range(stream * mpp, (stream + 1) * mpp))
    base = b * mpp + stream * msp
    special = list(range(base, base + msp))
    return patch, special


class StreamPages:
    """Bookkeeping of one stream.  Page ids are the same for every block."""

    def __init__(self, *, patches_per_frame: int, specials_per_frame: int, page_size: int,
                 scale_frames: int, sliding_window: int, patch_ids, special_ids):
        self.P = patches_per_frame
        self.S = specials_per_frame
        self.ps = page_size
        self.sc = scale_frames
        self.w = sliding_window
        self.num_patch_ids = len(patch_ids)
        self.free = deque(int(x) for x in patch_ids)          # free_patch_pages
        self.scale: list[int] = []                             # scale_patch_pages
        self.live: deque[int] = deque()                        # live_window_patch_pages
        self.special_free = deque(int(x) for x in special_ids)  # free_special_pages
        self.special_pages: list[int] = []                     # all_special_pages
        self.special_tokens = 0
        self.frame_count = 0
        self.defer = False          # deferred eviction
        self.undo = None            # what the newest append took, while it can be rolled back
        # provenance of every written slot: page -> {slot: (frame, row of that frame)}
        self.contents: dict[int, dict[int, tuple[int, int]]] = {}

    # -- append_frame: allocation of one frame's targets --------------------
    def append(self):
        """Take the new frame's patch page and special slots; record what lands where.

        Returns (patch_page, [(special_page, slot), ...]) for the frame's S
        special tokens in row order.
        """
        if not self.free:
            raise OutOfPatchPages("no free patch page")
        first, last = self.special_tokens, self.special_tokens + self.S - 1
        pages_needed = last // self.ps + 1 - len(self.special_pages)
        if pages_needed > len(self.special_free):
            raise OutOfSpecialPages("special page pool exhausted")

        f = self.frame_count
        pid = self.free.popleft()
        in_scale = len(self.scale) < self.sc
        if in_scale:
            self.scale.append(pid)
        else:
            self.live.append(pid)
        opened = []
        page = self.contents.setdefault(pid, {})
        for t in range(self.P):
            page[t] = (f, t)

        targets = []
        for j in range(self.S):
            pos = first + j
            if pos // self.ps == len(self.special_pages):
                self.special_pages.append(self.special_free.popleft())
                opened.append(self.special_pages[-1])
            sp = self.special_pages[pos // self.ps]
            slot = pos % self.ps
            self.contents.setdefault(sp, {})[slot] = (f, self.P + j)
            targets.append((sp, slot))
        self.special_tokens += self.S
        self.frame_count += 1
        self.undo = (pid, in_scale, opened, targets)
        return pid, targets

    # -- evict_frames -------------------------------------------------------
    def evict(self):
        """Return the oldest live-window pages to the free list until the window fits
        (nothing while eviction is deferred)."""
        if self.defer:
            return
        while len(self.live) > self.w:
            self.free.append(self.live.popleft())

    # -- deferred eviction and rollback ---------------------------------------
    def set_defer(self, on: bool):
        self.defer = bool(on)

    def rollback(self):
        """Remove the newest frame: the state returns to just before its append."""
        if self.undo is None:
            raise RollbackUnavailable("no frame to roll back since the last append")
        pid, in_scale, opened, targets = self.undo
        held = self.scale if in_scale else self.live
        if not held or held[-1] != pid:
            raise RollbackUnavailable("the newest frame's patch page was already evicted")
        held.pop()
        self.free.appendleft(pid)
        self.contents.pop(pid, None)
        for sp, slot in targets:
            del self.contents[sp][slot]
        for sp in reversed(opened):
            assert self.special_pages[-1] == sp
            self.special_pages.pop()
            self.special_free.appendleft(sp)
        self.special_tokens -= self.S
        self.frame_count -= 1
        self.undo = None

    # -- plan pieces ----------------------------------------------------------
    def visible_pages(self) -> list[int]:
        return list(self.scale) + list(self.live) + list(self.special_pages)

    def num_patch_pages(self) -> int:
        return len(self.scale) + len(self.live)

    def last_page_len(self) -> int:
        n = len(self.special_pages)
        return self.special_tokens - (n - 1) * self.ps

    def visible_sources(self) -> list[tuple[int, int]]:
        """(frame, row) of every visible key, in page-table order.

        Patch pages contribute their P valid slots; special pages all ps slots
        except the last, which contributes last_page_len slots.
        """
        out = []
        for pid in self.scale + list(self.live):
            page = self.contents[pid]
            out.extend(page[t] for t in range(self.P))
        n = len(self.special_pages)
        for i, sp in enumerate(self.special_pages):
            count = self.ps if i < n - 1 else self.last_page_len()
            page = self.contents[sp]
            out.extend(page[t] for t in range(count))
        return out

    def stats(self) -> dict:
        return {
            "frame_count": self.frame_count,
            "scale_pages": len(self.scale),
            "live_pages": len(self.live),
            "free_pages": len(self.free),
            "special_tokens": self.special_tokens,
        }


def plan(streams: list[StreamPages], tokens_per_frame: int) -> dict:
    """The per-frame plan over all streams, concatenated in stream order.

    indices         visible page ids (scale, live window, specials) per stream
    kv_indptr       [B+1] offsets into indices
    last_page_len   [B] valid tokens on each stream's last (special) page
    num_patch_pages [B] leading patch pages of each stream (P valid tokens each)
    qo_indptr       [B+1] query-row offsets, tokens_per_frame rows per stream
    """
    indices, kv_indptr, lpl, npp, qo = [], [0], [], [], [0]
    for st in streams:
        pages = st.visible_pages()
        indices.extend(pages)
        kv_indptr.append(kv_indptr[-1] + len(pages))
        lpl.append(st.last_page_len())
        npp.append(st.num_patch_pages())
        qo.append(qo[-1] + tokens_per_frame)
    return {"indices": indices, "kv_indptr": kv_indptr, "last_page_len": lpl,
            "num_patch_pages": npp, "qo_indptr": qo}
