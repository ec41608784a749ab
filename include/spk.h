/*
 * spk.h — C ABI of libspk: streaming two-stream paged-KV attention on GB300.
 *
 * What it computes.  Each new frame of a video stream brings T = P + S tokens
 * (P patch tokens, S special tokens).  Every transformer block keeps its K/V in
 * a pool of pages [num_pages, 2 (K/V), page_size, H, D] (NHD).  Patch pages are
 * recyclable: the first scale_frames frames are kept for good and the next
 * sliding_window frames form a live window whose oldest page is recycled.
 * Special pages are append-only: the S special tokens of every frame pack
 * contiguously across them and are never evicted.  Once per frame the visible
 * page table (scale -> live window -> specials, with last_page_len) is planned;
 * every block then runs exact, non-causal softmax(Q K^T / sqrt(D)) V of the
 * frame's T queries over all visible keys, including the frame's own.
 *
 * Sources (page title, section):
 *   "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction":
 *     "Patch Stream and Special Stream", "Physical Memory Layout",
 *     "Page Table Planning and Reuse", "Attention Kernel Execution",
 *     "Appending Frames and Eviction", "Running Attention in Streaming Mode".
 *   "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback in
 *     Streaming Inference": "Two-Stream Design", "Plan-Run Execution Workflow",
 *     "Inspecting Cache Statistics".
 *   "How FlashInfer KV Cache Attention Accelerates Streaming 3D Reconstruction
 *     Over SDPA": "FlashInferKVCacheManager Responsibilities",
 *     "FlashInferAttention Forward Pass", "Efficient Attention Masking and Padding".
 *   "How Paged KV Cache Attention Achieves Stable Inference in Ling-Bot-Map":
 *     "Frame Appending Without Dispatch Overhead", "Sliding-Window Eviction
 *     Strategy", "Resetting for New Sequences".
 *
 * Conventions.
 *   - Every call returns an int status (SPK_OK or an SPK_ERR_* code); no C++
 *     exception crosses the ABI.  spk_last_error() gives a message for the last
 *     failing call on the calling thread.
 *   - Device memory (pools, workspace, q/k/v/out) is owned by the caller.  The
 *     library owns its host bookkeeping and the TMA descriptors it builds.
 *   - GPU work is ordered on the cudaStream_t passed as `cuda_stream` (a
 *     cudaStream_t value cast to void*; NULL is the legacy default stream).
 *   - Several streams (independent videos) may share one cache; each has its
 *     own bookkeeping and they are planned and attended in one batched launch.
 *   - Page ids: stream s owns patch ids [s*MPP, (s+1)*MPP) and special ids
 *     [B*MPP + s*MSP, B*MPP + (s+1)*MSP), with MPP = max_patch_pages,
 *     MSP = max_special_pages and B = num_streams.  Pools have B*(MPP+MSP) pages.
 *   - A cache created with pools == NULL is a bookkeeping-only ("dry") cache:
 *     append/evict/plan run on the host with no device memory and no CUDA call;
 *     calls that would touch device memory return SPK_ERR_INVALID_ARG.
 */
#ifndef SPK_H
#define SPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum spk_status {
  SPK_OK = 0,
  SPK_ERR_INVALID_ARG = 1,          /* bad pointer, size, id or configuration */
  SPK_ERR_OUT_OF_PATCH_PAGES = 2,   /* no free patch page for a new frame */
  SPK_ERR_OUT_OF_SPECIAL_PAGES = 3, /* every special page is full: the special stream only grows */
  SPK_ERR_BAD_STATE = 4,            /* wrong call order: block order, stale or missing plan */
  SPK_ERR_CUDA = 5,                 /* a CUDA runtime/driver call failed */
  SPK_ERR_DEVICE_TIMEOUT = 6        /* a device-side wait ran past its limit; see spk_read_device_status */
};

enum spk_dtype {
  SPK_BF16 = 0, /* hot path: bf16 storage, tcgen05 tensor cores, fp32 softmax/accumulate, bf16 out */
  SPK_F32 = 1   /* accuracy path: fp32 storage and fp32 CUDA-core arithmetic, fp32 out */
};

typedef struct {
  int32_t num_blocks;          /* L: one pool per transformer block */
  int32_t num_streams;         /* B: independent streams batched in one launch */
  int32_t num_heads;           /* H (query heads = KV heads) */
  int32_t head_dim;            /* D: 64 or 128 */
  int32_t page_size;           /* ps: tokens per page, >= patches_per_frame, <= 32768 */
  int32_t patches_per_frame;   /* P >= 1: rows 0..P-1 of a frame's k/v/q */
  int32_t specials_per_frame;  /* S >= 1: rows P..P+S-1 */
  int32_t scale_frames;        /* sc >= 0: first frames kept for good */
  int32_t sliding_window;      /* w >= 0: live window, counting the current frame */
  int32_t max_patch_pages;     /* MPP per stream, >= 1 (the pages' sizing: sc + w + 16) */
  int32_t max_special_pages;   /* MSP per stream, >= 1 (ceil(max_total_frames * S / ps)) */
  int32_t dtype;               /* enum spk_dtype */
  int32_t splits_per_stream;   /* 0 = planner's choice; k > 0 forces k KV splits per stream (clamped to [1, chunks]) */
  int32_t max_query_frames;    /* most frames of queries one attention call may carry (spk_plan_queries);
                                  0 or 1 = one frame per call.  Sizes the workspace's split partials. */
  const int32_t* patch_page_order;   /* optional host array [B*MPP]: initial free-list order, global ids;
                                        entries [s*MPP, (s+1)*MPP) must permute stream s's patch ids. NULL = ascending */
  const int32_t* special_page_order; /* optional host array [B*MSP], same rule for special ids. NULL = ascending */
} spk_config;

typedef struct {
  int64_t frame_count;     /* frames appended since create/reset */
  int64_t scale_pages;     /* patch pages held as scale frames */
  int64_t live_pages;      /* patch pages in the live window */
  int64_t free_pages;      /* free patch pages */
  int64_t special_tokens;  /* special tokens appended (S per frame) */
} spk_stats;

typedef struct {
  int32_t num_chunks;      /* KV chunks (<= 128 tokens inside one page) over all streams */
  int32_t num_splits;      /* KV splits over all streams */
  int32_t num_ctas;        /* CTAs of one attention launch */
  int32_t merge_needed;    /* 1 when some stream has more than one split (merge kernel runs) */
  int64_t visible_tokens;  /* sum over streams of visible keys */
  int64_t split_scratch_bytes;     /* bytes of split-KV partials this plan writes (0 when no merge
                                      runs); spk_run_attention_static_scratch needs them to fit */
  int64_t static_scratch_capacity; /* bytes of the library's static split-KV array */
} spk_plan_info;

typedef struct spk_cache spk_cache;

/* Message for the last failing call on this thread ("" if none).  Owned by the library. */
const char* spk_last_error(void);

/* Sizes the caller must allocate: one pool per block (pool_bytes_per_block, 256-byte
 * aligned start) and one workspace (workspace_bytes, 256-byte aligned start).
 * Either output pointer may be NULL.  No CUDA call. */
int spk_required_bytes(const spk_config* cfg, size_t* pool_bytes_per_block, size_t* workspace_bytes);

/* Create a cache ("How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D
 * Reconstruction", "Initializing the Cache Manager" and "Physical Memory Layout": one
 * pool [max_num_pages, 2, page_size, H, D] per block, page ids shared by every block).
 * pools: host array of num_blocks device pointers, or NULL for a
 * bookkeeping-only cache.  The library keeps the pointers (the caller keeps
 * ownership) and zeroes every pool once, on the legacy default stream, before
 * returning, so slots that are never written read as 0.  Builds one TMA
 * descriptor per pool (bf16).  The current CUDA device must be the pools' device. */
int spk_create_cache(const spk_config* cfg, void* const* pools, spk_cache** out);

/* Free the host state.  The pools and workspace stay the caller's. NULL is accepted. */
int spk_destroy_cache(spk_cache* cache);

/* Clear the bookkeeping (free lists back to their initial order, counters to zero);
 * the pools are kept as they are ("How Paged KV Cache Attention Achieves Stable
 * Inference in Ling-Bot-Map", "Resetting for New Sequences"). */
int spk_reset(spk_cache* cache);

/* Append one frame's K/V for one block ("How Paged KV Cache Attention Achieves Stable
 * Inference in Ling-Bot-Map", "Frame Appending Without Dispatch Overhead": direct
 * writes into the frame's slots; "How FlashInfer's Paged KV Cache Attention
 * Outperforms SDPA Fallback in Streaming Inference", "Two-Stream Design": one patch
 * page per frame, special tokens packed over append-only pages).
 * k, v: device [T, H, D] contiguous NHD in
 * the cache dtype, rows 0..P-1 patch tokens, rows P..T-1 special tokens.
 * block 0 starts a new frame: it takes a free patch page (a scale page while
 * fewer than scale_frames exist, else a live-window page) and reserves S special
 * slots, taking new special pages as the tail fills; all-or-nothing, so on
 * SPK_ERR_OUT_OF_* nothing changes.  It marks the plan stale.  Blocks 1..L-1 of
 * the same frame write to the same targets; calling block b > 0 before block 0 of
 * a frame, or twice in one frame, is SPK_ERR_BAD_STATE.  The copy runs on
 * cuda_stream (one kernel).  On a bookkeeping-only cache k and v must be NULL. */
int spk_append_frame(spk_cache* cache, int stream, int block, const void* k, const void* v,
                     void* cuda_stream);

/* 3-D rotary position embedding applied on append ("How LingBot-Map Uses FlashInfer
 * KV Cache for Streaming 3D Reconstruction", "3D RoPE Position Encoding" and the FAQ
 * "How is temporal information preserved in the KV cache?": q and k are rotated with
 * positions that carry the global frame index before k enters the cache, so attention
 * needs no position lookup).  The pages name the embedding without writing it out;
 * the rotation taken is RoFormer's (Su et al. 2021) per position axis:
 *   - the head dimension is D/2 adjacent pairs (x[2i], x[2i+1]);
 *   - pairs [0, sections[0]) follow axis t, the next sections[1] pairs axis h, the
 *     next sections[2] pairs axis w; later pairs are not turned;
 *   - pair j of a section of n pairs turns by position_axis * theta^(-j/n):
 *     (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a).
 * V is never rotated. */
typedef struct {
  int32_t sections[3];  /* turned pairs per axis t, h, w; each >= 0, sum <= D/2 */
  int32_t reserved;     /* must be 0 */
  double theta;         /* frequency base; finite and > 0 */
} spk_rope;

/* spk_append_frame with the rotary embedding fused into the scatter: one kernel
 * writes rotate(k) and v into the frame's slots (the same targets, bookkeeping, call
 * order and errors as spk_append_frame) and rotate(q) into q_out.
 *   positions: device int32 [T, 3], 4-byte aligned, (t, h, w) of each token row
 *              (rows as in k); any int32 value, negative included.
 *   q:         device [T, H, D] in the cache dtype, or NULL (then q_out is NULL too
 *              and only k is rotated).
 *   q_out:     device [T, H, D]; either q itself (rotated in place) or a buffer that
 *              does not overlap it.  k, v, q, q_out are 16-byte aligned.
 *   rope:      host struct, read during the call only.
 * Arithmetic: theta^(-j/n) in double on the host; on the device the angle
 * position * theta^(-j/n) and its reduction modulo 2*pi in double, sin/cos and the
 * rotation in fp32, one rounding to the cache dtype.  All arguments are checked
 * before any bookkeeping changes (SPK_ERR_INVALID_ARG).  On a bookkeeping-only cache
 * every device pointer is NULL and only the bookkeeping runs. */
int spk_append_frame_rope(spk_cache* cache, int stream, int block, const void* k, const void* v,
                          const void* q, void* q_out, const int32_t* positions, const spk_rope* rope,
                          void* cuda_stream);

/* Evict: move the oldest live-window pages to the free list until at most
 * sliding_window remain ("How Paged KV Cache Attention Achieves Stable Inference in
 * Ling-Bot-Map", "Sliding-Window Eviction Strategy": page ids move, no data is
 * copied).  Host only.  Marks the plan stale. */
int spk_evict_frames(spk_cache* cache, int stream);

/* Deferred eviction ("How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D
 * Reconstruction", "Scale Frames vs Sliding Window": deferred eviction for algorithms
 * that roll frames back, such as key-frame selection).  While on, spk_evict_frames
 * leaves the stream's live window as it is, so the window may hold more than
 * sliding_window frames (all visible) and no page is recycled; turning it off
 * changes nothing by itself, the next spk_evict_frames applies the window rule
 * (oldest pages first).  Host only.  Off after create and reset. */
int spk_set_defer_eviction(spk_cache* cache, int stream, int on);

/* Roll back the stream's newest frame: the bookkeeping returns to its state just
 * before that frame's append(block 0) -- its patch page goes back to the front of
 * the free list, the special pages it opened to the front of the free special
 * list, its S special tokens are dropped, the frame count and the previous frame's
 * block-append marks are restored -- so the next append takes the same targets
 * again.  The pool data is not touched (the rolled-back slots are no longer
 * visible).  One rollback per append; SPK_ERR_BAD_STATE when nothing was appended
 * since the last rollback or reset, or when the frame's patch page was already
 * evicted (defer eviction to keep it).  Marks the plan stale.  Host only. */
int spk_rollback_frame(spk_cache* cache, int stream);

/* Plan the current frame for every stream ("How LingBot-Map Uses FlashInfer KV Cache
 * for Streaming 3D Reconstruction", "Page Table Planning and Reuse": one plan per
 * frame, ordered scale -> window -> specials, reused by every block; "How Paged KV
 * Cache Attention Achieves Stable Inference in Ling-Bot-Map", "Visible Page Table
 * Construction" and "Kernel Dispatch and Sequence Lengths"): visible page table, indptr,
 * last_page_len, patch-page counts, KV chunks and the split-KV work list.  Built on
 * the host and uploaded with one async copy into `workspace` on cuda_stream; the
 * same plan serves every block until the next append(block 0) or evict.  Every
 * stream must hold at least one frame.  A bookkeeping-only cache takes
 * workspace == NULL and builds the host tables only. */
int spk_plan(spk_cache* cache, void* workspace, void* cuda_stream);

/* Plan an attention call whose queries are the last `query_frames` frames of every
 * stream: q and out then hold query_frames * T rows per stream (stream-major, the
 * stream's frames oldest first, rows 0..P-1 patch and P..T-1 special within each
 * frame), attending over the same visible keys as spk_plan.  This is the scale phase
 * of "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction"
 * ("Frame Processing Loop": num_frames > 1): append and evict the initialisation
 * frames one by one as usual, then one call attends every one of their query rows
 * over all of them (full, non-causal attention over the frames).  Later in a stream
 * the same call lets several recent frames query the whole visible cache at once.
 * spk_plan(c, ws, s) is spk_plan_queries(c, 1, ws, s).  1 <= query_frames <=
 * max(1, max_query_frames) and every stream must hold at least query_frames frames,
 * else SPK_ERR_INVALID_ARG / SPK_ERR_BAD_STATE. */
int spk_plan_queries(spk_cache* cache, int query_frames, void* workspace, void* cuda_stream);

/* Attention of the current frame for one block, all streams in one launch ("How
 * LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction", "Attention
 * Kernel Execution": exact softmax(Q K^T / sqrt(D)) V over the visible keys, non-causal;
 * "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback in Streaming
 * Inference", "Memory Bandwidth Efficiency": only the visible pages are read).
 * q: device [B*T, H, D] (stream s owns rows s*T..s*T+T-1), out: device [B*T, H, D],
 * both in the cache dtype; with spk_plan_queries, T stands for query_frames * T.
 * workspace must be the one given to the plan.  Launches the attention kernel and,
 * when a stream has several KV splits, the merge kernel (as a programmatic dependent
 * launch that waits for the attention grid).  Requires a current plan and block's K/V
 * appended for this frame on every stream. */
int spk_run_attention(spk_cache* cache, int block, const void* q, void* out, void* workspace,
                      void* cuda_stream);

/* The same attention as spk_run_attention, for callers that must not allocate device
 * memory while they run: for example a real-time loop whose memory was fixed when it
 * started, or a process in which another allocator already owns all device memory.
 * spk_run_attention keeps each KV split's partial results in the caller's workspace;
 * this call keeps them in a file-scope array inside the library instead
 * (32 MiB per device, held by every device that loads the library until the
 * process exits), so it needs nothing beyond its inputs and outputs and calls no
 * allocator.  The plan tables are still read from `workspace`, the buffer given to
 * spk_plan.  The pages describe no counterpart: this is a property of this
 * library's interface only.
 *   - spk_create_cache looks up the array's device address, with the cache's device
 *     current; that is when the array's module is loaded and its 32 MiB reserved.
 *     A call made while another device is current returns SPK_ERR_INVALID_ARG.
 *   - A plan whose partials exceed the array (splits * H * T * (D + 1) * 4 bytes,
 *     rounded up; spk_plan_info.split_scratch_bytes after spk_plan, against
 *     spk_plan_info.static_scratch_capacity) returns SPK_ERR_INVALID_ARG and launches
 *     nothing.  With splits_per_stream = 0 the planner's split count grows with the
 *     visible keys, so a stream with many query rows (large T) can outgrow the array
 *     part way through; force splits_per_stream to keep it within bounds.
 *   - Every call on a device shares the array and leaves its contents behind.
 *     Nothing in it needs to start at zero: each partial is written before it is
 *     read.  Calls whose GPU work overlaps (other streams, other caches) race on
 *     the array; order them on one stream. */
int spk_run_attention_static_scratch(spk_cache* cache, int block, const void* q, void* out, void* workspace,
                                     void* cuda_stream);

/* Copy one raw page [2, page_size, H, D] of block's pool to dst (host or device
 * memory, page_bytes = 2*ps*H*D*elem), for tests ("How FlashInfer's Paged KV Cache
 * Attention Outperforms SDPA Fallback in Streaming Inference", "Physical Memory
 * Layout").  Synchronizes cuda_stream before returning. */
int spk_read_kv(spk_cache* cache, int block, int page_id, void* dst, void* cuda_stream);

/* Host copy of the last plan: the tables the pages' planner hands its kernel
 * ("How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction", "Page
 * Table Planning and Reuse").  indices has room for `capacity` entries; kv_indptr
 * and qo_indptr [B+1]; last_page_len and num_patch_pages [B].  *nnz receives the
 * number of indices even when capacity is too small (then SPK_ERR_INVALID_ARG).
 * Array pointers other than nnz may be NULL to skip them. */
int spk_get_plan_host(const spk_cache* cache, int32_t* indices, int32_t capacity, int32_t* kv_indptr,
                      int32_t* last_page_len, int32_t* num_patch_pages, int32_t* qo_indptr,
                      int32_t* nnz);

/* Launch shape of the last plan. */
int spk_get_plan_info(const spk_cache* cache, spk_plan_info* info);

/* Targets of the stream's current frame: its patch page, and for each special row j
 * the special page and slot.  special_pages / special_slots have room for S entries. */
int spk_get_frame_targets(const spk_cache* cache, int stream, int32_t* patch_page,
                          int32_t* special_pages, int32_t* special_slots);

/* get_cache_stats() of one stream ("How FlashInfer's Paged KV Cache Attention
 * Outperforms SDPA Fallback in Streaming Inference", "Inspecting Cache Statistics"). */
int spk_get_stats(const spk_cache* cache, int stream, spk_stats* stats);

/* Synchronize cuda_stream, read and clear the device status word at the start of
 * `workspace`.  *code receives 0 or the raw device code; returns
 * SPK_ERR_DEVICE_TIMEOUT when a kernel recorded a wait that ran past its limit. */
int spk_read_device_status(void* workspace, void* cuda_stream, int32_t* code);

/* Self-test of the bounded device wait: one CTA waits on an mbarrier that nothing
 * signals, gives up after limit_ns nanoseconds, records the timeout in the status
 * word of `workspace` and returns normally.  Read it with spk_read_device_status. */
int spk_selftest_wait_timeout(void* workspace, int64_t limit_ns, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SPK_H */
