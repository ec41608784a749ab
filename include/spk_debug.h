/*
 * spk_debug.h — diagnostic entry points of libspk (not needed to use the cache).
 *
 * These calls run the bf16 tensor-core attention kernel in an instrumented variant,
 * compiled separately from the one spk_run_attention launches, so the production
 * kernel carries none of their code.  They exist for tests and for measuring where a
 * launch spends its time.  Same conventions as spk.h (int status, caller-owned device
 * memory, work ordered on cuda_stream).
 */
#ifndef SPK_DEBUG_H
#define SPK_DEBUG_H

#include "spk.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Diagnostics for the bf16 tensor-core kernel: run block's attention launch in
 * score-dump mode.  Every CTA stops after the first chunk of its KV split and writes
 * the raw Q K^T tiles of that chunk (fp32, before scaling and masking) for its up to
 * two 128-row main query tiles to dst[cta][tile][row][key] (rows and keys 0..127;
 * rows past T come from zero queries; a tile slot the CTA does not own is left as
 * is).  cta = (split * H + head) * groups + group, where a group covers query rows
 * [256*group, 256*group + 256).  dst: device memory of num_ctas * 2 * 128 * 128 * 4
 * bytes (num_ctas from spk_get_plan_info).  out is not written; same preconditions
 * as spk_run_attention. */
int spk_debug_dump_scores(spk_cache* cache, int block, const void* q, float* dst, void* workspace,
                          void* cuda_stream);

/* Diagnostics for the bf16 tensor-core kernel: run block's attention exactly as
 * spk_run_attention does (same outputs) while the first CTA records the SM clock
 * (clock64) of its pipeline events for each of its first `capacity` chunks into
 * trace[event][chunk] (device memory, 20 * capacity + 2 uint64).  Events, in order:
 * TMA issue, MMA (tile 0) sees K/V landed, S0 keys 0..63 issued, its P seen, S1 keys
 * 0..63 issued, its P seen, tail S^T issued, tail P seen, S0 keys 64..127 issued, its
 * P seen, K/V stage released by tile 0, softmax 0 sees S (keys 0..63), softmax 0
 * signals P, softmax 1 sees S (keys 0..63), softmax 1 signals P, tail sees S^T, tail
 * signals P, softmax 0 sees S (keys 64..127), softmax 0 signals P, K/V landed in
 * shared memory.  Entries of events that do not happen are left as they were.  The two
 * words after the 20 * capacity event clocks count, over every CTA of the launch, the
 * times a running max moved after O had started to accumulate (so O was rescaled): by
 * a main-tile softmax warp, and by the tail warps; the call adds to what they hold. */
int spk_debug_trace_attention(spk_cache* cache, int block, const void* q, void* out, void* workspace,
                              uint64_t* trace, int32_t capacity, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SPK_DEBUG_H */
