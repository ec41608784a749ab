// Paged-prefill attention on the 5th-generation tensor cores (sm_103a).
//
// What it computes: for every stream, head and query row of the current frame,
// softmax(q K_vis^T / sqrt(D)) V_vis over the stream's visible keys, non-causal,
// the frame's own keys included ("How LingBot-Map Uses FlashInfer KV Cache for
// Streaming 3D Reconstruction", "Frame Processing Loop" and "Attention Kernel
// Execution"; "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback
// in Streaming Inference", "Memory Bandwidth Efficiency": only visible pages are
// read).  Visible keys arrive as the planner's chunks (<= 128 tokens inside one
// page), so patch-page padding and the tail special page's unused slots never
// enter the softmax ("How FlashInfer KV Cache Attention Accelerates Streaming 3D
// Reconstruction Over SDPA", "Efficient Attention Masking and Padding").
//
// One CTA (one per SM) = (KV split, head, query-row group).  A group is up to two
// 128-row "main" tiles, plus, on the last group, a "tail" of at most 8 trailing rows
// (262 = 2 x 128 + 6).  Keys are processed in 64-key halves of the 128-key chunks.
// Warp roles (16 warps):
//   warps 4-7   softmax of main tile 0, warps 8-11 softmax of main tile 1: one
//               thread per query row (= TMEM lane).  fp32 online softmax in log2 units:
//               a half's scores are exponentiated against the running max m and the
//               packed bf16 P words OR-ed together; only when one of them reaches 2.0 (a
//               score more than 1 above m) does the warp move m, rescale O in TMEM and
//               recompute the half; masking of the chunk's ragged tail.  Two schedules:
//               head_dim 64: each tile has two 64-key S buffers, so Q K^T of the next
//               half runs while the softmax works on the current one, and P is written
//               back over S (measured faster for D = 64);
//               head_dim 128: one S buffer per tile, released as soon as the softmax
//               has loaded its scores into registers (the next Q K^T then overlaps the
//               exponentials), and P goes to the tile's own P buffer once the previous
//               half's PV has read it; this frees the TMEM for the tail.
//   warps 0-3   tail softmax.  The tail is computed transposed: S2^T = K Q2^T
//               (M = 128 keys, N = 16 rows), so a thread holds one key's scores for
//               every tail row; warp q owns keys [32q, 32q+32) of each chunk.  The four
//               warps share one running max per row (moved, rarely, after a barrier
//               that ORs their "score above the max" flags), so one
//               O2^T += V^T P2^T (M = D columns of V, N = 8 or 16 rows, K = 128 keys, P2
//               from shared memory) accumulates a whole chunk.
//   warp 12     TMA producer: K and V chunk tiles gathered by page id through a
//               4-D tensor map over the pool (d, head, token, 2*page+kv), 128-byte
//               swizzle, into a ring of shared-memory stages.
//   warps 13-15 MMA issuers, one thread per consumer (main tile 0, main tile 1,
//               tail).  Main tile t, half chunk g: S = Q_t K_g^T (M=128, N=64, K=D) and,
//               once the softmax has written P_g, O_t += P_g V_g (M=128, N=D, K=64);
//               head_dim 64 issues Q K^T of half g+2 into the buffer the PV just read,
//               head_dim 128 issues Q K^T of half g+1 once the softmax has released
//               the S buffer.  The consumers advance independently; a K/V stage is
//               released once every consumer is done with it.
// The PV MMA's B operand is V extended by a 16-column block of ones in shared memory, so
// O0/O1 are D + 16 columns wide and column D accumulates the row sum of the bf16 P that
// the MMA consumed.
// head_dim 64: Q_t is the TMEM A operand of Q K^T (only K is read from shared memory).
// TMEM (512 columns): S0[0] | S0[1] | S1[0] | S1[1] (64 each) | O0 | O1 (80 each) |
// Q0 | Q1 (32 each) | S2^T (16) | O2^T (8).
// head_dim 128: Q in shared memory; S0 | S1 (64 each) | P0 | P1 (32 each) | O0 | O1
// (144 each) | S2^T (16) | O2^T (16), all 512 columns; V's two column blocks and the
// ones block sit at one stride per stage (Cfg's split-V layout).
// Key rows past a ragged chunk's length are zeroed in the V tile before a PV MMA reads
// them, so whatever a slot past the valid tokens holds (a rolled-back frame, an earlier
// stream) cannot reach the output, not even as 0 * Inf.
// The epilogue writes bf16 output (one split) or an fp32 partial with its log2
// log-sum-exp (several splits, combined by the merge kernel).
// Every mbarrier wait is bounded: on timeout the kernel records a status word, drains
// its own copies and MMAs, frees TMEM and returns.
// kDiag instantiations carry the diagnostics (score dump, event trace); the kernel that
// spk_run_attention launches is compiled without them.
#include "ptx_sm100.cuh"
#include "spk_internal.h"

#include <cuda_bf16.h>

namespace spk {
namespace {

constexpr int kColBlockBytes = 128 * 128;  // 128 rows x 64 bf16: one 128-byte-swizzled column block
constexpr int kTailMaxRows = 8;            // rows of the tail
constexpr int kTailN = 16;                 // N of S2^T (M = 128 needs N >= 16)
constexpr int kHalfKeys = 64;              // keys per main-tile score buffer
constexpr int kThreads = 512;
constexpr int kWarpMain = 4;   // first warp of main tile 0; tile 1 starts at 8
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;   // warps 13, 14, 15 issue the MMAs of main tile 0, main tile 1 and the tail
constexpr int kSoftmaxThreads = 384;  // warps 0-11 (all arrive on q_full)
// A packed bf16 P word has bit 14 or bit 30 set when one of its two values is >= 2.0
// (or not finite): the score lies more than 1 (log2 units) above the running max.
constexpr uint32_t kPHighBits = 0x40004000u;
constexpr float kThreshold = 1.0f;  // the same bound for the tail's fp32 check

constexpr int align1024(int x) { return (x + 1023) & ~1023; }

template <int D>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;  // one Q, K or V tile in shared memory
  static constexpr bool kTail = true;
  // N of O2^T = V^T P2^T: 8 rows with M = 64 (D = 64); M = 128 needs N >= 16 (rows 8-15 zero)
  static constexpr int kTailPvN = (D == 64) ? 8 : 16;
  static constexpr int kP2ColBlock = kTailPvN * 128;  // one 64-key column block of a tail P tile
  static constexpr int kP2Bytes = 2 * kP2ColBlock;    // one tail P tile: kTailPvN rows x 128 keys bf16
  static constexpr int kQ2ColBlock = kTailN * 128;    // one 64-dim column block of the tail Q tile
  // the row sums come out of the PV MMA, whose B operand is V extended by a 16-column
  // block of ones (O gets 16 more columns, each holding the row sum)
  // D == 128: V has two column blocks, so the ones block must be the third at the same
  // stride (the MMA's leading offset) from each stage's V: each stage puts its second V
  // block halfway between its first and the one shared ones block (see the layout below)
  static constexpr bool kSplitV = (D == 128);
  // D == 64: Q lives in TMEM as the A operand of Q K^T
  static constexpr bool kQTmem = (D == 64);
  // D == 128: one S buffer per tile, released once loaded, and a separate P buffer
  static constexpr bool kEarly = (D == 128);
  static constexpr int kStages = (D == 64) ? 6 : 2;
  // shared memory
  static constexpr int kQ0 = 0;                                   // D == 128: the two Q tiles
  static constexpr int kQ1 = kTile;
  static constexpr int kQ2 = kQTmem ? 0 : 2 * kTile;              // tail Q: 16 rows, D/64 column blocks
  static constexpr int kP2 = kQ2 + (D / 64) * kQ2ColBlock;         // two tail P tiles
  static constexpr int kKV = align1024(kP2 + 2 * kP2Bytes);
  static constexpr int kStageBytes = 2 * kTile;
  // D == 128, in 16 KB column blocks: Q0 Q1 (0-3), Q2 and P2 (4), K of stage 1 (5-6), V0 of
  // stage 1 (7), K of stage 0 (8-9), V1 of stage 1 (10), V0 of stage 0 (11), V1 of stage 0
  // (12), ones (13): stage 0's V blocks and the ones block are 1 block apart, stage 1's 3
  static constexpr int kOnesBlk = kSplitV ? 13 * kColBlockBytes : kKV + kStages * kStageBytes;  // 128 rows x 64 bf16 ones
  static constexpr int kTailX = kOnesBlk + kColBlockBytes;
  // K tile, V column block 0 and V column block 1 of stage st (byte offsets)
  __host__ __device__ static constexpr int k_off(int st) {
    return kSplitV ? (st ? 5 : 8) * kColBlockBytes : kKV + st * kStageBytes;
  }
  __host__ __device__ static constexpr int v_off(int st) {
    return kSplitV ? (st ? 7 : 11) * kColBlockBytes : kKV + st * kStageBytes + kTile;
  }
  __host__ __device__ static constexpr int v1_off(int st) {
    return kSplitV ? (st ? 10 : 12) * kColBlockBytes : v_off(st) + kColBlockBytes;
  }  // tail exchange: [2][4][8] maxima, [2][4] flags
  static constexpr int kBars = kTailX + (kTail ? 2 * 4 * (kTailMaxRows + 1) * 4 + 32 : 0);
  // full[S], empty[S], q_full, s_full[2][2], s_free[2], p_ready[2][2], pv_done[2], o_done[3],
  // s2_full, s2_free, p2_ready[2], pv2_done; D == 128 also v_full[S], v_empty[S] (full/empty
  // then track K only)
  static constexpr int kNumBars = 2 * kStages + 21 + (kSplitV ? 2 * kStages : 0);
  static constexpr int kMisc = kBars + 8 * kNumBars;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kLaunch = kBytes + 1024;  // slack for 1024-byte alignment
  static constexpr int kOW = D + 16;  // TMEM columns of a main tile's O (the last 16: row sums)
  // D == 64: S_t[b] at 64 (2t + b), P over S; D == 128: S_t at 64 t, P_t at kP0 + 32 t
  static constexpr uint32_t kP0 = 2 * kHalfKeys;
  static constexpr uint32_t kO0 = kEarly ? kP0 + kHalfKeys : 4 * kHalfKeys, kO1 = kO0 + kOW;
  static constexpr uint32_t kTQ0 = kO1 + kOW, kTQ1 = kTQ0 + (kQTmem ? D / 2 : 0);  // D == 64: Q0, Q1
  static constexpr uint32_t kS2 = kTQ1 + (kQTmem ? D / 2 : 0), kO2 = kS2 + kTailN;  // S2^T, O2^T
  static_assert(kO2 + kTailPvN <= 512, "TMEM budget");
  static_assert(!kSplitV || (kStages == 2 && kP2 + 2 * kP2Bytes <= 5 * kColBlockBytes &&
                             kOnesBlk - v_off(0) == 2 * (v1_off(0) - v_off(0)) &&
                             kOnesBlk - v_off(1) == 2 * (v1_off(1) - v_off(1))),
                "split V layout: the ones block is the third block at each stage's V stride");
  static_assert(kKV % 1024 == 0 && kP2 % 1024 == 0 && kQ2 % 1024 == 0 && kOnesBlk % 1024 == 0 &&
                kP2ColBlock % 1024 == 0 && kQ2ColBlock % 1024 == 0,
                "128-byte-swizzled tiles start on 1024-byte boundaries");
  static_assert(kLaunch <= 227 * 1024, "shared memory per CTA");
};


// TMEM columns of main tile t's scores and P for half chunk b
template <int D>
__device__ __forceinline__ uint32_t s_col(int t, int b) {
  return Cfg<D>::kEarly ? uint32_t(kHalfKeys * t) : uint32_t(kHalfKeys * (2 * t + b));
}
template <int D>
__device__ __forceinline__ uint32_t p_col(int t, int b) {
  return Cfg<D>::kEarly ? Cfg<D>::kP0 + uint32_t(kHalfKeys / 2 * t) : s_col<D>(t, b);
}

// Trace mode (diagnostics): CTA 0 records the SM clock of an event for a chunk.
template <bool kDiag>
__device__ __forceinline__ void trace_at(const AttnParams& p, int ev, int chunk, long long clk) {
  if constexpr (kDiag)
    if (p.trace != nullptr && blockIdx.x == 0 && chunk < p.trace_cap) p.trace[int64_t(ev) * p.trace_cap + chunk] = clk;
}
template <bool kDiag>
__device__ __forceinline__ void trace(const AttnParams& p, int ev, int chunk) {
  if constexpr (kDiag) trace_at<kDiag>(p, ev, chunk, clock64());
}

__device__ __forceinline__ void signal_abort(int32_t* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(status, kStatusWaitTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// max over the 32 lanes of a warp
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Byte address of element (row, key) of a tail P tile: rows x 128 keys bf16, K-major,
// 128-byte swizzle, keys 0-63 and 64-127 in two column blocks of col_block bytes.
__device__ __forceinline__ uint32_t p2_addr(uint32_t base, int col_block, int row, int key) {
  return base + uint32_t((key >> 6) * col_block + (row >> 3) * 1024 + (row & 7) * 128 +
                         ((((key & 63) >> 3) ^ (row & 7)) << 4) + (key & 7) * 2);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Zero key rows [r0, r1) of a 128-key V tile (D/64 column blocks of 128-byte rows, the
// first at sv0, the second at sv1; the swizzle only permutes 16-byte pieces inside a row,
// so a whole row is zeroed as it lies) with `nthreads` threads, this one being `tid`.
template <int D>
__device__ __forceinline__ void zero_v_rows(uint32_t sv0, uint32_t sv1, int r0, int r1, int tid, int nthreads) {
  const int units = (r1 - r0) * 8;  // 16-byte pieces per column block
  for (int i = tid; i < units * (D / 64); i += nthreads) {
    const int cb = i / units, u = i - cb * units;
    st_shared_zero16((cb ? sv1 : sv0) + uint32_t((r0 + (u >> 3)) * 128 + (u & 7) * 16));
  }
}

// a | b | c in one instruction
__device__ __forceinline__ uint32_t or3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xFE;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Store one row of a 128-row Q tile in K-major 128-byte-swizzled layout: 16-byte
// chunk c of row r goes to chunk c ^ (r & 7) of its 128-byte row.
template <int D>
__device__ __forceinline__ void store_q_row(uint32_t sq, int r, const uint4* src, bool valid) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (valid) v = __ldg(src + c);
    const int cb = c >> 3, cc = c & 7;
    const uint32_t dst = sq + cb * kColBlockBytes + (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}

// p = 2^(s*sl2 - m) for the 64 fp32 scores of a half chunk (two 32-column quarters),
// as exponentials of the bf16-rounded argument pairs packed to bf16 pairs in pk (the row
// sums come from the PV MMA).  *orr receives the OR of the packed words (their high
// exponent bits flag a value >= 2).
__device__ __forceinline__ void exp_pack64(const uint32_t* sa, const uint32_t* sb, float sl2, float neg_m,
                                           uint32_t (&pk)[32], uint32_t* orr) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const uint32_t* s = e < 16 ? sa : sb;
    const int i = 2 * (e & 15);
    float x0, x1;
    ptx::fma2(x0, x1, __uint_as_float(s[i]), __uint_as_float(s[i + 1]), sl2, neg_m);
    // x < 1 unless the max moves, so the argument's bf16 rounding moves p by at most
    // 0.14 % (at x = 1), below P's own rounding
    pk[e] = ptx::ex2_bf16x2(pack_bf16(x0, x1));
  }
  uint32_t o0 = 0, o1 = 0;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    o0 = or3(o0, pk[e], pk[e + 1]);
    o1 = or3(o1, pk[e + 2], pk[e + 3]);
  }
  *orr = o0 | o1;
}

// max over 32 scores (three-input max: two new values per instruction)
__device__ __forceinline__ float max32(const uint32_t* s, float mx) {
  float a = mx, b = -INFINITY;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    a = ptx::max3(a, __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
    b = ptx::max3(b, __uint_as_float(s[e + 2]), __uint_as_float(s[e + 3]));
  }
  return fmaxf(a, b);
}

__device__ __forceinline__ void mask32(uint32_t* s, int first_key, int len) {
  if (first_key + 32 > len) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (first_key + e >= len) s[e] = __float_as_uint(-INFINITY);
  }
}

// Scale `ncols` (a multiple of 16) TMEM columns of this warp's lanes by corr (per lane).
__device__ __forceinline__ void rescale_tmem(uint32_t taddr, int ncols, float corr) {
  int j = 0;
  for (; j + 32 <= ncols; j += 32) {
    uint32_t o[32];
    ptx::tmem_ld32(taddr + j, o);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
    ptx::tmem_st32(taddr + j, o);
  }
  if (j < ncols) {
    uint32_t o[16];
    ptx::tmem_ld16(taddr + j, o);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
    ptx::tmem_st16(taddr + j, o);
  }
}

// Rare path of the online softmax, taken when some P value of the warp reached 2: every
// row that did (`need`) moves its running max m to max(m, the half's max); O (every
// earlier PV of this tile: when o_cols > 0, wait for the previous half's PV, tracked by
// pv_bar) is scaled by corr = 2^(m - m_new), and the half's P is recomputed with the new
// offset.  Returns (m_new, 1 if the wait succeeded else 0).
//
// head_dim 64: the scores are still in TMEM (the S buffer is not released before P is
// stored over it), so this path reloads them and stores P itself; kept out of line so
// the hot loop's registers are not spent on it.
__device__ __noinline__ float2 move_running_max_tmem(uint32_t tO, uint32_t tS, int o_cols, bool need, float m,
                                                     float sl2, int first_key, int len, uint32_t pv_bar,
                                                     uint32_t parity, long long limit, const volatile int* abort_flag) {
  uint32_t sa[32], sb[32], pk[32], orr;
  ptx::tmem_ld32(tS, sa);
  ptx::tmem_ld32(tS + 32, sb);
  ptx::tmem_wait_ld();
  mask32(sa, first_key, len);
  mask32(sb, first_key + 32, len);
  const float mx = fmaxf(max32(sa, -INFINITY), max32(sb, -INFINITY)) * sl2;
  const float m_new = need ? fmaxf(m, mx) : m;
  const float corr = m_new == m ? 1.f : ptx::ex2(m - m_new);  // 0 while m is -inf
  bool ok = true;
  if (o_cols) {
    ok = ptx::mbar_wait_warp(pv_bar, parity, limit, abort_flag);
    ptx::tc_fence_after();
    rescale_tmem(tO, o_cols, corr);
  }
  exp_pack64(sa, sb, sl2, -m_new, pk, &orr);
  ptx::tmem_st32(tS, pk);
  ptx::tmem_wait_st();
  return make_float2(m_new, ok ? 1.f : 0.f);
}

// head_dim 128: the S buffer has been released, so the path works on the (masked)
// scores held in registers and leaves the new P in pk; inlined, because an out-of-line
// call would put those arrays in local memory for the whole loop.
__device__ __forceinline__ float2 move_running_max_regs(const uint32_t (&sa)[32], const uint32_t (&sb)[32],
                                                        uint32_t (&pk)[32], uint32_t tO, int o_cols, bool need,
                                                        float m, float sl2, uint32_t pv_bar, uint32_t parity,
                                                        long long limit, const volatile int* abort_flag) {
  const float mx = fmaxf(max32(sa, -INFINITY), max32(sb, -INFINITY)) * sl2;
  const float m_new = need ? fmaxf(m, mx) : m;
  const float corr = m_new == m ? 1.f : ptx::ex2(m - m_new);  // 0 while m is -inf
  bool ok = true;
  if (o_cols) {
    ok = ptx::mbar_wait_warp(pv_bar, parity, limit, abort_flag);
    ptx::tc_fence_after();
    rescale_tmem(tO, o_cols, corr);
  }
  uint32_t orr;
  exp_pack64(sa, sb, sl2, -m_new, pk, &orr);
  return make_float2(m_new, ok ? 1.f : 0.f);
}

// Write 32 columns [col0, col0+32) of one output row from raw fp32 TMEM values times
// `scale`: bf16 output when the stream has one split, else the fp32 partial.
template <int D>
__device__ __forceinline__ void store_output_cols(const AttnParams& p, const WorkDesc& work, int split, int head,
                                                  int row, const uint32_t (&v)[32], int col0, float scale) {
  if (work.nsplit == 1) {
    const int64_t qrow = int64_t(work.stream) * p.T + row;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (qrow * p.H + head) * D + col0);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      dst[k] = make_uint4(pack_bf16(__uint_as_float(v[8 * k]) * scale, __uint_as_float(v[8 * k + 1]) * scale),
                          pack_bf16(__uint_as_float(v[8 * k + 2]) * scale, __uint_as_float(v[8 * k + 3]) * scale),
                          pack_bf16(__uint_as_float(v[8 * k + 4]) * scale, __uint_as_float(v[8 * k + 5]) * scale),
                          pack_bf16(__uint_as_float(v[8 * k + 6]) * scale, __uint_as_float(v[8 * k + 7]) * scale));
  } else {
    // one float4 per column group; the 32 rows of a warp write 512 contiguous bytes
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<float4*>(p.part_o + part_o_offset<D>(split, head, row, col0 + 4 * k, p.H, p.T)) =
          make_float4(__uint_as_float(v[4 * k]) * scale, __uint_as_float(v[4 * k + 1]) * scale,
                      __uint_as_float(v[4 * k + 2]) * scale, __uint_as_float(v[4 * k + 3]) * scale);
  }
}

// OR of a predicate over the 128 threads of the tail warps (named barrier 1): every
// tail thread must call it the same number of times.
__device__ __forceinline__ bool tail_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tail_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int D, bool kDiag>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap kv_map) {
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t sQ0 = sbase + C::kQ0, sQ1 = sbase + C::kQ1, sQ2 = sbase + C::kQ2, sP2 = sbase + C::kP2;
  auto sK = [&](int st) { return sbase + uint32_t(C::k_off(st)); };
  auto sV = [&](int st) { return sbase + uint32_t(C::v_off(st)); };    // V, column block 0
  auto sV1 = [&](int st) { return sbase + uint32_t(C::v1_off(st)); };  // V, column block 1 (D = 128)
  const uint32_t bars = sbase + C::kBars;
  auto full_bar = [&](int st) { return bars + 8 * st; };
  auto empty_bar = [&](int st) { return bars + 8 * (S + st); };
  const uint32_t q_full = bars + 8 * (2 * S);
  // head_dim 64 uses s_full / p_ready per (tile, half buffer); head_dim 128 buffer 0 only
  auto s_full = [&](int t, int b) { return q_full + 8 * (1 + 2 * t + b); };
  auto s_free = [&](int t) { return q_full + 8 * (5 + t); };
  auto p_ready = [&](int t, int b) { return q_full + 8 * (7 + 2 * t + b); };
  auto pv_done = [&](int t) { return q_full + 8 * (11 + t); };
  auto o_done = [&](int t) { return q_full + 8 * (13 + t); };
  const uint32_t s2_full = q_full + 8 * 16, s2_free = q_full + 8 * 17;
  auto p2_ready = [&](int b) { return q_full + 8 * (18 + b); };
  const uint32_t pv2_done = q_full + 8 * 20;
  // head_dim 128: K and V of a stage land and are released separately.  K is read only
  // by the chunk's Q K^T (and the tail's S2^T), V until its last PV, so the next chunk's K
  // can be requested about a period earlier than the stage as a whole; with two stages
  // that had bound the chunk period.
  constexpr bool kSplitKV = C::kSplitV;
  auto v_full = [&](int st) { return kSplitKV ? q_full + 8 * (21 + st) : full_bar(st); };
  auto v_empty = [&](int st) { return kSplitKV ? q_full + 8 * (21 + S + st) : empty_bar(st); };
  constexpr bool kEarly = C::kEarly;
  const uint32_t sOnes = sbase + C::kOnesBlk;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int x = blockIdx.x;
  const int group = x % p.ngroups;
  x /= p.ngroups;
  const int head = x % p.H;
  const int split = x / p.H;
  const WorkDesc work = p.works[split];
  const int c0 = work.chunk_begin;
  const int n = work.chunk_end - work.chunk_begin;
  const int row0 = group * 2 * kTileRows;
  const int n_main = min(2, p.main_tiles - 2 * group);
  const bool has_tail = group == p.ngroups - 1 && p.tail_rows > 0;
  const int tail_row0 = p.main_tiles * kTileRows;
  const long long limit = p.wait_limit_ns;
  bool dump = false;
  if constexpr (kDiag) dump = p.dump_scores != nullptr;
  const float sl2 = p.scale_log2;

  if (threadIdx.x == 0) {
    const int ncons = max(1, n_main + (has_tail ? 1 : 0));
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), ncons);  // one release per consumer of the chunk
      if (kSplitKV) {
        ptx::mbar_init(v_full(i), 1);
        ptx::mbar_init(v_empty(i), ncons);
      }
    }
    ptx::mbar_init(q_full, kSoftmaxThreads);
    for (int t = 0; t < 2; ++t) {
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(s_full(t, b), 1);
        ptx::mbar_init(p_ready(t, b), 128);
      }
      ptx::mbar_init(s_free(t), 128);
      ptx::mbar_init(pv_done(t), 1);
    }
    for (int t = 0; t < 3; ++t) ptx::mbar_init(o_done(t), 1);
    ptx::mbar_init(s2_full, 1);
    ptx::mbar_init(s2_free, 128);
    for (int b = 0; b < 2; ++b) ptx::mbar_init(p2_ready(b), 128);
    ptx::mbar_init(pv2_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as a programmatic dependent: the set-up above overlaps the previous kernel;
  // Q, the pool and the outputs are touched only once that kernel (and with it
  // everything before) has completed.  The plan tables read above come from a copy,
  // which no launch overlaps.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the merge kernel that follows may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&kv_map);
      int issued = 0;
      bool k_only_last = false;
      const int nload = dump ? min(n, 1) : n;
      for (int i = 0; i < nload; ++i) {
        const int st = i % S;
        if (!ptx::mbar_wait_bounded(empty_bar(st), ((i / S) & 1) ^ 1, limit, abort_flag)) {
          signal_abort(p.status, abort_flag);
          break;
        }
        const ChunkDesc cd = p.chunks[c0 + i];
        const int start = cd.start_len & 0xFFFF;
        ptx::mbar_arrive_expect_tx(full_bar(st), (kSplitKV ? 1 : 2) * C::kTile);
        trace<kDiag>(p, kTrTmaIssue, i);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          ptx::tma_load_4d(sK(st) + cb * kColBlockBytes, &kv_map, cb * 64, head, start, 2 * cd.page, full_bar(st));
        bool v_ok = true;
        if (kSplitKV) {  // V once the stage's previous V is released
          v_ok = ptx::mbar_wait_bounded(v_empty(st), ((i / S) & 1) ^ 1, limit, abort_flag);
          if (v_ok) ptx::mbar_arrive_expect_tx(v_full(st), C::kTile);
        }
        if (v_ok) {
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb)
            ptx::tma_load_4d(cb ? sV1(st) : sV(st), &kv_map, cb * 64, head, start, 2 * cd.page + 1, v_full(st));
        }
        ++issued;
        if (!v_ok) {  // this chunk's K is in flight (the drain waits for it), its V is not
          k_only_last = true;
          signal_abort(p.status, abort_flag);
          break;
        }
      }
      // drain: copies must land before exit
      for (int i = issued > S ? issued - S : 0; i < issued; ++i) {
        ptx::mbar_wait_bounded(full_bar(i % S), (i / S) & 1, limit, nullptr);
        if (kSplitKV && !(k_only_last && i == issued - 1))
          ptx::mbar_wait_bounded(v_full(i % S), (i / S) & 1, limit, nullptr);
      }
    } else if (kDiag && lane == 1 && p.trace != nullptr && blockIdx.x == 0) {
      // trace mode: watch the full barriers and record when each chunk's K/V lands
      for (int i = 0; i < n; ++i)
        if (ptx::mbar_wait_bounded(full_bar(i % S), (i / S) & 1, limit, abort_flag)) trace<kDiag>(p, kTrLanded, i);
    }
    __syncwarp();
  } else if (warp >= kWarpMma) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per consumer: warp 13 main tile 0, warp 14 main tile 1,
    // warp 15 the tail.  Shared-memory descriptors are built once, split into a
    // constant high word (stride, version, 128-byte swizzle) and a low word (start
    // address >> 4, leading offset); a k-step only adds a constant to the low word.
    const int t = warp - kWarpMma;
    const bool mine = (t < 2) ? (t < n_main) : has_tail;
    if (lane == 0 && mine) {
      const uint32_t hi = uint32_t(ptx::smem_desc_sw128(sbase, 16, 1024) >> 32);
      auto k_lo_of = [&](int st) { return uint32_t(ptx::smem_desc_sw128(sK(st), 16, 1024)); };
      // V as an MN-major operand: the leading offset is the distance to the next 64-column
      // block (D = 64: the ones block; D = 128: V's second block, the ones block one more
      // stride on)
      auto v_lo_of = [&](int st) {
        return uint32_t(ptx::smem_desc_sw128(sV(st), C::kSplitV ? sV1(st) - sV(st) : sOnes - sV(st), 1024));
      };
      constexpr uint32_t kHalfRows = (kHalfKeys * 128) >> 4;     // 64 key rows of a K or V column block
      bool ok = ptx::mbar_wait_bounded(q_full, 0, limit, abort_flag);
      ptx::tc_fence_after();
      if (t < 2) {
        constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, kHalfKeys, 0, 0);
        constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, C::kOW, 0, 1);
        const uint32_t q_lo = uint32_t(ptx::smem_desc_sw128(t ? sQ1 : sQ0, 16, 1024));
        const uint32_t tQ = tmem + (t ? C::kTQ1 : C::kTQ0);
        const uint32_t tO = tmem + (t ? C::kO1 : C::kO0);
        const int halves = dump ? min(2 * n, 2) : 2 * n;
        // S = Q_t K^T over the 64 keys of half chunk g, into the buffer of half g
        auto issue_qk = [&](int g) -> bool {
          const int c = g >> 1, st = c % S;
          if ((g & 1) == 0) {
            if (!ptx::mbar_wait_bounded(full_bar(st), (c / S) & 1, limit, abort_flag)) return false;
            ptx::tc_fence_after();
            if (t == 0) trace<kDiag>(p, kTrFullSeen, c);
          }
          const uint32_t k_lo = k_lo_of(st) + uint32_t(g & 1) * kHalfRows;
          const uint32_t tS = tmem + s_col<D>(t, g & 1);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = uint32_t((k >> 2) * (kColBlockBytes >> 4) + (k & 3) * 2);
            if constexpr (C::kQTmem) {
              // A = Q_t from TMEM: a k-step is 16 dims, 8 columns of bf16 pairs
              ptx::mma_ts_lh(tS, tQ + 8 * k, k_lo + off, hi, idesc_qk, k > 0 ? 1u : 0u);
            } else {
              if (k == 0) ptx::mma_ss_lh<0>(tS, q_lo + off, k_lo + off, hi, idesc_qk);
              else ptx::mma_ss_lh<1>(tS, q_lo + off, k_lo + off, hi, idesc_qk);
            }
          }
          ptx::mma_commit(s_full(t, kEarly ? 0 : (g & 1)));
          if (kSplitKV && (g & 1)) ptx::mma_commit(empty_bar(st));  // the chunk's K is read
          if (t == 0) trace<kDiag>(p, (g & 1) ? kTrQk0h1 : kTrQk0, c);
          else if ((g & 1) == 0) trace<kDiag>(p, kTrQk1, c);
          return true;
        };
        // O_t (+)= P V over the 64 keys of half g: a k-step is 16 key rows (2 KB) of V and 8
        // TMEM columns of packed P
        auto issue_pv = [&](int g) -> bool {
          const int b = g & 1, c = g >> 1, st = c % S;
          if (kSplitKV && b == 0) {
            if (!ptx::mbar_wait_bounded(v_full(st), (c / S) & 1, limit, abort_flag)) return false;
            ptx::tc_fence_after();
          }
          const uint32_t v_lo = v_lo_of(st) + uint32_t(b) * kHalfRows;
          const uint32_t tP = tmem + p_col<D>(t, b);
#pragma unroll
          for (int k = 0; k < kHalfKeys / 16; ++k)
            ptx::mma_ts_lh(tO, tP + 8 * k, v_lo + uint32_t(128 * k), hi, idesc_pv, (g > 0 || k > 0) ? 1u : 0u);
          ptx::mma_commit(pv_done(t));
          if (b) {
            ptx::mma_commit(v_empty(st));  // this consumer is done with the stage (its V)
            if (t == 0) trace<kDiag>(p, kTrEmpty, c);
          }
          return true;
        };
        auto wait_p = [&](int g) -> bool {
          const int b = g & 1, c = g >> 1;
          if (!ptx::mbar_wait_bounded(p_ready(t, kEarly ? 0 : b), kEarly ? (g & 1) : (c & 1), limit, abort_flag))
            return false;
          ptx::tc_fence_after();
          if (t == 0) trace<kDiag>(p, b ? kTrP0h1Seen : kTrP0Seen, c);
          else if (b == 0) trace<kDiag>(p, kTrP1Seen, c);
          return true;
        };
        if constexpr (kEarly) {
          // one S buffer: Q K^T of half g+1 as soon as the softmax has loaded half g
          if (halves > 0) ok = ok && issue_qk(0);
          for (int g = 0; ok && g < halves; ++g) {
            if (g + 1 < halves) {
              if (!(ok = ptx::mbar_wait_bounded(s_free(t), g & 1, limit, abort_flag))) break;
              ptx::tc_fence_after();
              if (!(ok = issue_qk(g + 1))) break;
            }
            if (dump) continue;
            if (!(ok = wait_p(g))) break;
            if (!(ok = issue_pv(g))) break;
          }
        } else {
          // two S buffers: Q K^T of half g+2 into the buffer the PV of half g reads (in order)
          for (int g = 0; ok && g < min(halves, 2); ++g) ok = issue_qk(g);
          for (int g = 0; ok && !dump && g < halves; ++g) {
            if (!(ok = wait_p(g))) break;
            if (!(ok = issue_pv(g))) break;
            if (g + 2 < halves) ok = issue_qk(g + 2);
          }
        }
      } else {
        // Tail: S2^T = K Q2^T (M = 128 keys, N = 16, K = D) into one TMEM buffer, then
        // O2^T (+)= V^T P2^T (M = D columns of V, N = kTailPvN rows, K = 128 keys): A = V^T
        // read MN-major from the V tile, B = P2^T K-major from shared memory.  With M = 64
        // the accumulator's rows (V columns) 16q..16q+15 live in TMEM lanes 32q..32q+15;
        // with M = 128 row i lives in lane i.
        constexpr uint32_t idesc_st = ptx::idesc_bf16_f32(128, kTailN, 0, 0);
        constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(D, C::kTailPvN, 1, 0);
        const uint32_t q2_lo = uint32_t(ptx::smem_desc_sw128(sQ2, 16, 1024));
        const uint32_t p2_lo = uint32_t(ptx::smem_desc_sw128(sP2, 16, 1024));
        const uint32_t tS2 = tmem + C::kS2, tO2 = tmem + C::kO2;
        const int nmma = dump ? 0 : n;
        auto issue_st = [&](int c) -> bool {
          const int st = c % S;
          if (!ptx::mbar_wait_bounded(full_bar(st), (c / S) & 1, limit, abort_flag)) return false;
          ptx::tc_fence_after();
          const uint32_t k_lo = k_lo_of(st);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t aoff = uint32_t((k >> 2) * (kColBlockBytes >> 4) + (k & 3) * 2);
            const uint32_t boff = uint32_t((k >> 2) * (C::kQ2ColBlock >> 4) + (k & 3) * 2);
            if (k == 0) ptx::mma_ss_lh<0>(tS2, k_lo, q2_lo, hi, idesc_st);
            else ptx::mma_ss_lh<1>(tS2, k_lo + aoff, q2_lo + boff, hi, idesc_st);
          }
          ptx::mma_commit(s2_full);
          if (kSplitKV) ptx::mma_commit(empty_bar(st));  // the tail is done with the chunk's K
          trace<kDiag>(p, kTrQk2, c);
          return true;
        };
        if (nmma > 0 && ok) ok = issue_st(0);
        for (int c = 0; ok && c < nmma; ++c) {
          const int st = c % S;
          if (c + 1 < nmma) {
            // the single S2^T buffer is free once the tail warps have loaded chunk c's scores
            if (!(ok = ptx::mbar_wait_bounded(s2_free, c & 1, limit, abort_flag))) break;
            ptx::tc_fence_after();
            if (!(ok = issue_st(c + 1))) break;
          }
          if (!(ok = ptx::mbar_wait_bounded(p2_ready(c & 1), (c >> 1) & 1, limit, abort_flag))) break;
          ptx::tc_fence_after();
          trace<kDiag>(p, kTrP2Seen, c);
          if (kSplitKV) {
            if (!(ok = ptx::mbar_wait_bounded(v_full(st), (c / S) & 1, limit, abort_flag))) break;
            ptx::tc_fence_after();
          }
          const uint32_t v_lo = v_lo_of(st);
          const uint32_t b_lo = p2_lo + uint32_t((c & 1) * (C::kP2Bytes >> 4));
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t boff = uint32_t((k >> 2) * (C::kP2ColBlock >> 4) + (k & 3) * 2);
            if (c == 0 && k == 0) ptx::mma_ss_lh<0>(tO2, v_lo, b_lo, hi, idesc_pv);
            else ptx::mma_ss_lh<1>(tO2, v_lo + uint32_t(128 * k), b_lo + boff, hi, idesc_pv);
          }
          ptx::mma_commit(pv2_done);
          ptx::mma_commit(v_empty(st));
        }
      }
      if (!ok) signal_abort(p.status, abort_flag);
      ptx::mma_commit(o_done(t));  // arrives once every MMA this thread issued has completed
      ptx::mbar_wait_bounded(o_done(t), 0, limit, nullptr);
    }
    __syncwarp();
  } else if (warp >= kWarpMain) {
    // ------------------------------------------------------------ main-tile softmax
    const int t = (warp - kWarpMain) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int row = row0 + t * kTileRows + r;
    const bool tile_on = t < n_main;
    const bool row_ok = tile_on && row < p.T;
    const bool warp_on = tile_on && row0 + t * kTileRows + q4 * 32 < p.T;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const uint32_t tO = tmem + (t ? C::kO1 : C::kO0) + lane_off;
    const int64_t qrow = int64_t(work.stream) * p.T + row;
    const uint4* qsrc =
        reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + (qrow * p.H + head) * D);
    if (tile_on) {
      if constexpr (C::kQTmem) {
        // this row of Q into TMEM lane r: column j holds dims 2j (low half) and 2j + 1
        uint32_t qv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = row_ok ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
          qv[4 * c] = v.x;
          qv[4 * c + 1] = v.y;
          qv[4 * c + 2] = v.z;
          qv[4 * c + 3] = v.w;
        }
        ptx::tmem_st32(tmem + (t ? C::kTQ1 : C::kTQ0) + lane_off, qv);
        ptx::tmem_wait_st();
      } else {
        store_q_row<D>(t ? sQ1 : sQ0, r, qsrc, row_ok);
      }
    }
    {  // the ones block: 16 KB over the 256 main-softmax threads
      const uint32_t ones = 0x3F803F80u;  // two bf16 1.0
#pragma unroll
      for (int i = 0; i < 4; ++i)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sOnes + uint32_t(((i * 256) + (threadIdx.x - 128)) * 16)),
                     "r"(ones)
                     : "memory");
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::mbar_arrive(q_full);

    if (tile_on && dump) {
      if constexpr (kDiag) {
        // the first chunk's two halves of scores, as the tensor core wrote them
        float* dst = p.dump_scores + ((int64_t(blockIdx.x) * 2 + t) * 128 + r) * 128;
        for (int b = 0; b < 2 && b < 2 * n; ++b) {
          if (!ptx::mbar_wait_warp(s_full(t, kEarly ? 0 : b), kEarly ? b : 0, limit, abort_flag)) break;
          ptx::tc_fence_after();
          uint32_t sd[2][32];
          const uint32_t tS = tmem + s_col<D>(t, b) + lane_off;
          ptx::tmem_ld32(tS, sd[0]);
          ptx::tmem_ld32(tS + 32, sd[1]);
          ptx::tmem_wait_ld();
          if constexpr (kEarly) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(s_free(t));
          }
          for (int j = 0; j < 2; ++j)
            for (int e = 0; e < 32; ++e) dst[kHalfKeys * b + 32 * j + e] = __uint_as_float(sd[j][e]);
        }
      }
    } else if (tile_on) {
      float m = -INFINITY;  // running max of scaled logits (log2 units); the first half sets it
      bool ok = true;
      int len = 0;
      int len_next = n > 0 ? (__ldg(&p.chunks[c0].start_len) >> 16) : 0;
      for (int g = 0; ok && g < 2 * n; ++g) {
        const int b = g & 1;
        if (b == 0) {
          len = len_next;
          if ((g >> 1) + 1 < n) len_next = __ldg(&p.chunks[c0 + (g >> 1) + 1].start_len) >> 16;
        }
        if (!(ok = ptx::mbar_wait_warp(s_full(t, kEarly ? 0 : b), kEarly ? (g & 1) : ((g >> 1) & 1), limit,
                                       abort_flag)))
          break;
        ptx::tc_fence_after();
        if (q4 == 0 && lane == 0) trace<kDiag>(p, t ? kTrS1Seen : (b ? kTrS0h1Seen : kTrS0Seen), g >> 1);
        const uint32_t tS = tmem + s_col<D>(t, b) + lane_off;
        uint32_t sa[32], sb[32], pk[32];
        ptx::tmem_ld32(tS, sa);
        ptx::tmem_ld32(tS + 32, sb);
        ptx::tmem_wait_ld();
        if constexpr (kEarly) {  // the scores are in registers: the buffer goes back to the issuer
          ptx::tc_fence_before();
          ptx::mbar_arrive(s_free(t));
        }
        bool waited_pv = g == 0;  // the previous half's PV (none before half 0)
        bool p_stored = false;
        if (warp_on) {
          // exponentiated against the running max m; only when some P value reaches 2 (the
          // first half, and rare jumps of the max) does the warp take the path that moves
          // m, rescales O and recomputes this half's P
          mask32(sa, kHalfKeys * b, len);
          mask32(sb, kHalfKeys * b + 32, len);
          uint32_t orr;
          exp_pack64(sa, sb, sl2, -m, pk, &orr);
          const bool need = (orr & kPHighBits) != 0;
          if (__any_sync(0xffffffffu, need)) {
            float2 r2;
            if constexpr (kEarly) {
              r2 = move_running_max_regs(sa, sb, pk, tO, g > 0 ? C::kOW : 0, need, m, sl2, pv_done(t),
                                         uint32_t(g - 1) & 1u, limit, abort_flag);
            } else {
              r2 = move_running_max_tmem(tO, tS, g > 0 ? C::kOW : 0, need, m, sl2, kHalfKeys * b, len, pv_done(t),
                                         uint32_t(g - 1) & 1u, limit, abort_flag);
              p_stored = true;
            }
            m = r2.x;
            waited_pv = true;
            if constexpr (kDiag)  // diagnostics: count rescales of an accumulated O (any CTA)
              if (p.trace != nullptr && g > 0 && lane == 0) atomicAdd(p.trace + int64_t(kTraceEvents) * p.trace_cap, 1ull);
            if (r2.y == 0.f) {
              ok = false;
              break;
            }
          }
          if (!kEarly && !p_stored) {  // P over the scores it came from
            ptx::tmem_st32(tS, pk);
            ptx::tmem_wait_st();
          }
        }
        if constexpr (kEarly) {
          // the tile's P buffer: the previous half's PV must have read it
          if (!waited_pv && !(ok = ptx::mbar_wait_warp(pv_done(t), uint32_t(g - 1) & 1u, limit, abort_flag))) break;
          ptx::tc_fence_after();
          if (warp_on) {
            ptx::tmem_st32(tmem + p_col<D>(t, b) + lane_off, pk);
            ptx::tmem_wait_st();
          }
        }
        if (len < kHalfKeys * (b + 1)) {
          // ragged chunk: zero this half's V rows past the valid keys before the PV reads them
          // (head_dim 128: once the chunk's V, which lands apart from K, is there)
          const int c = g >> 1;
          if (kSplitKV && !(ok = ptx::mbar_wait_warp(v_full(c % S), (c / S) & 1, limit, abort_flag))) break;
          zero_v_rows<D>(sV(c % S), sV1(c % S), max(len, kHalfKeys * b), kHalfKeys * (b + 1), r, 128);
          ptx::fence_proxy_async_smem();
        }
        ptx::tc_fence_before();
        // an arrive releases this thread's earlier writes, so the trace store follows it
        long long t_arrive = 0;
        if constexpr (kDiag) t_arrive = clock64();
        ptx::mbar_arrive(p_ready(t, kEarly ? 0 : b));
        if (q4 == 0 && lane == 0 && (t == 0 || b == 0))
          trace_at<kDiag>(p, t ? kTrP1Arrive : (b ? kTrP0h1Arrive : kTrP0Arrive), g >> 1, t_arrive);
      }
      if (!ok) signal_abort(p.status, abort_flag);
      if (ok && ptx::mbar_wait_warp(o_done(t), 0, limit, abort_flag) && warp_on) {
        ptx::tc_fence_after();
        uint32_t lv[16];  // the row sum, as accumulated by the PV MMA
        ptx::tmem_ld16(tO + D, lv);
        ptx::tmem_wait_ld();
        const float l = __uint_as_float(lv[0]);
        const float inv_l = 1.f / l;
#pragma unroll 1
        for (int j = 0; j < D / 32; ++j) {
          uint32_t v[32];
          ptx::tmem_ld32(tO + 32 * j, v);
          ptx::tmem_wait_ld();
          if (row_ok) store_output_cols<D>(p, work, split, head, row, v, 32 * j, inv_l);
        }
        if (row_ok && work.nsplit > 1) p.part_lse[(int64_t(split) * p.H + head) * p.T + row] = m + __log2f(l);
      }
    }
  } else {
    // ------------------------------------------------------------ tail softmax (warps 0-3)
    const int q = warp;  // key group [32q, 32q+32) of each chunk; TMEM lane quarter q
    const int tid = q * 32 + lane;
    const int tail_rows = p.tail_rows;
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t tS2 = tmem + C::kS2 + lane_off;
    const uint32_t tO2 = tmem + C::kO2 + lane_off;
    // exchange area: [2][4 warps][8 rows] maxima, then [2][4 warps] "waits succeeded" flags
    float* xmax = reinterpret_cast<float*>(smem + C::kTailX);
    int* xok = reinterpret_cast<int*>(xmax + 2 * 4 * kTailMaxRows);
    if (has_tail) {
      // zero both P tiles (rows past tail_rows stay zero), then stage the tail's Q rows
      // (rows past tail_rows are zero) as the B operand of S2^T: 16 rows, D/64 column blocks
      for (int i = tid; i < 2 * C::kP2Bytes / 16; i += 128) st_shared_zero16(sP2 + uint32_t(i * 16));
      for (int u = tid; u < kTailN * (D / 8); u += 128) {
        const int qr = u / (D / 8), qc = u % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (qr < tail_rows) {
          const int64_t qrow = int64_t(work.stream) * p.T + tail_row0 + qr;
          v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + (qrow * p.H + head) * D) +
                    qc);
        }
        const uint32_t dst = sQ2 + uint32_t((qc >> 3) * C::kQ2ColBlock + (qr >> 3) * 1024 + (qr & 7) * 128 +
                                            (((qc & 7) ^ (qr & 7)) << 4));
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(q_full);
    if (has_tail && !dump) {
      // per row r: m[r] the running max (log2 units; the same in all four warps), l[r]
      // this lane's share of the row sum of the rounded P
      float m[kTailMaxRows], l[kTailMaxRows];
#pragma unroll
      for (int rr = 0; rr < kTailMaxRows; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
      }
      // Every tail thread passes the same barriers in every chunk, whatever its waits
      // returned, so no warp can be left waiting at a barrier another one skipped; a
      // failed wait ends the loop of all four warps at the next exchange.
      bool ok = true;
      const int key = 32 * q + lane;
      int len_next = n > 0 ? (__ldg(&p.chunks[c0].start_len) >> 16) : 0;
      for (int j = 0; j < n; ++j) {
        const int len = len_next;
        if (j + 1 < n) len_next = __ldg(&p.chunks[c0 + j + 1].start_len) >> 16;
        const bool okj = ok && ptx::mbar_wait_warp(s2_full, j & 1, limit, abort_flag);
        float xs[kTailMaxRows];
        bool need = false;
        if (okj) {
          ptx::tc_fence_after();
          if (q == 0 && lane == 0) trace<kDiag>(p, kTrS2Seen, j);
          uint32_t s[16];
          ptx::tmem_ld16(tS2, s);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(s2_free);  // the issuer may now write the next chunk's S2^T
          const bool valid = key < len;
#pragma unroll
          for (int rr = 0; rr < kTailMaxRows; ++rr) {
            xs[rr] = valid ? __uint_as_float(s[rr]) * sl2 : -INFINITY;
            if (rr < tail_rows && xs[rr] > m[rr] + kThreshold) need = true;
          }
        } else {
#pragma unroll
          for (int rr = 0; rr < kTailMaxRows; ++rr) xs[rr] = -INFINITY;
        }
        if (tail_bar_or(need || !okj)) {
          // rare: a running max moves (or a wait failed): each warp's maxima and status
          // through shared memory, double-buffered by chunk parity
          float* xm = xmax + (j & 1) * 4 * kTailMaxRows;
#pragma unroll
          for (int rr = 0; rr < kTailMaxRows; ++rr) {
            const float wm = warp_max(xs[rr]);
            if (lane == rr) xm[q * kTailMaxRows + rr] = wm;
          }
          if (lane == 0) xok[(j & 1) * 4 + q] = okj ? 1 : 0;
          tail_bar_sync();
          if (!(xok[(j & 1) * 4] && xok[(j & 1) * 4 + 1] && xok[(j & 1) * 4 + 2] && xok[(j & 1) * 4 + 3])) {
            ok = false;
            break;  // all four warps read the same flags and leave together
          }
          float corr[kTailMaxRows];
#pragma unroll
          for (int rr = 0; rr < kTailMaxRows; ++rr) {
            float mx = m[rr];
#pragma unroll
            for (int g = 0; g < 4; ++g) mx = fmaxf(mx, xm[g * kTailMaxRows + rr]);
            corr[rr] = mx == m[rr] ? 1.f : ptx::ex2(m[rr] - mx);  // 0 while m is -inf
            l[rr] *= corr[rr];
            m[rr] = mx;
          }
          if (j > 0) {  // O2^T must first hold the previous chunk's PV
            if (!ptx::mbar_wait_warp(pv2_done, uint32_t(j - 1) & 1u, limit, abort_flag)) {
              ok = false;  // reported at the next chunk's exchange (or after the loop)
              continue;
            }
            ptx::tc_fence_after();
            uint32_t o[8];
            ptx::tmem_ld8(tO2, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int rr = 0; rr < kTailMaxRows; ++rr) o[rr] = __float_as_uint(__uint_as_float(o[rr]) * corr[rr]);
            ptx::tmem_st8(tO2, o);
            ptx::tmem_wait_st();
            if constexpr (kDiag)
              if (p.trace != nullptr && lane == 0) atomicAdd(p.trace + int64_t(kTraceEvents) * p.trace_cap + 1, 1ull);
          }
        }
        const uint32_t p2 = sP2 + uint32_t((j & 1) * C::kP2Bytes);
#pragma unroll
        for (int rr = 0; rr < kTailMaxRows; ++rr) {
          if (rr < tail_rows) {
            const __nv_bfloat16 pb = __float2bfloat16_rn(ptx::ex2(xs[rr] - m[rr]));
            l[rr] += __bfloat162float(pb);
            st_shared_u16(p2_addr(p2, C::kP2ColBlock, rr, key), __bfloat16_as_ushort(pb));
          }
        }
        if (len < kChunkTokens) {
          // head_dim 128: the chunk's V lands apart from K; a failed wait skips the zeroing
          // and is reported at the next chunk's exchange (or after the loop)
          if (!kSplitKV || ptx::mbar_wait_warp(v_full(j % S), (j / S) & 1, limit, abort_flag))
            zero_v_rows<D>(sV(j % S), sV1(j % S), len, kChunkTokens, tid, 128);
          else
            ok = false;
        }
        ptx::fence_proxy_async_smem();  // P2 stores (and zeroed V rows) -> visible to the tensor core
        ptx::tc_fence_before();
        long long t_arrive = 0;
        if constexpr (kDiag) t_arrive = clock64();
        ptx::mbar_arrive(p2_ready(j & 1));
        if (q == 0 && lane == 0) trace_at<kDiag>(p, kTrP2Arrive, j, t_arrive);
      }
      if (!ok) signal_abort(p.status, abort_flag);
      // Row sums over all 128 keys of every chunk: each warp's share through shared
      // memory.  The exchange reuses the K/V stage ring, so it is written only once every
      // consumer's MMAs (and with them every load of this CTA) have completed.
      float* scratch = reinterpret_cast<float*>(smem + C::kKV);
      bool done = ok;
      for (int u = 0; u < 3 && done; ++u)
        if (u == 2 || u < n_main) done = ptx::mbar_wait_warp(o_done(u), 0, limit, abort_flag);
      if (done) {
#pragma unroll
        for (int rr = 0; rr < kTailMaxRows; ++rr) {
          const float lt = warp_sum(l[rr]);
          if (lane == 0) scratch[q * kTailMaxRows + rr] = lt;
        }
      }
      tail_bar_sync();
      if (done && !*abort_flag) {
        ptx::tc_fence_after();
        uint32_t o[8];
        ptx::tmem_ld8(tO2, o);  // this lane's column of V (see below), the first 8 rows
        ptx::tmem_wait_ld();
        // M = 64: lanes 0-15 of quarter q hold V columns 16q..16q+15; M = 128: lane i of
        // quarter q holds column 32q + i
        constexpr int kLanesUsed = D == 64 ? 16 : 32;
        if (lane < kLanesUsed) {
          const int d = kLanesUsed * q + lane;
#pragma unroll
          for (int rr = 0; rr < kTailMaxRows; ++rr) {
            if (rr < tail_rows) {
              const float L = (scratch[rr] + scratch[kTailMaxRows + rr]) +
                              (scratch[2 * kTailMaxRows + rr] + scratch[3 * kTailMaxRows + rr]);
              const float val = __uint_as_float(o[rr]) / L;
              const int orow = tail_row0 + rr;
              if (work.nsplit == 1) {
                const int64_t qr = int64_t(work.stream) * p.T + orow;
                static_cast<__nv_bfloat16*>(p.out)[(qr * p.H + head) * D + d] = __float2bfloat16_rn(val);
              } else {
                p.part_o[part_o_offset<D>(split, head, orow, d, p.H, p.T)] = val;
                if (d == 0) p.part_lse[(int64_t(split) * p.H + head) * p.T + orow] = m[rr] + __log2f(L);
              }
            }
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kDiag>
cudaError_t configure_tc() {
  return cudaFuncSetAttribute(attention_tc_kernel<D, kDiag>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<D>::kLaunch);
}

template <int D>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap* map, cudaStream_t s) {
  constexpr int smem = Cfg<D>::kLaunch;
  const int64_t grid = int64_t(p.num_splits) * p.H * p.ngroups;
  if (grid <= 0 || grid > 0x7fffffff) return cudaErrorInvalidValue;
  if (p.trace != nullptr || p.dump_scores != nullptr)
    return launch_dependent(attention_tc_kernel<D, true>, dim3(unsigned(grid)), dim3(kThreads), smem, s, p, *map);
  return launch_dependent(attention_tc_kernel<D, false>, dim3(unsigned(grid)), dim3(kThreads), smem, s, p, *map);
}

}  // namespace

cudaError_t configure_attention_bf16() {
  cudaError_t e;
  if ((e = configure_tc<64, false>()) != cudaSuccess) return e;
  if ((e = configure_tc<64, true>()) != cudaSuccess) return e;
  if ((e = configure_tc<128, false>()) != cudaSuccess) return e;
  return configure_tc<128, true>();
}

cudaError_t launch_attention_bf16(const AttnParams& p, const CUtensorMap* kv_map, cudaStream_t s) {
  return p.D == 64 ? launch_tc<64>(p, kv_map, s) : launch_tc<128>(p, kv_map, s);
}

TileShape attention_bf16_tiles(int T, int head_dim) {
  TileShape ts{};
  const int full = T / kTileRows, rem = T % kTileRows;
  if (rem > 0 && rem <= kTailMaxRows) {
    ts.main_tiles = full;
    ts.tail_rows = rem;
  } else {
    ts.main_tiles = full + (rem > 0 ? 1 : 0);
    ts.tail_rows = 0;
  }
  ts.ngroups = ts.main_tiles > 0 ? (ts.main_tiles + 1) / 2 : 1;
  return ts;
}

}  // namespace spk
