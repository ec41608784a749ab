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
// 128-row "main" tiles, plus, on the last group when head_dim is 64, a "tail" of at
// most 32 trailing rows (262 = 2 x 128 + 6).  Warp roles (16 warps):
//   warps 0-3   tail softmax.  The tail's Q rows are replicated in the four TMEM
//               lane quarters; warp q owns keys [16q, 16q+16) of every 64-key half
//               chunk, so the tail's exponentials are spread evenly over the four
//               SM sub-partitions.  Each warp keeps its own (max, sum, O) and the
//               four partial states are merged at the end.
//   warps 4-7   softmax of main tile 0, warps 8-11 softmax of main tile 1: one
//               thread per query row (= TMEM lane).  fp32 online softmax in log2
//               units, masking of the chunk's ragged tail, P written back as bf16
//               over S, row sums taken from the rounded P that the MMA consumes,
//               O rescaled in TMEM only when the running maximum grows by > 2^8.
//   warp 12     TMA producer: K and V chunk tiles gathered by page id through a
//               4-D tensor map over the pool (d, head, token, 2*page+kv), 128-byte
//               swizzle, into a ring of shared-memory stages.
//   warps 13-15 MMA issuers, one thread per consumer (main tile 0, main tile 1,
//               tail): S_t = Q_t K^T (M=128, N=128, K=D) and O_t += P_t V
//               (M=128, N=D, K=128); the tail works on 64-key halves (N=64, K=64).
//               The consumers advance independently, so one tile's MMAs run while
//               the other tile's softmax runs; a K/V stage is released once every
//               consumer is done with it.
// TMEM (512 columns): S0 | S1 | O0 | O1 [| S2 (64) | O2 (64) when D = 64].
// The epilogue writes bf16 output (one split) or an fp32 partial with its log2
// log-sum-exp (several splits, combined by the merge kernel).
// Every wait is bounded: on timeout the kernel records a status word, drains its
// own copies and MMAs, frees TMEM and returns.
#include "ptx_sm100.cuh"
#include "spk_internal.h"

#include <cuda_bf16.h>

#include <type_traits>

namespace spk {
namespace {

constexpr int kColBlockBytes = 128 * 128;  // 128 rows x 64 bf16: one 128-byte-swizzled column block
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kTailMaxRows = 32;
constexpr int kThreads = 512;
constexpr int kWarpMain = 4;   // first warp of main tile 0; tile 1 starts at 8
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;   // warps 13, 14, 15 issue the MMAs of main tile 0, main tile 1 and the tail
constexpr int kSoftmaxThreads = 384;  // warps 0-11 (all arrive on q_full)

template <int D>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;  // one Q, K or V tile in shared memory
  static constexpr bool kTail = (D == 64);
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTile;
  static constexpr int kQ2 = 2 * kTile;  // tail Q (D == 64)
  static constexpr int kKV = (kTail ? 3 : 2) * kTile;
  static constexpr int kStageBytes = 2 * kTile;
  static constexpr int kBars = kKV + kStages * kStageBytes;
  static constexpr int kNumBars = 2 * kStages + 10;  // full, empty, q_full, s_full[3], p_ready[3], o_done[3]
  static constexpr int kMisc = kBars + 8 * kNumBars;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kLaunch = kBytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kS0 = 0, kS1 = 128, kO0 = 256, kO1 = 256 + D;
  static constexpr uint32_t kS2 = 256 + 2 * D, kO2 = 256 + 2 * D + 64;  // D == 64 only
  static_assert(!kTail || kO2 + 64 <= 512, "TMEM budget");
  static_assert(kStages * kStageBytes >= 4 * kTailMaxRows * (64 + 2) * 4, "tail merge scratch");
};

// Trace mode (diagnostics): CTA 0 records the SM clock of an event for a chunk.
__device__ __forceinline__ void trace(const AttnParams& p, int ev, int chunk) {
  if (p.trace != nullptr && blockIdx.x == 0 && chunk < p.trace_cap)
    p.trace[int64_t(ev) * p.trace_cap + chunk] = clock64();
}

__device__ __forceinline__ void signal_abort(int32_t* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(status, kStatusWaitTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// sum of the two bf16 values held in a packed pair, in fp32
__device__ __forceinline__ float packed_sum(uint32_t pk) {
  return __uint_as_float(pk << 16) + __uint_as_float(pk & 0xFFFF0000u);
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

// p = 2^(s*sl2 - m) for N fp32 scores in registers, packed to bf16 pairs and stored to
// TMEM at column `dst`; returns the fp32 sum of the rounded values.  The argument is
// one packed fp32x2 FMA per pair and the sum adds the two bf16 halves directly.
template <int N>
__device__ __forceinline__ float exp_pack_store(const uint32_t* s, float sl2, float neg_m, uint32_t dst) {
  static_assert(N % 32 == 0, "");
  float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < N / 32; ++j) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float x0, x1;
      ptx::fma2(x0, x1, __uint_as_float(s[32 * j + 2 * e]), __uint_as_float(s[32 * j + 2 * e + 1]), sl2, neg_m);
      pk[e] = pack_bf16(ptx::ex2(x0), ptx::ex2(x1));
      sum[e & 3] = ptx::add_bf16x2_to(pk[e], sum[e & 3]);
    }
    ptx::tmem_st16(dst + 16 * j, pk);
  }
  return (sum[0] + sum[1]) + (sum[2] + sum[3]);
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

// Scale `ncols` TMEM columns of this warp's lanes by corr (per lane).
__device__ __forceinline__ void rescale_tmem(uint32_t taddr, int ncols, float corr) {
  for (int j = 0; j < ncols; j += 32) {
    uint32_t o[32];
    ptx::tmem_ld32(taddr + j, o);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
    ptx::tmem_st32(taddr + j, o);
  }
}

// Scale the bf16 pairs in packed TMEM columns [0, ncols) of this warp's lanes by corr.
__device__ __forceinline__ void rescale_packed_p(uint32_t taddr, int ncols, float corr) {
  for (int j = 0; j < ncols; j += 16) {
    uint32_t v[16];
    ptx::tmem_ld16(taddr + j, v);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e)
      v[e] = pack_bf16(__uint_as_float(v[e] << 16) * corr, __uint_as_float(v[e] & 0xFFFF0000u) * corr);
    ptx::tmem_st16(taddr + j, v);
  }
}

// Rare path of the online softmax (kept out of line so the hot loop's registers are
// not spent on it): scale the first o_cols columns of O and the first p_cols packed
// P columns of this chunk by corr.
__device__ __noinline__ void rescale_running(uint32_t tO, uint32_t tS, int o_cols, int p_cols, float corr) {
  if (o_cols) rescale_tmem(tO, o_cols, corr);
  if (p_cols) {
    ptx::tmem_wait_st();
    rescale_packed_p(tS, p_cols, corr);
  }
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
    const int64_t idx = (int64_t(split) * p.H + head) * p.T + row;
    float4* dst = reinterpret_cast<float4*>(p.part_o + idx * D + col0);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      dst[k] = make_float4(__uint_as_float(v[4 * k]) * scale, __uint_as_float(v[4 * k + 1]) * scale,
                           __uint_as_float(v[4 * k + 2]) * scale, __uint_as_float(v[4 * k + 3]) * scale);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap kv_map) {
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t sQ0 = sbase + C::kQ0, sQ1 = sbase + C::kQ1, sQ2 = sbase + C::kQ2;
  auto sK = [&](int st) { return sbase + C::kKV + st * C::kStageBytes; };
  auto sV = [&](int st) { return sbase + C::kKV + st * C::kStageBytes + C::kTile; };
  const uint32_t bars = sbase + C::kBars;
  auto full_bar = [&](int st) { return bars + 8 * st; };
  auto empty_bar = [&](int st) { return bars + 8 * (S + st); };
  const uint32_t q_full = bars + 8 * (2 * S);
  auto s_full = [&](int t) { return q_full + 8 * (1 + t); };
  auto p_ready = [&](int t) { return q_full + 8 * (4 + t); };
  auto o_done = [&](int t) { return q_full + 8 * (7 + t); };
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
  const bool has_tail = C::kTail && group == p.ngroups - 1 && p.tail_rows > 0;
  const int tail_row0 = p.main_tiles * kTileRows;
  const long long limit = p.wait_limit_ns;
  const bool dump = p.dump_scores != nullptr;
  const float sl2 = p.scale_log2;

  if (threadIdx.x == 0) {
    const int ncons = max(1, n_main + (has_tail ? 1 : 0));
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), ncons);  // one release per consumer of the chunk
    }
    ptx::mbar_init(q_full, kSoftmaxThreads);
    for (int t = 0; t < 3; ++t) {
      ptx::mbar_init(s_full(t), 1);
      ptx::mbar_init(p_ready(t), 128);
      ptx::mbar_init(o_done(t), 1);
    }
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

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&kv_map);
      int issued = 0;
      const int nload = dump ? min(n, 1) : n;
      for (int i = 0; i < nload; ++i) {
        const int st = i % S;
        if (!ptx::mbar_wait_bounded(empty_bar(st), ((i / S) & 1) ^ 1, limit, abort_flag)) {
          signal_abort(p.status, abort_flag);
          break;
        }
        const ChunkDesc cd = p.chunks[c0 + i];
        const int start = cd.start_len & 0xFFFF;
        ptx::mbar_arrive_expect_tx(full_bar(st), 2 * C::kTile);
        trace(p, kTrTmaIssue, i);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
          ptx::tma_load_4d(sK(st) + cb * kColBlockBytes, &kv_map, cb * 64, head, start, 2 * cd.page, full_bar(st));
          ptx::tma_load_4d(sV(st) + cb * kColBlockBytes, &kv_map, cb * 64, head, start, 2 * cd.page + 1,
                           full_bar(st));
        }
        ++issued;
      }
      for (int i = issued > S ? issued - S : 0; i < issued; ++i)  // drain: copies must land before exit
        ptx::mbar_wait_bounded(full_bar(i % S), (i / S) & 1, limit, nullptr);
    } else if (lane == 1 && p.trace != nullptr && blockIdx.x == 0) {
      // trace mode: watch the full barriers and record when each chunk's K/V lands
      for (int i = 0; i < n; ++i)
        if (ptx::mbar_wait_bounded(full_bar(i % S), (i / S) & 1, limit, abort_flag)) trace(p, kTrLanded, i);
    }
    __syncwarp();
  } else if (warp >= kWarpMma) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per consumer: warp 13 main tile 0, warp 14 main tile 1,
    // warp 15 the tail.  Each runs its consumer's chain in order: wait for the K/V
    // stage, S = Q K^T, commit; wait for P, O += P V, release the stage.  Shared-
    // memory descriptors are built once; a k-step only adds to the address field.
    const int t = warp - kWarpMma;
    const bool mine = (t < 2) ? (t < n_main) : has_tail;
    if (lane == 0 && mine) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_qk_half = ptx::idesc_bf16_f32(128, 64, 0, 0);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, D, 0, 1);
      const uint32_t tS = tmem + (t == 0 ? C::kS0 : t == 1 ? C::kS1 : C::kS2);
      const uint32_t tO = tmem + (t == 0 ? C::kO0 : t == 1 ? C::kO1 : C::kO2);
      // Descriptors split into a constant high word (stride, version, 128-byte swizzle)
      // and a low word (start address >> 4, leading offset); k-steps add constants.
      const uint64_t dq = ptx::smem_desc_sw128(t == 0 ? sQ0 : t == 1 ? sQ1 : sQ2, 16, 1024);
      const uint32_t hi = uint32_t(dq >> 32);
      const uint32_t q_lo = uint32_t(dq);
      const uint32_t k0_lo = uint32_t(ptx::smem_desc_sw128(sK(0), 16, 1024));
      const uint32_t v0_lo = uint32_t(ptx::smem_desc_sw128(sV(0), kColBlockBytes, 1024));
      constexpr uint32_t kStageStep = C::kStageBytes >> 4;  // 16-byte units
      // S (+)= Q K^T over D: k-step k moves 32 bytes inside a 128-byte row, 16 KB per 64 columns
      auto qk = [&](uint32_t k_lo, uint32_t idesc) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = uint32_t((k >> 2) * (kColBlockBytes >> 4) + (k & 3) * 2);
          if (k == 0) ptx::mma_ss_lh<0>(tS, q_lo + off, k_lo + off, hi, idesc);
          else ptx::mma_ss_lh<1>(tS, q_lo + off, k_lo + off, hi, idesc);
        }
      };
      // O (+)= P V over KSTEPS x 16 keys: a k-step is 16 key rows (2 KB) of V and 8 TMEM columns of P
      auto pv = [&](auto ksteps_tag, uint32_t v_lo, uint32_t p_col, uint32_t first_accumulate) {
        constexpr int KSTEPS = decltype(ksteps_tag)::value;
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k)
          ptx::mma_ts_lh(tO, p_col + 8 * k, v_lo + uint32_t(128 * k), hi, idesc_pv, k == 0 ? first_accumulate : 1u);
      };
      using K8 = std::integral_constant<int, 8>;
      using K4 = std::integral_constant<int, 4>;
      bool ok = ptx::mbar_wait_bounded(q_full, 0, limit, abort_flag);
      ptx::tc_fence_after();
      const int nmma = dump ? (t < 2 ? min(n, 1) : 0) : n;
      for (int c = 0; ok && c < nmma; ++c) {
        const int st = c % S;
        if (!(ok = ptx::mbar_wait_bounded(full_bar(st), (c / S) & 1, limit, abort_flag))) break;
        ptx::tc_fence_after();
        trace(p, kTrFullSeen, c);
        const uint32_t k_lo = k0_lo + uint32_t(st) * kStageStep;
        const uint32_t v_lo = v0_lo + uint32_t(st) * kStageStep;
        const uint32_t acc0 = c > 0 ? 1u : 0u;
        if (t < 2) {
          qk(k_lo, idesc_qk);
          ptx::mma_commit(s_full(t));
          trace(p, t ? kTrQk1 : kTrQk0, c);
          if (dump) break;
          if (!(ok = ptx::mbar_wait_bounded(p_ready(t), c & 1, limit, abort_flag))) break;
          ptx::tc_fence_after();
          trace(p, t ? kTrP1Seen : kTrP0Seen, c);
          pv(K8{}, v_lo, tS, acc0);
        } else {
          qk(k_lo, idesc_qk_half);                                  // keys 0..63
          ptx::mma_commit(s_full(2));
          trace(p, kTrQk2a, c);
          if (!(ok = ptx::mbar_wait_bounded(p_ready(2), 0, limit, abort_flag))) break;
          ptx::tc_fence_after();
          trace(p, kTrP2aSeen, c);
          pv(K4{}, v_lo, tS, acc0);
          qk(k_lo + uint32_t(64 * 128 >> 4), idesc_qk_half);        // keys 64..127
          ptx::mma_commit(s_full(2));
          trace(p, kTrQk2b, c);
          if (!(ok = ptx::mbar_wait_bounded(p_ready(2), 1, limit, abort_flag))) break;
          ptx::tc_fence_after();
          trace(p, kTrP2bSeen, c);
          pv(K4{}, v_lo + uint32_t(64 * 128 >> 4), tS, 1u);
        }
        ptx::mma_commit(empty_bar(st));  // this consumer is done with the stage
        trace(p, kTrEmpty, c);
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
    const uint32_t tS = tmem + (t ? C::kS1 : C::kS0) + lane_off;
    const uint32_t tO = tmem + (t ? C::kO1 : C::kO0) + lane_off;
    const int64_t qrow = int64_t(work.stream) * p.T + row;
    if (tile_on)
      store_q_row<D>(t ? sQ1 : sQ0, r,
                     reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + (qrow * p.H + head) * D),
                     row_ok);
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(q_full);

    if (tile_on && dump) {
      if (ptx::mbar_wait_warp(s_full(t), 0, limit, abort_flag) && n > 0) {
        ptx::tc_fence_after();
        float* dst = p.dump_scores + ((int64_t(blockIdx.x) * 2 + t) * 128 + r) * 128;
        for (int j = 0; j < 4; ++j) {
          uint32_t s[32];
          ptx::tmem_ld32(tS + 32 * j, s);
          ptx::tmem_wait_ld();
          for (int e = 0; e < 32; ++e) dst[32 * j + e] = __uint_as_float(s[e]);
        }
      }
    } else if (tile_on) {
      float m = -INFINITY;  // running max of scaled logits (log2 units)
      float l = 0.f;        // running sum of the bf16-rounded P
      bool ok = true;
      int len_next = n > 0 ? (__ldg(&p.chunks[c0].start_len) >> 16) : 0;
      for (int j = 0; j < n; ++j) {
        const int len = len_next;
        if (j + 1 < n) len_next = __ldg(&p.chunks[c0 + j + 1].start_len) >> 16;
        if (!(ok = ptx::mbar_wait_warp(s_full(t), j & 1, limit, abort_flag))) break;
        ptx::tc_fence_after();
        if (q4 == 0 && lane == 0) trace(p, t ? kTrS1Seen : kTrS0Seen, j);
        if (warp_on) {
          // One pass over S in 32-column quarters; the next quarter's TMEM load is in
          // flight while this one is exponentiated.  The running max m only moves when
          // a quarter's max exceeds it by more than 2^8; then O (earlier chunks), the
          // P already written for this chunk and l are rescaled, so every P of the
          // chunk shares one offset.  P of keys 32k..32k+31 goes to packed columns
          // 16k..16k+15, which only overwrite S columns already read.
          uint32_t qa[32], qb[32];
          ptx::tmem_ld32(tS, qa);
          ptx::tmem_wait_ld();
          auto quarter = [&](const int k, uint32_t(&cur)[32], uint32_t(&nxt)[32]) {
            if (k < 3) ptx::tmem_ld32(tS + 32 * (k + 1), nxt);
            mask32(cur, 32 * k, len);
            const float m_cand = max32(cur, -INFINITY) * sl2;
            const bool need = m_cand > m + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
              const float m_new = need ? m_cand : m;
              const float corr = need ? ptx::ex2(m - m_new) : 1.f;  // 0 while m is -inf
              rescale_running(tO, tS, j > 0 ? D : 0, 16 * k, corr);
              l *= corr;
              m = m_new;
            }
            l += exp_pack_store<32>(cur, sl2, -m, tS + 16 * k);
            if (k < 3) ptx::tmem_wait_ld();
          };
          quarter(0, qa, qb);
          quarter(1, qb, qa);
          quarter(2, qa, qb);
          quarter(3, qb, qa);
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        if (q4 == 0 && lane == 0) trace(p, t ? kTrP1Arrive : kTrP0Arrive, j);
        ptx::mbar_arrive(p_ready(t));
      }
      if (!ok) signal_abort(p.status, abort_flag);
      if (ok && ptx::mbar_wait_warp(o_done(t), 0, limit, abort_flag) && warp_on) {
        ptx::tc_fence_after();
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
  } else if constexpr (!C::kTail) {
    // warps 0-3 have no tail to work on; they still count towards q_full
    ptx::mbar_arrive(q_full);
  } else {
    // ------------------------------------------------------------ tail softmax (warps 0-3)
    const int q = warp;                       // lane quarter = key group
    const int i = lane;                       // tail row
    const bool row_ok = has_tail && i < p.tail_rows;
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t tS = tmem + C::kS2 + lane_off;
    const uint32_t tO = tmem + C::kO2 + lane_off;
    const int row = tail_row0 + i;
    const int64_t qrow = int64_t(work.stream) * p.T + row;
    if (has_tail)
      store_q_row<D>(sQ2, q * 32 + i,
                     reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + (qrow * p.H + head) * D),
                     row_ok);
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(q_full);
    if (has_tail && !dump) {
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      int len_next = n > 0 ? (__ldg(&p.chunks[c0].start_len) >> 16) : 0;
      for (int j = 0; ok && j < n; ++j) {
        const int len = len_next;
        if (j + 1 < n) len_next = __ldg(&p.chunks[c0 + j + 1].start_len) >> 16;
        for (int h = 0; h < 2; ++h) {
          if (!(ok = ptx::mbar_wait_warp(s_full(2), h, limit, abort_flag))) break;
          ptx::tc_fence_after();
          if (q == 0 && lane == 0) trace(p, h ? kTrS2bSeen : kTrS2aSeen, j);
          const int key0 = 64 * h + 16 * q;
          uint32_t s[16];
          ptx::tmem_ld16(tS + 16 * q, s);
          ptx::tmem_wait_ld();
          float mx = -INFINITY;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            if (key0 + e >= len) s[e] = __float_as_uint(-INFINITY);
            mx = fmaxf(mx, __uint_as_float(s[e]));
          }
          const float m_cand = mx * sl2;
          const bool need = m_cand > m + kRescaleThreshold;
          const float m_new = need ? m_cand : m;
          if ((j > 0 || h > 0) && __any_sync(0xffffffffu, need)) {
            const float corr = need ? ptx::ex2(m - m_new) : 1.f;
            rescale_tmem(tO, 64, corr);
            l *= corr;
          }
          m = m_new;
          const float neg_m = (m == -INFINITY) ? 0.f : -m;  // no key seen yet: every p is 0
          uint32_t pk[8], zero[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pk[e] = pack_bf16(ptx::ex2(fmaf(__uint_as_float(s[2 * e]), sl2, neg_m)),
                              ptx::ex2(fmaf(__uint_as_float(s[2 * e + 1]), sl2, neg_m)));
            l += packed_sum(pk[e]);
            zero[e] = 0u;
          }
          // this lane quarter's P is nonzero only on its own 16 keys (packed columns 8q..8q+7)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t(&src)[8] = (b == q) ? pk : zero;
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(tS + 8 * b),
                "r"(src[0]), "r"(src[1]), "r"(src[2]), "r"(src[3]), "r"(src[4]), "r"(src[5]), "r"(src[6]),
                "r"(src[7])
                : "memory");
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          if (q == 0 && lane == 0) trace(p, h ? kTrP2bArrive : kTrP2aArrive, j);
          ptx::mbar_arrive(p_ready(2));
        }
      }
      if (!ok) signal_abort(p.status, abort_flag);
      // merge the four key-group partial states of every tail row
      // The merge scratch reuses the K/V stage ring, so it may be written only once every
      // consumer's MMAs (and with them every load of this CTA) have completed.
      float* scratch = reinterpret_cast<float*>(smem + C::kKV);
      float* sm = scratch + 4 * kTailMaxRows * 64;
      float* sl = sm + 4 * kTailMaxRows;
      bool done = ok;
      for (int u = 0; u < 3 && done; ++u)
        if (u == 2 || u < n_main) done = ptx::mbar_wait_warp(o_done(u), 0, limit, abort_flag);
      if (done) {
        ptx::tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
          uint32_t v[32];
          ptx::tmem_ld32(tO + 32 * j, v);
          ptx::tmem_wait_ld();
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(scratch + (q * kTailMaxRows + i) * 64 + 32 * j);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                   __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
          }
        }
        if (row_ok) {
          sm[q * kTailMaxRows + i] = m;
          sl[q * kTailMaxRows + i] = l;
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (done && !*abort_flag) {
        for (int rr = q; rr < p.tail_rows; rr += 4) {
          float mm = -INFINITY;
#pragma unroll
          for (int g = 0; g < 4; ++g) mm = fmaxf(mm, sm[g * kTailMaxRows + rr]);
          float w[4], L = 0.f;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            w[g] = exp2f(sm[g * kTailMaxRows + rr] - mm);
            L += w[g] * sl[g * kTailMaxRows + rr];
          }
          float acc[2] = {0.f, 0.f};
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float* src = scratch + (g * kTailMaxRows + rr) * 64 + 2 * lane;
            acc[0] += w[g] * src[0];
            acc[1] += w[g] * src[1];
          }
          const float inv = 1.f / L;
          const int orow = tail_row0 + rr;
          if (work.nsplit == 1) {
            const int64_t qr = int64_t(work.stream) * p.T + orow;
            uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + (qr * p.H + head) * D);
            dst[lane] = pack_bf16(acc[0] * inv, acc[1] * inv);
          } else {
            const int64_t idx = (int64_t(split) * p.H + head) * p.T + orow;
            reinterpret_cast<float2*>(p.part_o + idx * D)[lane] = make_float2(acc[0] * inv, acc[1] * inv);
            if (lane == 0) p.part_lse[idx] = mm + __log2f(L);
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

template <int D>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap* map, cudaStream_t s) {
  constexpr int smem = Cfg<D>::kLaunch;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int64_t grid = int64_t(p.num_splits) * p.H * p.ngroups;
  if (grid <= 0 || grid > 0x7fffffff) return cudaErrorInvalidValue;
  attention_tc_kernel<D><<<unsigned(grid), kThreads, smem, s>>>(p, *map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_bf16(const AttnParams& p, const CUtensorMap* kv_map, cudaStream_t s) {
  return p.D == 64 ? launch_tc<64>(p, kv_map, s) : launch_tc<128>(p, kv_map, s);
}

TileShape attention_bf16_tiles(int T, int head_dim) {
  TileShape ts{};
  const int full = T / kTileRows, rem = T % kTileRows;
  if (head_dim == 64 && rem > 0 && rem <= kTailMaxRows) {
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
