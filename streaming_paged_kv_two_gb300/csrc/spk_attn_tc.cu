// Paged-prefill attention on the 5th-generation tensor cores (sm_103a).
//
// What it computes: for every stream, head and query row of the current frame,
// softmax(q K_vis^T / sqrt(D)) V_vis over the stream's visible keys, non-causal,
// the frame's own keys included ("How LingBot-Map Uses FlashInfer KV Cache for
// Streaming 3D Reconstruction", "Frame Processing Loop" and "Attention Kernel
// Execution"; "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback
// in Streaming Inference", "Memory Bandwidth Efficiency": only visible pages are
// read).  Visible keys arrive as the planner's chunks (<= 128 tokens inside one
// page), so patch-page padding and the tail special page's unused slots are
// never part of the softmax ("How FlashInfer KV Cache Attention Accelerates
// Streaming 3D Reconstruction Over SDPA", "Efficient Attention Masking and
// Padding").
//
// One CTA = (KV split, head, 128-row query tile).  Warp roles:
//   warp 0    TMA producer: K and V chunk tiles gathered by page id from a 4-D
//             tensor map over the pool (d, head, token, page*2+kv), 128-byte swizzle,
//             into a 2-stage shared-memory ring.
//   warp 1    MMA issuer (one thread): S = Q K^T into TMEM (M=128, N=128, K=D),
//             then O += P V with P read from TMEM (M=128, N=D, K=128).
//   warps 2-5 softmax: one thread per query row (TMEM lane); fp32 online
//             softmax in log2 units with masking of the chunk's ragged tail; P
//             written back as bf16 over S; O rescaled in TMEM only when the
//             running maximum grows by more than 2^8; epilogue normalises O and
//             writes bf16 output (one split) or an fp32 partial and its
//             log-sum-exp (several splits, combined by the merge kernel).
// Every wait is bounded: on timeout the kernel records a status word, drains its
// own copies and MMAs, frees TMEM and returns.
#include "ptx_sm100.cuh"
#include "spk_internal.h"

#include <cuda_bf16.h>

namespace spk {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;  // S/P at [0,128), O at [128, 128+D)
constexpr int kColBlockBytes = 128 * 128;  // 128 rows x 64 bf16: one 128-byte-swizzled column block
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Smem {
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V tile
  static constexpr int kQ = 0;
  static constexpr int kK0 = kTileBytes;
  static constexpr int kBars = kTileBytes + kStages * 2 * kTileBytes;
  static constexpr int kNumBars = 2 * kStages + 4;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kLaunchBytes = kBytes + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ void signal_abort(int32_t* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(status, kStatusWaitTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kThreads, (D == 64) ? 2 : 1)
    attention_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap kv_map) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t sQ = sbase + L::kQ;
  auto sK = [&](int st) { return sbase + L::kK0 + st * 2 * L::kTileBytes; };
  auto sV = [&](int st) { return sbase + L::kK0 + st * 2 * L::kTileBytes + L::kTileBytes; };
  const uint32_t bars = sbase + L::kBars;
  auto full_bar = [&](int st) { return bars + 8 * st; };
  auto empty_bar = [&](int st) { return bars + 8 * (kStages + st); };
  const uint32_t q_full = bars + 8 * (2 * kStages);
  const uint32_t s_full = q_full + 8;
  const uint32_t p_ready = q_full + 16;
  const uint32_t o_done = q_full + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int x = blockIdx.x;
  const int tile = x % p.ntiles;
  x /= p.ntiles;
  const int head = x % p.H;
  const int split = x / p.H;
  const WorkDesc work = p.works[split];
  const int c0 = work.chunk_begin;
  const int n = work.chunk_end - work.chunk_begin;
  const int row0 = tile * kTileRows;
  const long long limit = p.wait_limit_ns;
  const bool dump = p.dump_scores != nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), 1);
    }
    ptx::mbar_init(q_full, 128);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(p_ready, 128);
    ptx::mbar_init(o_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&kv_map);
      int issued = 0;
      const int nload = dump ? (n > 0 ? 1 : 0) : n;
      for (int i = 0; i < nload; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!ptx::mbar_wait_bounded(empty_bar(st), ph ^ 1, limit, abort_flag)) {
          signal_abort(p.status, abort_flag);
          break;
        }
        const ChunkDesc cd = p.chunks[c0 + i];
        const int start = cd.start_len & 0xFFFF;
        ptx::mbar_arrive_expect_tx(full_bar(st), 2 * L::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
          ptx::tma_load_4d(sK(st) + cb * kColBlockBytes, &kv_map, cb * 64, head, start, 2 * cd.page, full_bar(st));
          ptx::tma_load_4d(sV(st) + cb * kColBlockBytes, &kv_map, cb * 64, head, start, 2 * cd.page + 1,
                           full_bar(st));
        }
        ++issued;
      }
      // drain: every issued copy must land before the CTA may exit
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        ptx::mbar_wait_bounded(full_bar(i % kStages), (i / kStages) & 1, limit, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, D, 0, 1);
      bool ok = ptx::mbar_wait_bounded(q_full, 0, limit, abort_flag);
      ptx::tc_fence_after();
      const int nmma = dump ? (n > 0 ? 1 : 0) : n;
      for (int i = 0; ok && i < nmma; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!(ok = ptx::mbar_wait_bounded(full_bar(st), ph, limit, abort_flag))) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kColBlockBytes + (k & 3) * 32;
          const uint64_t a = ptx::smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t b = ptx::smem_desc_sw128(sK(st) + off, 16, 1024);
          ptx::mma_ss(tS, a, b, idesc_qk, k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full);
        if (dump) break;
        if (!(ok = ptx::mbar_wait_bounded(p_ready, i & 1, limit, abort_flag))) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t b = ptx::smem_desc_sw128(sV(st) + k * 2048, kColBlockBytes, 1024);
          ptx::mma_ts(tO, tS + k * 8, b, idesc_pv, (i > 0 || k > 0) ? 1u : 0u);
        }
        ptx::mma_commit(empty_bar(st));
      }
      if (!ok) signal_abort(p.status, abort_flag);
      ptx::mma_commit(o_done);  // arrives once every MMA issued above has completed
      ptx::mbar_wait_bounded(o_done, 0, limit, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q4 * 32 + lane;            // row within the tile
    const int row = row0 + r;
    const bool row_ok = row < p.T;
    const bool warp_active = row0 + q4 * 32 < p.T;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const int64_t qrow = int64_t(work.stream) * p.T + row;

    // Q tile: 128 rows x D bf16, K-major, 128-byte swizzle (16-byte chunk c of row r
    // stored at chunk c ^ (r & 7) of its 128-byte row).
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                        (qrow * p.H + head) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row_ok) v = __ldg(src + c);
        const int cb = c >> 3, cc = c & 7;
        const uint32_t dst = sQ + cb * kColBlockBytes + (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                     "r"(v.w)
                     : "memory");
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(q_full);
    }

    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max of scaled logits (log2 units)
    float l = 0.f;        // running sum of 2^(logit - m)
    bool ok = true;

    if (dump) {
      ok = ptx::mbar_wait_warp(s_full, 0, limit, abort_flag);
      if (ok && n > 0) {
        ptx::tc_fence_after();
        float* dst = p.dump_scores + (int64_t(blockIdx.x) * 128 + r) * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t s[32];
          ptx::tmem_ld32(tS + lane_off + 32 * j, s);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) dst[32 * j + e] = __uint_as_float(s[e]);
        }
      }
    } else {
      int len_next = n > 0 ? (__ldg(&p.chunks[c0].start_len) >> 16) : 0;
      for (int i = 0; i < n; ++i) {
        const int len = len_next;
        if (i + 1 < n) len_next = __ldg(&p.chunks[c0 + i + 1].start_len) >> 16;
        if (!(ok = ptx::mbar_wait_warp(s_full, i & 1, limit, abort_flag))) break;
        ptx::tc_fence_after();
        if (warp_active) {
          uint32_t s[128];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t(&sj)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32 * j]);
            ptx::tmem_ld32(tS + lane_off + 32 * j, sj);
          }
          ptx::tmem_wait_ld();
          if (len < 128) {
#pragma unroll
            for (int j = 0; j < 128; ++j)
              if (j >= len) s[j] = __float_as_uint(-INFINITY);
          }
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int j = 0; j < 128; j += 4) {
            mx0 = fmaxf(mx0, __uint_as_float(s[j]));
            mx1 = fmaxf(mx1, __uint_as_float(s[j + 1]));
            mx2 = fmaxf(mx2, __uint_as_float(s[j + 2]));
            mx3 = fmaxf(mx3, __uint_as_float(s[j + 3]));
          }
          const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
          const bool need = m_cand > m + kRescaleThreshold;
          const float m_new = need ? m_cand : m;
          if (i > 0 && __any_sync(0xffffffffu, need)) {
            // O has PV of earlier chunks (complete: S of this chunk was issued after them)
            const float corr = need ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
              uint32_t o[32];
              ptx::tmem_ld32(tO + lane_off + 32 * j, o);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              ptx::tmem_st32(tO + lane_off + 32 * j, o);
            }
          }
          if (need) {
            l *= ptx::ex2(m - m_new);
            m = m_new;
          }
          const float neg_m = -m;
          float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = ptx::ex2(fmaf(__uint_as_float(s[32 * j + 2 * e]), sl2, neg_m));
              const float p1 = ptx::ex2(fmaf(__uint_as_float(s[32 * j + 2 * e + 1]), sl2, neg_m));
              sum0 += p0;
              sum1 += p1;
              pk[e] = pack_bf16(p0, p1);
            }
            ptx::tmem_st16(tS + lane_off + 16 * j, pk);
          }
          ptx::tmem_wait_st();
          l += sum0 + sum1;
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_ready);
      }
      if (!ok) signal_abort(p.status, abort_flag);

      // ---------------------------------------------------------- epilogue
      if (ok && ptx::mbar_wait_warp(o_done, 0, limit, abort_flag) && warp_active) {
        ptx::tc_fence_after();
        const float inv_l = 1.f / l;
        if (work.nsplit == 1) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (qrow * p.H + head) * D);
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + lane_off + 32 * j, o);
            ptx::tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
            if (row_ok) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[4 * j + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        } else {
          const int64_t idx = (int64_t(split) * p.H + head) * p.T + row;
          float4* dst = reinterpret_cast<float4*>(p.part_o + idx * D);
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + lane_off + 32 * j, o);
            ptx::tmem_wait_ld();
            if (row_ok) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[8 * j + v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                             __uint_as_float(o[4 * v + 2]) * inv_l,
                                             __uint_as_float(o[4 * v + 3]) * inv_l);
            }
          }
          if (row_ok) p.part_lse[idx] = m + __log2f(l);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap* map, cudaStream_t s) {
  constexpr int smem = Smem<D>::kLaunchBytes;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int64_t grid = int64_t(p.num_splits) * p.H * p.ntiles;
  if (grid <= 0 || grid > 0x7fffffff) return cudaErrorInvalidValue;
  attention_tc_kernel<D><<<unsigned(grid), kThreads, smem, s>>>(p, *map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_bf16(const AttnParams& p, const CUtensorMap* kv_map, cudaStream_t s) {
  return p.D == 64 ? launch_tc<64>(p, kv_map, s) : launch_tc<128>(p, kv_map, s);
}

int attention_bf16_ctas_per_sm(int head_dim) { return head_dim == 64 ? 2 : 1; }

}  // namespace spk
