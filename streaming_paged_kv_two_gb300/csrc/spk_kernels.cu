// Append (scatter) kernel, log-sum-exp merge kernel, fp32 CUDA-core attention
// for the SPK_F32 accuracy path, and the bounded-wait self-test kernel.
#include "ptx_sm100.cuh"
#include "spk_internal.h"

#include <cuda_bf16.h>

namespace spk {

// ------------------------------------------------------------------ append
// A frame's K/V rows land in the pool by slice assignment: rows 0..P-1 into the
// frame's patch page (slots 0..P-1), special row j into its reserved special
// slot ("How Paged KV Cache Attention Achieves Stable Inference in Ling-Bot-Map",
// "Frame Appending Without Dispatch Overhead"; "How FlashInfer's Paged KV Cache
// Attention Outperforms SDPA Fallback in Streaming Inference", "Two-Stream
// Design").  One thread moves 16 bytes; K and V in one launch.
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int32_t upr = int32_t(p.row_bytes >> 4);  // 16-byte units per token row
  const int32_t per_kv = p.T * upr;
  const int32_t total = 2 * per_kv;
  for (int32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += gridDim.x * blockDim.x) {
    const int32_t kv = u >= per_kv;
    const int32_t rem = u - kv * per_kv;
    const int32_t r = rem / upr;
    const int32_t c = rem - r * upr;
    const char* src = (kv ? p.v : p.k) + int64_t(r) * p.row_bytes + int64_t(c) * 16;
    int32_t page, slot;
    if (r < p.P) {
      page = p.patch_page;
      slot = r;
    } else {
      page = p.special_page[r - p.P];
      slot = p.special_slot[r - p.P];
    }
    char* dst = p.pool + int64_t(page) * p.page_bytes + kv * p.half_bytes + int64_t(slot) * p.row_bytes +
                int64_t(c) * 16;
    *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
  }
}

cudaError_t launch_append(const AppendParams& p, int /*elem_bytes*/, cudaStream_t s) {
  const int64_t units = 2 * int64_t(p.T) * (p.row_bytes >> 4);
  int64_t blocks = (units + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  append_kernel<<<int(blocks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ merge
// Exact recombination of softmax attention over disjoint key sets: with
// M = max_j lse_j (log2 units) and w_j = 2^(lse_j - M),
// out = sum_j w_j O_j / sum_j w_j.  One thread per (stream, head, 4 columns, query
// row), rows fastest, so a warp reads 32 consecutive rows' float4s of a split in one
// 512-byte run; the split loop is unrolled so the loads of several splits are in flight.
template <int D, typename OutT>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  // launched as a programmatic dependent of the attention kernel: wait until that grid
  // has completed and its partials are visible (returns at once otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int V = D / 4;  // float4 per row
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = int64_t(p.B) * p.H * V * p.T;
  if (idx >= total) return;
  const int t = int(idx % p.T);
  int64_t rest = idx / p.T;
  const int c4 = int(rest % V);
  rest /= V;
  const int h = int(rest % p.H);
  const int s = int(rest / p.H);
  const StreamDesc sd = p.streams[s];
  if (sd.nsplit <= 1) return;  // written by the attention kernel
  const int64_t lse0 = (int64_t(sd.split_base) * p.H + h) * p.T + t;  // split 0's log-sum-exp
  const int64_t lse_step = int64_t(p.H) * p.T;                         // next split, same (head, row)
  const int64_t o0 = part_o_offset<D>(sd.split_base, h, t, 4 * c4, p.H, p.T);
  const int64_t o_step = int64_t(p.H) * D * p.T;
  // every split's log-sum-exp in flight at once, then the weights
  float lse[kMaxSplitsPerStream];
#pragma unroll
  for (int j = 0; j < kMaxSplitsPerStream; ++j)
    lse[j] = j < sd.nsplit ? __ldg(&p.part_lse[lse0 + j * lse_step]) : -INFINITY;
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kMaxSplitsPerStream; ++j) m = fmaxf(m, lse[j]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxSplitsPerStream; ++j) {
    if (j < sd.nsplit) {
      const float w = exp2f(lse[j] - m);
      const float4 v = __ldg(reinterpret_cast<const float4*>(p.part_o + o0 + j * o_step));
      wsum += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  const float inv = 1.f / wsum;
  OutT* out = static_cast<OutT*>(p.out) + ((int64_t(s) * p.T + t) * p.H + h) * D + 4 * c4;
  if constexpr (sizeof(OutT) == 2) {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&a);
    pk.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(out) = pk;
  } else {
    *reinterpret_cast<float4*>(out) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

cudaError_t launch_merge(const MergeParams& p, int dtype, cudaStream_t s) {
  const int64_t threads = int64_t(p.B) * p.T * p.H * (p.D / 4);
  const int blocks = int((threads + 255) / 256);
  // programmatic dependent launch: the merge grid may be scheduled while the attention
  // kernel still runs (that kernel signals early); its griddepcontrol.wait orders it
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (dtype == 0) {
    if (p.D == 64) return cudaLaunchKernelEx(&cfg, merge_kernel<64, __nv_bfloat16>, p);
    return cudaLaunchKernelEx(&cfg, merge_kernel<128, __nv_bfloat16>, p);
  }
  if (p.D == 64) return cudaLaunchKernelEx(&cfg, merge_kernel<64, float>, p);
  return cudaLaunchKernelEx(&cfg, merge_kernel<128, float>, p);
}

// ------------------------------------------------------------------ fp32 attention
// Accuracy path (SPK_F32): exact attention over the split's chunks in fp32 on
// CUDA cores, the paged counterpart of the manager's force_fp32 dense path ("How
// LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction", "Attention
// Kernel Execution").  One warp per (query row, head); lanes split D; online
// softmax in log2 units.
template <int D>
__global__ void __launch_bounds__(256) attention_f32_kernel(const AttnParams p) {
  constexpr int E = D / 32;
  constexpr int kRowsPerCta = 8;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row_tiles = (p.T + kRowsPerCta - 1) / kRowsPerCta;
  int x = blockIdx.x;
  const int rt = x % row_tiles;
  x /= row_tiles;
  const int h = x % p.H;
  const int split = x / p.H;
  const int t = rt * kRowsPerCta + warp;
  if (t >= p.T) return;
  const WorkDesc w = p.works[split];
  const float* pool = static_cast<const float*>(p.pool);
  const int64_t qrow = int64_t(w.stream) * p.T + t;
  const float* qp = static_cast<const float*>(p.q) + (qrow * p.H + h) * D + lane * E;
  float q[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = qp[e] * p.scale_log2;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int c = w.chunk_begin; c < w.chunk_end; ++c) {
    const ChunkDesc cd = p.chunks[c];
    const int start = cd.start_len & 0xFFFF;
    const int len = cd.start_len >> 16;
    const float* kbase = pool + int64_t(cd.page) * p.page_stride + int64_t(start) * p.row_stride + h * D + lane * E;
    const float* vbase = kbase + p.half_stride;
    for (int j = 0; j < len; ++j) {
      const float* kr = kbase + int64_t(j) * p.row_stride;
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(q[e], __ldg(kr + e), s);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float m_new = fmaxf(m, s);
      const float corr = exp2f(m - m_new);
      const float pj = exp2f(s - m_new);
      const float* vr = vbase + int64_t(j) * p.row_stride;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(acc[e], corr, pj * __ldg(vr + e));
      l = fmaf(l, corr, pj);
      m = m_new;
    }
  }
  const float inv = 1.f / l;
  if (w.nsplit == 1) {
    float* o = static_cast<float*>(p.out) + (qrow * p.H + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = acc[e] * inv;
  } else {
    const int64_t idx = (int64_t(split) * p.H + h) * p.T + t;
#pragma unroll
    for (int e = 0; e < E; ++e) p.part_o[part_o_offset<D>(split, h, t, lane * E + e, p.H, p.T)] = acc[e] * inv;
    if (lane == 0) p.part_lse[idx] = m + log2f(l);
  }
}

cudaError_t launch_attention_f32(const AttnParams& p, cudaStream_t s) {
  const int row_tiles = (p.T + 7) / 8;
  const int64_t blocks = int64_t(p.num_splits) * p.H * row_tiles;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (p.D == 64) attention_f32_kernel<64><<<int(blocks), 256, 0, s>>>(p);
  else attention_f32_kernel<128><<<int(blocks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ wait self-test
// Waits on an mbarrier that nothing signals; the bounded wait gives up after
// limit_ns and the kernel records the timeout in the status word.
__global__ void selftest_wait_kernel(int32_t* status, long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, limit_ns, &abort_flag)) {
      atomicExch(status, kStatusWaitTimeout);
      atomicExch(status + 1, 1);
    }
  }
}

cudaError_t launch_selftest_wait(int32_t* status, long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace spk
