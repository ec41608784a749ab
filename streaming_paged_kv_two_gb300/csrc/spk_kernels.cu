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
  // launched as a programmatic dependent: the previous kernel's writes (and everything
  // before it) are visible once the wait returns; the next kernel may then be scheduled
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
  return launch_dependent(append_kernel, dim3(unsigned(blocks)), dim3(256), 0, s, p);
}

// ------------------------------------------------------------------ merge
// Exact recombination of softmax attention over disjoint key sets: with
// M = max_j lse_j (log2 units) and w_j = 2^(lse_j - M),
// out = sum_j w_j O_j / sum_j w_j.  One thread per (stream, head, 4 columns, query
// row), rows fastest, so a warp reads 32 consecutive rows' float4s of a split in one
// 512-byte run.  The kernel is a chain of memory latencies, not a bandwidth problem
// (a few MB for the whole grid), so every split's log-sum-exp and partial of a group of
// kMergeGroup splits is requested at once (predicated loads, no branch between them) and
// the groups are combined online: M is raised group by group and the sums rescaled.
constexpr int kMergeGroup = 16;

template <int D, typename OutT>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  // launched as a programmatic dependent of the attention kernel: wait until that grid
  // has completed and its partials are visible (returns at once otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int V = D / 4;  // float4 per row
  const int per_head = V * p.T;
  const int idx = int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x);  // < B * H * V * T < 2^31 (host check)
  if (idx >= p.B * p.H * per_head) return;
  const int sh = idx / per_head;  // stream * H + head
  const int rem = idx - sh * per_head;
  const int c4 = rem / p.T;
  const int t = rem - c4 * p.T;
  const int s = sh / p.H, h = sh - s * p.H;
  const StreamDesc sd = p.streams[s];
  const int n = sd.nsplit;
  if (n <= 1) return;  // written by the attention kernel
  const float* lse_p = p.part_lse + (int64_t(sd.split_base) * p.H + h) * p.T + t;  // split 0's log-sum-exp
  const int64_t lse_step = int64_t(p.H) * p.T;                                     // next split, same (head, row)
  const float* o_p = p.part_o + part_o_offset<D>(sd.split_base, h, t, 4 * c4, p.H, p.T);
  const int64_t o_step = int64_t(p.H) * D * p.T;
  float m = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < n; j0 += kMergeGroup) {
    float l[kMergeGroup];
    float4 v[kMergeGroup];
#pragma unroll
    for (int g = 0; g < kMergeGroup; ++g) {
      const bool in = j0 + g < n;
      l[g] = in ? __ldg(lse_p + (j0 + g) * lse_step) : -INFINITY;
      v[g] = in ? __ldg(reinterpret_cast<const float4*>(o_p + (j0 + g) * o_step)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float gm = m;
#pragma unroll
    for (int g = 0; g < kMergeGroup; ++g) gm = fmaxf(gm, l[g]);
    // the first group's own split 0 is present, so gm is finite from the first group on
    const float r = gm == m ? 1.f : exp2f(m - gm);
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
    wsum *= r;
    m = gm;
#pragma unroll
    for (int g = 0; g < kMergeGroup; ++g) {
      const float w = exp2f(l[g] - m);  // 0 for the splits past n
      wsum += w;
      acc.x = fmaf(w, v[g].x, acc.x);
      acc.y = fmaf(w, v[g].y, acc.y);
      acc.z = fmaf(w, v[g].z, acc.z);
      acc.w = fmaf(w, v[g].w, acc.w);
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
  if (threads + 255 > INT32_MAX) return cudaErrorInvalidValue;  // the kernel indexes threads in 32 bits
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
// Accuracy path (SPK_F32): exact attention over the split's chunks in fp32 on the CUDA
// cores, the paged counterpart of the manager's force_fp32 dense path ("How LingBot-Map
// Uses FlashInfer KV Cache for Streaming 3D Reconstruction", "Attention Kernel
// Execution"; "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback in
// Streaming Inference", "Precision and Hardware Utilization").
// One CTA = (KV split, head, 64 query rows), 256 threads as 16 x 16: thread (ty, tx)
// owns rows 4ty..4ty+3; for S it computes keys tx + 16j (j < 4) of each 64-key tile,
// for O the columns [tx*D/16, (tx+1)*D/16).  Q (scaled to log2 units) stays in shared
// memory; K and V arrive in 64-key tiles (each a piece of one planner chunk, rows past
// its length zero-filled) through a double-buffered cp.async ring, so every visible key
// is read from memory once per CTA.  Online softmax in log2 units: per tile, the row max
// over the 16 threads of a row (shuffles), O rescaled when it grows, P written
// transposed to shared memory for the P V product.
constexpr int kF32Rows = 64;
constexpr int kF32Keys = 64;
constexpr int kF32Threads = 256;

template <int D>
struct F32Cfg {
  static constexpr int kLd = D + 4;  // shared row stride in floats (16-byte aligned, no bank conflicts)
  static constexpr int kTileFloats = kF32Keys * kLd;
  static constexpr int kQ = 0;
  static constexpr int kKV = kF32Rows * kLd;              // [2 buffers][K, V][64][kLd]
  static constexpr int kP = kKV + 4 * kTileFloats;        // P^T [64 keys][68]
  static constexpr int kFloats = kP + kF32Keys * (kF32Rows + 4);
  static constexpr int kBytes = kFloats * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The k-th 64-key tile of the split: walks the chunk list (a chunk of len keys gives
// ceil(len / 64) tiles).  Returns false past the split's end.
struct F32Tile {
  int page, start, len;  // pool page, first token, valid keys (<= 64)
};
__device__ __forceinline__ bool next_f32_tile(const AttnParams& p, int& c, int& h, int c_end, F32Tile& t) {
  while (c < c_end) {
    const ChunkDesc cd = p.chunks[c];
    const int len = cd.start_len >> 16;
    if (h * kF32Keys < len) {
      t.page = cd.page;
      t.start = (cd.start_len & 0xFFFF) + h * kF32Keys;
      t.len = min(kF32Keys, len - h * kF32Keys);
      ++h;
      return true;
    }
    ++c;
    h = 0;
  }
  return false;
}

template <int D>
__device__ __forceinline__ void load_f32_tile(const AttnParams& p, int head, const F32Tile& t, uint32_t sk, uint32_t sv) {
  using C = F32Cfg<D>;
  const float* pool = static_cast<const float*>(p.pool);
  const float* kbase = pool + int64_t(t.page) * p.page_stride + int64_t(t.start) * p.row_stride + int64_t(head) * D;
  constexpr int kVec = D / 4;  // float4 per key row
  for (int i = threadIdx.x; i < kF32Keys * kVec; i += kF32Threads) {
    const int key = i / kVec, c4 = i % kVec;
    const bool valid = key < t.len;
    const float* src = kbase + int64_t(valid ? key : 0) * p.row_stride + 4 * c4;
    const uint32_t off = uint32_t((key * C::kLd + 4 * c4) * 4);
    cp_async16(sk + off, src, valid);
    cp_async16(sv + off, src + p.half_stride, valid);
  }
}

// c += a * b elementwise on a pair of floats, one packed instruction (fma.rn.f32x2)
__device__ __forceinline__ void ffma2(float& c0, float& c1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, z;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "mov.b64 z, {%0, %1};\n\t"
      "fma.rn.f32x2 z, x, y, z;\n\t"
      "mov.b64 {%0, %1}, z;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

template <int D>
__global__ void __launch_bounds__(kF32Threads) attention_f32_kernel(const AttnParams p) {
  using C = F32Cfg<D>;
  constexpr int kCols = D / 16;  // O columns per thread
  extern __shared__ float4 f32_smem4[];
  float* sm = reinterpret_cast<float*>(f32_smem4);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int row_tiles = (p.T + kF32Rows - 1) / kF32Rows;
  int x = blockIdx.x;
  const int rt = x % row_tiles;
  x /= row_tiles;
  const int head = x % p.H;
  const int split = x / p.H;
  const WorkDesc w = p.works[split];

  // Q tile (rows past T are zero), scaled to log2 units
  float* Qs = sm + C::kQ;
  for (int i = tid; i < kF32Rows * (D / 4); i += kF32Threads) {
    const int r = i / (D / 4), c4 = i % (D / 4);
    const int t = rt * kF32Rows + r;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < p.T) {
      v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.q) +
                                                ((int64_t(w.stream) * p.T + t) * p.H + head) * D) + c4);
      v.x *= p.scale_log2;
      v.y *= p.scale_log2;
      v.z *= p.scale_log2;
      v.w *= p.scale_log2;
    }
    *reinterpret_cast<float4*>(Qs + r * C::kLd + 4 * c4) = v;
  }
  float* Ps = sm + C::kP;  // P^T: [key][row], row stride 68
  auto sk = [&](int b) { return sbase + uint32_t((C::kKV + (2 * b) * C::kTileFloats) * 4); };
  auto sv = [&](int b) { return sbase + uint32_t((C::kKV + (2 * b + 1) * C::kTileFloats) * 4); };
  const float* Ks_base = sm + C::kKV;

  float m[4], l[4], o[4][kCols];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < kCols; ++c) o[r][c] = 0.f;
  }
  int c = w.chunk_begin, h = 0;
  F32Tile cur, nxt;
  bool have = next_f32_tile(p, c, h, w.chunk_end, cur);
  if (have) load_f32_tile<D>(p, head, cur, sk(0), sv(0));
  cp_async_commit();
  for (int it = 0; have; ++it) {
    const int b = it & 1;
    const bool more = next_f32_tile(p, c, h, w.chunk_end, nxt);
    if (more) load_f32_tile<D>(p, head, nxt, sk(b ^ 1), sv(b ^ 1));
    cp_async_commit();
    cp_async_wait<1>();  // this tile's copies have landed
    __syncthreads();
    const float* Ks = Ks_base + (2 * b) * C::kTileFloats;
    const float* Vs = Ks_base + (2 * b + 1) * C::kTileFloats;
    // S = Q K^T for rows 4ty.. and keys tx + 16j: each dot product accumulates its even
    // and its odd dimensions in the two halves of a packed pair, added at the end
    float s[4][4], se[4][4], so[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j) se[r][j] = so[r][j] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
      float4 q4[4], k4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) q4[r] = *reinterpret_cast<const float4*>(Qs + (4 * ty + r) * C::kLd + d);
#pragma unroll
      for (int j = 0; j < 4; ++j) k4[j] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * j) * C::kLd + d);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ffma2(se[r][j], so[r][j], q4[r].x, q4[r].y, k4[j].x, k4[j].y);
          ffma2(se[r][j], so[r][j], q4[r].z, q4[r].w, k4[j].z, k4[j].w);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[r][j] = se[r][j] + so[r][j];
    // online softmax over the tile's valid keys
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (tx + 16 * j >= cur.len) s[r][j] = -INFINITY;
        mx = fmaxf(mx, s[r][j]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[r], mx);  // finite: every tile has at least one valid key
      const float corr = exp2f(m[r] - m_new);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pj = exp2f(s[r][j] - m_new);
        Ps[(tx + 16 * j) * (kF32Rows + 4) + 4 * ty + r] = pj;
        sum += pj;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l[r] = l[r] * corr + sum;
      m[r] = m_new;
#pragma unroll
      for (int cc = 0; cc < kCols; ++cc) o[r][cc] *= corr;
    }
    __syncthreads();
    // O += P V over the tile's keys (keys past len have P = 0 and zero-filled V rows)
#pragma unroll 4
    for (int j = 0; j < kF32Keys; ++j) {
      const float4 p4 = *reinterpret_cast<const float4*>(Ps + j * (kF32Rows + 4) + 4 * ty);
      const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
      for (int q = 0; q < kCols / 4; ++q) {
        const float4 v4 = *reinterpret_cast<const float4*>(Vs + j * C::kLd + tx * kCols + 4 * q);
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // two columns per packed instruction
          ffma2(o[r][4 * q], o[r][4 * q + 1], pr[r], pr[r], v4.x, v4.y);
          ffma2(o[r][4 * q + 2], o[r][4 * q + 3], pr[r], pr[r], v4.z, v4.w);
        }
      }
    }
    __syncthreads();  // the buffers and P^T are rewritten next
    cur = nxt;
    have = more;
  }
  cp_async_wait<0>();
  // epilogue: rows of this tile that exist
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = rt * kF32Rows + 4 * ty + r;
    if (t >= p.T) continue;
    const float inv = 1.f / l[r];
    if (w.nsplit == 1) {
      float* out = static_cast<float*>(p.out) + ((int64_t(w.stream) * p.T + t) * p.H + head) * D + tx * kCols;
#pragma unroll
      for (int q = 0; q < kCols / 4; ++q)
        *reinterpret_cast<float4*>(out + 4 * q) =
            make_float4(o[r][4 * q] * inv, o[r][4 * q + 1] * inv, o[r][4 * q + 2] * inv, o[r][4 * q + 3] * inv);
    } else {
#pragma unroll
      for (int q = 0; q < kCols / 4; ++q)
        *reinterpret_cast<float4*>(p.part_o + part_o_offset<D>(split, head, t, tx * kCols + 4 * q, p.H, p.T)) =
            make_float4(o[r][4 * q] * inv, o[r][4 * q + 1] * inv, o[r][4 * q + 2] * inv, o[r][4 * q + 3] * inv);
      if (tx == 0) p.part_lse[(int64_t(split) * p.H + head) * p.T + t] = m[r] + log2f(l[r]);
    }
  }
}

cudaError_t configure_attention_f32() {
  cudaError_t e = cudaFuncSetAttribute(attention_f32_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       F32Cfg<64>::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attention_f32_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              F32Cfg<128>::kBytes);
}

cudaError_t launch_attention_f32(const AttnParams& p, cudaStream_t s) {
  const int row_tiles = (p.T + kF32Rows - 1) / kF32Rows;
  const int64_t blocks = int64_t(p.num_splits) * p.H * row_tiles;
  if (blocks <= 0 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (p.D == 64) attention_f32_kernel<64><<<int(blocks), kF32Threads, F32Cfg<64>::kBytes, s>>>(p);
  else attention_f32_kernel<128><<<int(blocks), kF32Threads, F32Cfg<128>::kBytes, s>>>(p);
  return cudaGetLastError();
}

int f32_row_tiles(int T) { return (T + kF32Rows - 1) / kF32Rows; }

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
