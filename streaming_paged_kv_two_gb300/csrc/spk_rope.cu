// Append with the 3-D rotary embedding of q and k fused into the scatter ("How
// LingBot-Map Uses FlashInfer KV Cache for Streaming 3D Reconstruction", "3D RoPE
// Position Encoding": q and k are rotated with positions that carry the global frame
// index before k enters the cache).  The rotation is RoFormer's (Su et al. 2021) per
// position axis: adjacent pairs (x[2i], x[2i+1]); pair j of an n-pair axis section turns
// by position * theta^(-j/n).
#include "spk_internal.h"

#include <cuda_bf16.h>

namespace spk {

namespace {

constexpr double kTwoPiHi = 6.283185307179586;       // 2*pi rounded to double
constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2*pi - kTwoPiHi
constexpr double kInvTwoPi = 0.15915494309189535;
constexpr int kRopeThreads = 256;

template <typename E>
__device__ __forceinline__ float elem_to_float(E x);
template <>
__device__ __forceinline__ float elem_to_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ float elem_to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename E>
__device__ __forceinline__ E float_to_elem(float x);
template <>
__device__ __forceinline__ float float_to_elem<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 float_to_elem<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Where unit u (16 bytes) of token row r comes from and goes to: units [0, upr) are K,
// [upr, 2 upr) V, [2 upr, 3 upr) Q.
struct RowIo {
  const AppendRopeParams* p;
  char* kdst;
  int64_t row_off;
  int32_t upr;
  __device__ __forceinline__ uint4 load(int32_t u) const {
    const int32_t t = u / upr;
    const int32_t c = u - t * upr;
    const AppendParams& a = p->a;
    const char* src = (t == 0 ? a.k : t == 1 ? a.v : p->q) + row_off + int64_t(c) * 16;
    // q may be rotated in place: a plain load (this thread alone reads and writes the unit)
    return t == 2 ? *reinterpret_cast<const uint4*>(src) : __ldg(reinterpret_cast<const uint4*>(src));
  }
};

// Rotate the pairs of unit u that lie in the turned sections, then store it.
template <typename E>
__device__ __forceinline__ void rotate_store(const RowIo& io, int32_t u, uint4 x, const float2* cs) {
  constexpr int kPer = 16 / int(sizeof(E));  // elements per unit (even)
  const AppendRopeParams& p = *io.p;
  const int32_t t = u / io.upr;
  const int32_t c = u - t * io.upr;
  const int32_t pair0 = (c % (p.head_dim / kPer)) * (kPer / 2);
  if (t != 1 && pair0 < p.rot_pairs) {
    E* e = reinterpret_cast<E*>(&x);
#pragma unroll
    for (int j = 0; j < kPer / 2; ++j) {
      if (pair0 + j < p.rot_pairs) {
        const float2 w = cs[pair0 + j];
        const float x0 = elem_to_float(e[2 * j]), x1 = elem_to_float(e[2 * j + 1]);
        e[2 * j] = float_to_elem<E>(fmaf(x0, w.x, -x1 * w.y));
        e[2 * j + 1] = float_to_elem<E>(fmaf(x0, w.y, x1 * w.x));
      }
    }
  }
  char* dst = (t == 0 ? io.kdst : t == 1 ? io.kdst + p.a.half_bytes : p.q_out + io.row_off) + int64_t(c) * 16;
  *reinterpret_cast<uint4*>(dst) = x;
}

// One CTA per token row.  Each thread first issues the loads of its first two units, so
// their latency overlaps the angle computation: (cos, sin) of every turned pair of the
// row, with the angle and its reduction modulo 2*pi in double (positions up to 2^31 times
// frequencies up to 1 keep their fraction of a turn) and sin/cos in fp32, into shared
// memory.  Then the units are rotated (K and Q units holding turned pairs) and stored;
// V is copied.
template <typename E>
__global__ void __launch_bounds__(kRopeThreads) append_rope_kernel(const AppendRopeParams p) {
  __shared__ float2 cs[kMaxRopePairs];
  // launched as a programmatic dependent (see append_kernel)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const AppendParams& a = p.a;
  const int32_t r = blockIdx.x;
  int32_t page, slot;
  if (r < a.P) {
    page = a.patch_page;
    slot = r;
  } else {
    page = a.special_page[r - a.P];
    slot = a.special_slot[r - a.P];
  }
  RowIo io;
  io.p = &p;
  io.kdst = a.pool + int64_t(page) * a.page_bytes + int64_t(slot) * a.row_bytes;
  io.row_off = int64_t(r) * a.row_bytes;
  io.upr = int32_t(a.row_bytes >> 4);
  const int32_t units = (p.q ? 3 : 2) * io.upr;
  const int32_t u0 = threadIdx.x, u1 = threadIdx.x + kRopeThreads;
  uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
  if (u0 < units) x0 = io.load(u0);
  if (u1 < units) x1 = io.load(u1);
  for (int i = threadIdx.x; i < p.rot_pairs; i += kRopeThreads) {
    const double ang = double(p.pos[3 * r + p.axis[i]]) * p.inv_freq[i];
    const double n = rint(ang * kInvTwoPi);
    const double red = fma(-n, kTwoPiLo, fma(-n, kTwoPiHi, ang));
    float s, c;
    sincosf(float(red), &s, &c);
    cs[i] = make_float2(c, s);
  }
  __syncthreads();
  if (u0 < units) rotate_store<E>(io, u0, x0, cs);
  if (u1 < units) rotate_store<E>(io, u1, x1, cs);
  for (int32_t u = threadIdx.x + 2 * kRopeThreads; u < units; u += kRopeThreads) rotate_store<E>(io, u, io.load(u), cs);
}

}  // namespace

cudaError_t launch_append_rope(const AppendRopeParams& p, int elem_bytes, cudaStream_t s) {
  if (elem_bytes == 2)
    return launch_dependent(append_rope_kernel<__nv_bfloat16>, dim3(unsigned(p.a.T)), dim3(kRopeThreads), 0, s, p);
  return launch_dependent(append_rope_kernel<float>, dim3(unsigned(p.a.T)), dim3(kRopeThreads), 0, s, p);
}

}  // namespace spk
