// Split-KV scratch held in a file-scope device array, for callers that must not
// allocate device memory while they run.
//
// The attention kernels write one fp32 partial output and one log-sum-exp per
// (KV split, head, query row) and the merge kernel reads them back.  The regular
// entry point keeps these partials in the caller's workspace.  This file owns a
// fixed array instead, so spk_run_attention_static_scratch needs no buffer beyond
// its inputs and outputs.  The array exists once per device that loads the library
// and stays until the process exits; every call on that device uses the same
// array.
#include "spk_internal.h"

#include <mutex>

namespace spk {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB of partials per device
__device__ __align__(256) unsigned char g_split_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

size_t static_scratch_bytes() { return kScratchBytes; }

// Device address of the array on the current device.  The first call on a device
// resolves it with cudaGetSymbolAddress (with that device current) and keeps it; the
// library makes that call when a cache is created, so the module holding the array is
// loaded (and its memory reserved) at set-up rather than by the first attention call.
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace spk
