// Internal declarations shared by the host library and the CUDA kernels of libspk.
// Not part of the public ABI (include/spk.h is).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace spk {

// KV chunk: a run of at most kChunkTokens consecutive tokens inside one page.
constexpr int kChunkTokens = 128;
// Upper bound of KV splits per stream (the workspace holds partials for this many).
constexpr int kMaxSplitsPerStream = 32;
// Special rows per frame that one append carries in its kernel parameters.
constexpr int kMaxSpecials = 64;
// Upper bound of spk_config.max_query_frames (frames of queries in one attention call).
constexpr int kMaxQueryFrames = 64;
// Query rows per tensor-core tile (tcgen05 M).
constexpr int kTileRows = 128;
// Events recorded by the bf16 attention kernel's trace mode (per chunk, CTA 0).
enum TraceEvent {
  kTrTmaIssue = 0, kTrFullSeen, kTrQk0, kTrP0Seen, kTrQk1, kTrP1Seen, kTrQk2, kTrP2Seen, kTrQk0h1, kTrP0h1Seen,
  kTrEmpty, kTrS0Seen, kTrP0Arrive, kTrS1Seen, kTrP1Arrive, kTrS2Seen, kTrP2Arrive, kTrS0h1Seen, kTrP0h1Arrive,
  kTrLanded, kTraceEvents
};
// Device status word codes (first int32 of the workspace).
constexpr int kStatusOk = 0;
constexpr int kStatusWaitTimeout = 1;
// Default limit of one device-side wait before it gives up (nanoseconds).
constexpr long long kDefaultWaitLimitNs = 2000000000LL;

// Chunk descriptor: page id, and start | len << 16 (start < 65536, 1 <= len <= 128).
struct ChunkDesc {
  int32_t page;
  int32_t start_len;
};

// One KV split of one stream.
struct WorkDesc {
  int32_t stream;
  int32_t chunk_begin;
  int32_t chunk_end;
  int32_t nsplit;  // splits of this stream; 1 = the attention kernel writes the output itself
};

// Per-stream merge table.
struct StreamDesc {
  int32_t split_base;  // index of the stream's first split
  int32_t nsplit;
  int32_t pad0, pad1;
};

// Workspace layout (byte offsets from its start, all 256-aligned).
struct WorkspaceLayout {
  size_t status = 0;     // int32 status, int32 detail
  size_t streams = 0;    // StreamDesc[B]
  size_t chunks = 0;     // ChunkDesc[max_chunks]
  size_t works = 0;      // WorkDesc[max_splits]
  size_t plan_end = 0;   // end of the part uploaded by plan
  size_t part_o = 0;     // float[max_splits][H][D/4][T][4] (see part_o_offset)
  size_t part_lse = 0;   // float[max_splits][H][T]  (log2 units)
  size_t total = 0;
  int64_t max_chunks = 0;
  int64_t max_splits = 0;
};

struct AppendParams {
  char* pool;                 // block pool base
  const char* k;              // [T, H, D]
  const char* v;
  int64_t row_bytes;          // H * D * elem
  int64_t page_bytes;         // 2 * ps * row_bytes (K half then V half)
  int64_t half_bytes;         // ps * row_bytes
  int32_t T, P;
  int32_t patch_page;
  int32_t special_page[kMaxSpecials];
  int32_t special_slot[kMaxSpecials];
};

// Rotary embedding fused into the append: per turned pair its position axis and
// theta^(-j/n) (double, from the host); kMaxRopePairs covers D <= 128.
constexpr int kMaxRopePairs = 64;
struct AppendRopeParams {
  AppendParams a;
  const char* q;              // [T, H, D] or nullptr
  char* q_out;                // [T, H, D] (may be q)
  const int32_t* pos;         // [T, 3]
  int32_t head_dim;
  int32_t rot_pairs;          // pairs turned (sections' sum)
  double inv_freq[kMaxRopePairs];
  int8_t axis[kMaxRopePairs];
};

struct AttnParams {
  const void* pool;
  const void* q;              // [B*T, H, D]
  void* out;                  // [B*T, H, D]
  const ChunkDesc* chunks;
  const WorkDesc* works;
  float* part_o;
  float* part_lse;
  int32_t* status;
  int64_t row_stride;         // elements between consecutive tokens in the pool (H*D)
  int64_t page_stride;        // elements between pages (2*ps*H*D)
  int64_t half_stride;        // elements between K and V halves of a page (ps*H*D)
  int32_t T, H, D, ps;
  int32_t num_splits;
  int32_t ntiles;             // query tiles of kTileRows per stream (fp32 path)
  int32_t main_tiles;         // bf16 path: 128-row query tiles handled by full warpgroups
  int32_t tail_rows;          // bf16 path: trailing rows (<= 16) handled by the key-split tail warps
  int32_t ngroups;            // bf16 path: CTAs per (split, head): pairs of main tiles, the tail on the last
  float scale_log2;           // log2(e) / sqrt(D)
  long long wait_limit_ns;
  unsigned long long* trace;  // diagnostics only: non-NULL makes CTA 0 record event clocks [kTraceEvents][trace_cap]
  int32_t trace_cap;
  float* dump_scores;         // diagnostics only: non-NULL makes the bf16 kernel write the raw
                              // Q K^T tile of each CTA's first chunk ([ctas][128][128] fp32) and stop
};

// Offset (in floats) of element d of query row `row` in the split-KV partial O of
// (split, head): the layout is [split][head][d/4][row][4], so the float4s of 32
// consecutive rows at one column group are contiguous (the attention kernels store
// one row per thread; the merge reads one row per thread).
template <int D>
__host__ __device__ inline int64_t part_o_offset(int split, int head, int row, int d, int H, int T) {
  return (((int64_t(split) * H + head) * (D / 4) + d / 4) * T + row) * 4 + (d & 3);
}

struct MergeParams {
  const float* part_o;
  const float* part_lse;
  const StreamDesc* streams;
  void* out;
  int32_t B, T, H, D;
};

// Kernel launchers (defined in the .cu files).  All return the launch error.
// Launch a kernel as a programmatic dependent of the previous kernel on the stream: its
// grid may be scheduled before that kernel has finished, so it executes
// griddepcontrol.wait before it touches memory that earlier work writes (the wait
// returns at once when nothing earlier is running).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_append(const AppendParams& p, int elem_bytes, cudaStream_t s);
cudaError_t launch_append_rope(const AppendRopeParams& p, int elem_bytes, cudaStream_t s);
cudaError_t launch_attention_bf16(const AttnParams& p, const CUtensorMap* kv_map, cudaStream_t s);
// Once per cache, with its device current: kernel attributes (dynamic shared memory) of the
// bf16 attention kernels.
cudaError_t configure_attention_bf16();
cudaError_t launch_attention_f32(const AttnParams& p, cudaStream_t s);
// Once per fp32 cache, with its device current: dynamic shared memory of the fp32 kernels.
cudaError_t configure_attention_f32();
// CTAs of the fp32 attention kernel per (split, head) for T query rows.
int f32_row_tiles(int T);
cudaError_t launch_merge(const MergeParams& p, int dtype, cudaStream_t s);
cudaError_t launch_selftest_wait(int32_t* status, long long limit_ns, cudaStream_t s);

// Split-KV scratch in a file-scope device array (spk_static_scratch.cu): its size, and
// its device address on the current device (resolved once per device).
size_t static_scratch_bytes();
cudaError_t static_scratch_address(void** out);

// Query-row tiling of the bf16 attention kernel for T rows and head_dim D.
struct TileShape {
  int main_tiles;
  int tail_rows;
  int ngroups;
};
TileShape attention_bf16_tiles(int T, int head_dim);

}  // namespace spk
