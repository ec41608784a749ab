// Host side of libspk: the C ABI, page bookkeeping of the two-stream paged KV
// cache, and the once-per-frame planner.
//
// Bookkeeping follows "How LingBot-Map Uses FlashInfer KV Cache for Streaming 3D
// Reconstruction" ("Patch Stream and Special Stream", "Page Table Planning and
// Reuse") and "How FlashInfer's Paged KV Cache Attention Outperforms SDPA Fallback
// in Streaming Inference" ("Two-Stream Design"): one frame per patch page taken
// from free_patch_pages into the scale pages (while fewer than scale_frames) or
// the live window; special tokens packed contiguously over append-only special
// pages; eviction returns the oldest live-window pages to the free list; the
// visible table is scale -> live -> specials with last_page_len for the tail page.
// Free lists are FIFO (take from the front, recycle to the back).
//
// The planner turns the visible table into KV chunks (<= 128 tokens inside one
// page: P valid tokens on patch pages, page_size on full special pages,
// last_page_len on the tail page) and splits each stream's chunks into KV splits
// so that one attention launch fills the GPU; the split results are combined by
// a log-sum-exp merge.
#include "spk.h"
#include "spk_debug.h"
#include "spk_internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <string>
#include <vector>

using namespace spk;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() { return SPK_OK; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct StreamState {
  std::deque<int32_t> free_patch;     // free_patch_pages
  std::vector<int32_t> scale;         // scale_patch_pages
  std::deque<int32_t> live;           // live_window_patch_pages
  std::deque<int32_t> special_free;   // free_special_pages
  std::vector<int32_t> special_pages; // all_special_pages
  int64_t special_tokens = 0;
  int64_t frame_count = 0;
  int32_t cur_patch = -1;
  std::vector<int32_t> cur_spage, cur_sslot;
  std::vector<uint8_t> appended;      // per block: appended in the current frame
  std::vector<int32_t> init_patch, init_special;
  bool defer_eviction = false;        // evict_frames leaves the live window as it is
  // What the newest append took, kept until the next append, a rollback or a reset.
  struct Undo {
    bool valid = false;
    int32_t pid = -1;
    bool in_scale = false;
    std::vector<int32_t> opened;      // special pages the frame opened, in order
    int32_t prev_patch = -1;
    std::vector<int32_t> prev_spage, prev_sslot;
    std::vector<uint8_t> prev_appended;
  } undo;
};

int elem_bytes(int dtype) { return dtype == SPK_BF16 ? 2 : 4; }

int validate_config(const spk_config* c) {
  if (!c) return fail(SPK_ERR_INVALID_ARG, "config is NULL");
  if (c->num_blocks < 1) return fail(SPK_ERR_INVALID_ARG, "num_blocks must be >= 1");
  if (c->num_streams < 1 || c->num_streams > 4096) return fail(SPK_ERR_INVALID_ARG, "num_streams must be in [1, 4096]");
  if (c->num_heads < 1 || c->num_heads > 1024) return fail(SPK_ERR_INVALID_ARG, "num_heads must be in [1, 1024]");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(SPK_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (c->patches_per_frame < 1) return fail(SPK_ERR_INVALID_ARG, "patches_per_frame must be >= 1");
  if (c->page_size < c->patches_per_frame || c->page_size > 32768)
    return fail(SPK_ERR_INVALID_ARG, "page_size must be in [patches_per_frame, 32768]");
  if (c->specials_per_frame < 1 || c->specials_per_frame > kMaxSpecials)
    return fail(SPK_ERR_INVALID_ARG, "specials_per_frame must be in [1, %d]", kMaxSpecials);
  if (c->patches_per_frame + c->specials_per_frame > 16384)
    return fail(SPK_ERR_INVALID_ARG, "tokens per frame must be <= 16384");
  if (c->scale_frames < 0 || c->sliding_window < 0) return fail(SPK_ERR_INVALID_ARG, "scale_frames and sliding_window must be >= 0");
  if (c->max_patch_pages < 1 || c->max_special_pages < 1) return fail(SPK_ERR_INVALID_ARG, "max pages must be >= 1");
  if (c->dtype != SPK_BF16 && c->dtype != SPK_F32) return fail(SPK_ERR_INVALID_ARG, "dtype must be SPK_BF16 or SPK_F32");
  if (c->splits_per_stream < 0) return fail(SPK_ERR_INVALID_ARG, "splits_per_stream must be >= 0");
  if (c->max_query_frames < 0 || c->max_query_frames > kMaxQueryFrames)
    return fail(SPK_ERR_INVALID_ARG, "max_query_frames must be in [0, %d]", kMaxQueryFrames);
  int64_t pages = int64_t(c->num_streams) * (int64_t(c->max_patch_pages) + c->max_special_pages);
  if (pages > (int64_t(1) << 30)) return fail(SPK_ERR_INVALID_ARG, "too many pages");
  const int64_t B = c->num_streams, mpp = c->max_patch_pages, msp = c->max_special_pages;
  auto check_perm = [&](const int32_t* order, int64_t per, int64_t base0, int64_t stride, const char* what) -> int {
    if (!order) return SPK_OK;
    std::vector<uint8_t> seen(per);
    for (int64_t s = 0; s < B; ++s) {
      std::fill(seen.begin(), seen.end(), 0);
      const int64_t base = base0 + s * stride;
      for (int64_t i = 0; i < per; ++i) {
        int64_t id = order[s * per + i] - base;
        if (id < 0 || id >= per || seen[id])
          return fail(SPK_ERR_INVALID_ARG, "%s order of stream %lld is not a permutation of its ids", what, (long long)s);
        seen[id] = 1;
      }
    }
    return SPK_OK;
  };
  int rc = check_perm(c->patch_page_order, mpp, 0, mpp, "patch page");
  if (rc) return rc;
  return check_perm(c->special_page_order, msp, B * mpp, msp, "special page");
}

WorkspaceLayout make_layout(const spk_config& c) {
  WorkspaceLayout L;
  const int64_t B = c.num_streams, T = c.patches_per_frame + c.specials_per_frame;
  const int64_t cpp = (c.page_size + kChunkTokens - 1) / kChunkTokens;
  L.max_chunks = B * (int64_t(c.max_patch_pages) + c.max_special_pages) * cpp;
  L.max_splits = B * kMaxSplitsPerStream;
  size_t off = 0;
  L.status = off;  off = align256(off + 256);
  L.streams = off; off = align256(off + sizeof(StreamDesc) * B);
  L.chunks = off;  off = align256(off + sizeof(ChunkDesc) * L.max_chunks);
  L.works = off;   off = align256(off + sizeof(WorkDesc) * L.max_splits);
  L.plan_end = off;
  const int64_t Tq = T * std::max(1, c.max_query_frames);  // query rows per stream of the largest plan
  L.part_o = off;  off = align256(off + sizeof(float) * size_t(L.max_splits) * c.num_heads * Tq * c.head_dim);
  L.part_lse = off; off = align256(off + sizeof(float) * size_t(L.max_splits) * c.num_heads * Tq);
  L.total = off;
  return L;
}

size_t pool_bytes(const spk_config& c) {
  const size_t pages = size_t(c.num_streams) * (size_t(c.max_patch_pages) + c.max_special_pages);
  return pages * 2 * size_t(c.page_size) * c.num_heads * c.head_dim * elem_bytes(c.dtype);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

struct spk_cache {
  spk_config cfg{};
  bool dry = true;
  int T = 0;   // rows of one frame (P + S)
  int Tq = 0;  // query rows per stream of the current plan (query_frames * T)
  int device = 0;
  int num_sms = 152;
  std::vector<void*> pools;
  std::vector<CUtensorMap> maps;
  std::vector<StreamState> st;
  WorkspaceLayout ws;
  // plan
  bool plan_valid = false;
  void* plan_ws = nullptr;
  std::vector<int32_t> indices, kv_indptr, lpl, npp, qo;
  std::vector<ChunkDesc> chunks;
  std::vector<WorkDesc> works;
  std::vector<StreamDesc> sdesc;
  spk_plan_info info{};
  // pinned staging for the plan upload, double-buffered
  char* staging[2] = {nullptr, nullptr};
  cudaEvent_t staged[2] = {nullptr, nullptr};
  bool staged_used[2] = {false, false};
  int stage_idx = 0;
  long long wait_limit_ns = kDefaultWaitLimitNs;
  // device address of the library's static split-KV array on this cache's device,
  // looked up when the cache is created (spk_run_attention_static_scratch)
  void* static_scratch = nullptr;
};

namespace {

void reset_state(spk_cache* c) {
  const spk_config& g = c->cfg;
  for (auto& s : c->st) {
    s.free_patch.assign(s.init_patch.begin(), s.init_patch.end());
    s.scale.clear();
    s.live.clear();
    s.special_free.assign(s.init_special.begin(), s.init_special.end());
    s.special_pages.clear();
    s.special_tokens = 0;
    s.frame_count = 0;
    s.cur_patch = -1;
    s.cur_spage.assign(g.specials_per_frame, -1);
    s.cur_sslot.assign(g.specials_per_frame, -1);
    s.appended.assign(g.num_blocks, 0);
    s.defer_eviction = false;
    s.undo = StreamState::Undo{};
  }
  c->plan_valid = false;
  c->plan_ws = nullptr;
}

int check_cache(const spk_cache* c) {
  if (!c) return fail(SPK_ERR_INVALID_ARG, "cache is NULL");
  return SPK_OK;
}

int check_stream(const spk_cache* c, int stream) {
  if (stream < 0 || stream >= c->cfg.num_streams)
    return fail(SPK_ERR_INVALID_ARG, "stream %d out of range [0, %d)", stream, c->cfg.num_streams);
  return SPK_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SPK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Allocation of a new frame's targets (block 0).  All-or-nothing.
int allocate_frame(spk_cache* c, StreamState& s) {
  const spk_config& g = c->cfg;
  if (s.free_patch.empty()) return fail(SPK_ERR_OUT_OF_PATCH_PAGES, "no free patch page (frames %lld)", (long long)s.frame_count);
  const int64_t first = s.special_tokens, last = first + g.specials_per_frame - 1;
  const int64_t need = last / g.page_size + 1 - int64_t(s.special_pages.size());
  if (need > int64_t(s.special_free.size()))
    return fail(SPK_ERR_OUT_OF_SPECIAL_PAGES, "special page pool exhausted after %lld special tokens", (long long)first);
  StreamState::Undo& u = s.undo;
  u.valid = true;
  u.prev_patch = s.cur_patch;
  u.prev_spage = s.cur_spage;
  u.prev_sslot = s.cur_sslot;
  u.prev_appended = s.appended;
  u.opened.clear();
  const int32_t pid = s.free_patch.front();
  s.free_patch.pop_front();
  u.pid = pid;
  u.in_scale = int64_t(s.scale.size()) < g.scale_frames;
  if (u.in_scale) s.scale.push_back(pid);
  else s.live.push_back(pid);
  s.cur_patch = pid;
  for (int j = 0; j < g.specials_per_frame; ++j) {
    const int64_t pos = first + j;
    if (pos / g.page_size == int64_t(s.special_pages.size())) {
      s.special_pages.push_back(s.special_free.front());
      s.special_free.pop_front();
      u.opened.push_back(s.special_pages.back());
    }
    s.cur_spage[j] = s.special_pages[pos / g.page_size];
    s.cur_sslot[j] = int32_t(pos % g.page_size);
  }
  s.special_tokens += g.specials_per_frame;
  s.frame_count += 1;
  std::fill(s.appended.begin(), s.appended.end(), 0);
  return SPK_OK;
}

// KV splits per stream.  bf16: one CTA per SM and per (split, head, row group);
// pick n minimising waves * (chunks per split + per-CTA overhead) + a small
// charge per split for the partials it writes and the merge reads back.
int choose_splits(const spk_cache* c, const std::vector<int32_t>& nchunks, std::vector<int32_t>& nsplit) {
  const spk_config& g = c->cfg;
  const int B = g.num_streams;
  nsplit.assign(B, 1);
  if (g.splits_per_stream > 0) {
    for (int s = 0; s < B; ++s)
      nsplit[s] = std::max(1, std::min({g.splits_per_stream, nchunks[s], kMaxSplitsPerStream}));
    return SPK_OK;
  }
  int32_t cmax = 0;
  for (int s = 0; s < B; ++s) cmax = std::max(cmax, nchunks[s]);
  int per_split_ctas, slots;
  if (g.dtype == SPK_BF16) {
    per_split_ctas = B * g.num_heads * attention_bf16_tiles(c->Tq, g.head_dim).ngroups;
    slots = c->num_sms;
  } else {
    per_split_ctas = B * g.num_heads * f32_row_tiles(c->Tq);
    slots = c->num_sms * 2;
  }
  const double overhead_chunks = 2.0, split_charge = 0.25;
  int best = 1;
  double best_cost = 1e300;
  for (int n = 1; n <= std::min<int>(kMaxSplitsPerStream, std::max(1, cmax)); ++n) {
    const double waves = std::ceil(double(per_split_ctas) * n / slots);
    const double cost = waves * (std::ceil(double(cmax) / n) + overhead_chunks) + split_charge * n;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = n;
    }
  }
  for (int s = 0; s < B; ++s) nsplit[s] = std::max(1, std::min(best, nchunks[s]));
  return SPK_OK;
}

// Bytes of split-KV partials of the current plan's launch shape: fp32 O [splits][H][Tq][D]
// (256-byte aligned), then fp32 lse [splits][H][Tq].
size_t split_scratch_o_bytes(const spk_cache* c) {
  return align256(size_t(c->info.num_splits) * c->cfg.num_heads * c->Tq * c->cfg.head_dim * sizeof(float));
}
size_t split_scratch_bytes(const spk_cache* c) {
  return split_scratch_o_bytes(c) + size_t(c->info.num_splits) * c->cfg.num_heads * c->Tq * sizeof(float);
}

int build_plan(spk_cache* c) {
  const spk_config& g = c->cfg;
  const int B = g.num_streams;
  c->indices.clear(); c->kv_indptr.assign(1, 0); c->lpl.clear(); c->npp.clear(); c->qo.assign(1, 0);
  c->chunks.clear(); c->works.clear(); c->sdesc.assign(B, StreamDesc{0, 0, 0, 0});
  std::vector<int32_t> chunk_base(B + 1, 0), nchunks(B, 0);
  int64_t visible = 0;
  for (int s = 0; s < B; ++s) {
    const StreamState& x = c->st[s];
    if (x.frame_count < 1) return fail(SPK_ERR_BAD_STATE, "stream %d holds no frame; append before plan", s);
    const int32_t np = int32_t(x.scale.size() + x.live.size());
    const int32_t ns = int32_t(x.special_pages.size());
    const int32_t last_len = int32_t(x.special_tokens - int64_t(ns - 1) * g.page_size);
    std::vector<int32_t> pages;
    pages.insert(pages.end(), x.scale.begin(), x.scale.end());
    pages.insert(pages.end(), x.live.begin(), x.live.end());
    pages.insert(pages.end(), x.special_pages.begin(), x.special_pages.end());
    c->indices.insert(c->indices.end(), pages.begin(), pages.end());
    c->kv_indptr.push_back(c->kv_indptr.back() + int32_t(pages.size()));
    c->lpl.push_back(last_len);
    c->npp.push_back(np);
    c->qo.push_back(c->qo.back() + c->Tq);
    chunk_base[s] = int32_t(c->chunks.size());
    for (size_t i = 0; i < pages.size(); ++i) {
      int32_t ntok;
      if (int32_t(i) < np) ntok = g.patches_per_frame;
      else if (int32_t(i) < np + ns - 1) ntok = g.page_size;
      else ntok = last_len;
      visible += ntok;
      for (int32_t start = 0; start < ntok; start += kChunkTokens) {
        const int32_t len = std::min(kChunkTokens, ntok - start);
        c->chunks.push_back(ChunkDesc{pages[i], start | (len << 16)});
      }
    }
    nchunks[s] = int32_t(c->chunks.size()) - chunk_base[s];
  }
  if (int64_t(c->chunks.size()) > c->ws.max_chunks) return fail(SPK_ERR_INVALID_ARG, "internal: chunk table overflow");
  std::vector<int32_t> nsplit;
  choose_splits(c, nchunks, nsplit);
  bool merge = false;
  for (int s = 0; s < B; ++s) {
    c->sdesc[s].split_base = int32_t(c->works.size());
    c->sdesc[s].nsplit = nsplit[s];
    if (nsplit[s] > 1) merge = true;
    for (int j = 0; j < nsplit[s]; ++j) {
      const int32_t b0 = chunk_base[s] + int32_t(int64_t(nchunks[s]) * j / nsplit[s]);
      const int32_t b1 = chunk_base[s] + int32_t(int64_t(nchunks[s]) * (j + 1) / nsplit[s]);
      c->works.push_back(WorkDesc{s, b0, b1, nsplit[s]});
    }
  }
  c->info.num_chunks = int32_t(c->chunks.size());
  c->info.num_splits = int32_t(c->works.size());
  c->info.num_ctas = int32_t(c->works.size()) * g.num_heads *
                     (g.dtype == SPK_BF16 ? attention_bf16_tiles(c->Tq, g.head_dim).ngroups : f32_row_tiles(c->Tq));
  c->info.merge_needed = merge ? 1 : 0;
  c->info.visible_tokens = visible;
  c->info.split_scratch_bytes = merge ? int64_t(split_scratch_bytes(c)) : 0;
  c->info.static_scratch_capacity = int64_t(static_scratch_bytes());
  return SPK_OK;
}

int upload_plan(spk_cache* c, void* workspace, cudaStream_t stream) {
  const WorkspaceLayout& L = c->ws;
  const int i = c->stage_idx;
  c->stage_idx ^= 1;
  cudaError_t e;
  if (c->staged_used[i]) {
    e = cudaEventSynchronize(c->staged[i]);
    if (e != cudaSuccess) return cuda_fail(e, "plan staging wait");
  }
  char* h = c->staging[i];
  const size_t base = L.streams;
  std::memcpy(h + (L.streams - base), c->sdesc.data(), sizeof(StreamDesc) * c->sdesc.size());
  std::memcpy(h + (L.chunks - base), c->chunks.data(), sizeof(ChunkDesc) * c->chunks.size());
  std::memcpy(h + (L.works - base), c->works.data(), sizeof(WorkDesc) * c->works.size());
  const size_t bytes = L.works - base + sizeof(WorkDesc) * c->works.size();
  e = cudaMemcpyAsync(static_cast<char*>(workspace) + base, h, bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  e = cudaEventRecord(c->staged[i], stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan staging event");
  c->staged_used[i] = true;
  return SPK_OK;
}

}  // namespace

extern "C" {

const char* spk_last_error(void) { return g_last_error.c_str(); }

int spk_required_bytes(const spk_config* cfg, size_t* pool_bytes_per_block, size_t* workspace_bytes) {
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (pool_bytes_per_block) *pool_bytes_per_block = pool_bytes(*cfg);
  if (workspace_bytes) *workspace_bytes = make_layout(*cfg).total;
  return ok();
}

int spk_create_cache(const spk_config* cfg, void* const* pools, spk_cache** out) {
  if (!out) return fail(SPK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  spk_cache* c = new (std::nothrow) spk_cache();
  if (!c) return fail(SPK_ERR_INVALID_ARG, "out of host memory");
  c->cfg = *cfg;
  c->cfg.patch_page_order = nullptr;
  c->cfg.special_page_order = nullptr;
  c->T = cfg->patches_per_frame + cfg->specials_per_frame;
  c->Tq = c->T;
  c->ws = make_layout(c->cfg);
  const int B = cfg->num_streams;
  const int32_t mpp = cfg->max_patch_pages, msp = cfg->max_special_pages;
  c->st.resize(B);
  for (int s = 0; s < B; ++s) {
    auto& x = c->st[s];
    x.init_patch.resize(mpp);
    x.init_special.resize(msp);
    for (int32_t i = 0; i < mpp; ++i)
      x.init_patch[i] = cfg->patch_page_order ? cfg->patch_page_order[int64_t(s) * mpp + i] : s * mpp + i;
    for (int32_t i = 0; i < msp; ++i)
      x.init_special[i] = cfg->special_page_order ? cfg->special_page_order[int64_t(s) * msp + i]
                                                  : B * mpp + s * msp + i;
  }
  reset_state(c);
  c->dry = (pools == nullptr);
  if (!c->dry) {
    auto bail = [&](int code) { spk_destroy_cache(c); return code; };
    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGetDevice"));
    e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaDeviceGetAttribute"));
    const size_t pbytes = pool_bytes(c->cfg);
    c->pools.assign(pools, pools + cfg->num_blocks);
    for (int b = 0; b < cfg->num_blocks; ++b) {
      if (!c->pools[b] || (reinterpret_cast<uintptr_t>(c->pools[b]) & 255))
        return bail(fail(SPK_ERR_INVALID_ARG, "pool %d is NULL or not 256-byte aligned", b));
      e = cudaMemsetAsync(c->pools[b], 0, pbytes, 0);
      if (e != cudaSuccess) return bail(cuda_fail(e, "pool zeroing"));
    }
    e = cudaStreamSynchronize(0);
    if (e != cudaSuccess) return bail(cuda_fail(e, "pool zeroing"));
    const size_t stage_bytes = c->ws.plan_end - c->ws.streams;
    for (int i = 0; i < 2; ++i) {
      e = cudaMallocHost(reinterpret_cast<void**>(&c->staging[i]), stage_bytes);
      if (e != cudaSuccess) return bail(cuda_fail(e, "cudaMallocHost"));
      e = cudaEventCreateWithFlags(&c->staged[i], cudaEventDisableTiming);
      if (e != cudaSuccess) return bail(cuda_fail(e, "cudaEventCreate"));
    }
    // The static split-KV array's module is loaded here, at set-up, with the cache's device
    // current: spk_run_attention_static_scratch then reserves nothing when it runs.
    e = static_scratch_address(&c->static_scratch);
    if (e != cudaSuccess) return bail(cuda_fail(e, "static scratch address"));
    if (cfg->dtype == SPK_F32) {
      e = configure_attention_f32();
      if (e != cudaSuccess) return bail(cuda_fail(e, "fp32 attention kernel configuration"));
    }
    if (cfg->dtype == SPK_BF16) {
      e = configure_attention_bf16();
      if (e != cudaSuccess) return bail(cuda_fail(e, "attention kernel configuration"));
      auto encode = get_encode_fn();
      if (!encode) return bail(fail(SPK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable"));
      c->maps.resize(cfg->num_blocks);
      const int64_t H = cfg->num_heads, D = cfg->head_dim, ps = cfg->page_size;
      const int64_t pages = int64_t(B) * (mpp + msp);
      // dims (innermost first): d, head, token-in-page, page*2 + kv
      cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(ps), cuuint64_t(2 * pages)};
      cuuint64_t strides[3] = {cuuint64_t(D * 2), cuuint64_t(H * D * 2), cuuint64_t(ps * H * D * 2)};
      cuuint32_t box[4] = {64, 1, cuuint32_t(kChunkTokens), 1};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      for (int b = 0; b < cfg->num_blocks; ++b) {
        CUresult r = encode(&c->maps[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, c->pools[b], dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return bail(fail(SPK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for block %d", int(r), b));
      }
    }
  }
  *out = c;
  return ok();
}

int spk_destroy_cache(spk_cache* c) {
  if (!c) return ok();
  for (int i = 0; i < 2; ++i) {
    if (c->staged[i]) { cudaEventSynchronize(c->staged[i]); cudaEventDestroy(c->staged[i]); }
    if (c->staging[i]) cudaFreeHost(c->staging[i]);
  }
  delete c;
  return ok();
}

int spk_reset(spk_cache* c) {
  int rc = check_cache(c);
  if (rc) return rc;
  reset_state(c);
  return ok();
}

}  // extern "C"

namespace {

// The rotary part of spk_append_frame_rope, checked and turned into kernel tables.
struct RopeArgs {
  const void* q;
  void* q_out;
  const int32_t* pos;
  const spk_rope* rope;
};

int check_rope(const spk_cache* c, const RopeArgs& ra, AppendRopeParams* rp) {
  const spk_config& g = c->cfg;
  const spk_rope* r = ra.rope;
  if (!r) return fail(SPK_ERR_INVALID_ARG, "rope must point to an spk_rope");
  if (r->reserved != 0) return fail(SPK_ERR_INVALID_ARG, "spk_rope.reserved must be 0");
  if (!std::isfinite(r->theta) || !(r->theta > 0.0))
    return fail(SPK_ERR_INVALID_ARG, "spk_rope.theta must be finite and > 0");
  int64_t total = 0;
  for (int a = 0; a < 3; ++a) {
    if (r->sections[a] < 0) return fail(SPK_ERR_INVALID_ARG, "spk_rope.sections[%d] is negative", a);
    total += r->sections[a];
  }
  if (total > g.head_dim / 2)
    return fail(SPK_ERR_INVALID_ARG, "spk_rope.sections sum to %lld pairs, head_dim/2 = %d", (long long)total,
                g.head_dim / 2);
  if (c->dry) {
    if (ra.q || ra.q_out || ra.pos)
      return fail(SPK_ERR_INVALID_ARG, "bookkeeping-only cache takes q = q_out = positions = NULL");
  } else {
    if (!ra.pos || (reinterpret_cast<uintptr_t>(ra.pos) & 3))
      return fail(SPK_ERR_INVALID_ARG, "positions must be a 4-byte aligned device pointer");
    if ((ra.q == nullptr) != (ra.q_out == nullptr))
      return fail(SPK_ERR_INVALID_ARG, "q and q_out are both NULL or both device pointers");
    if ((reinterpret_cast<uintptr_t>(ra.q) | reinterpret_cast<uintptr_t>(ra.q_out)) & 15)
      return fail(SPK_ERR_INVALID_ARG, "q and q_out must be 16-byte aligned");
    if (ra.q && ra.q != ra.q_out) {
      const uintptr_t bytes = uintptr_t(c->T) * g.num_heads * g.head_dim * elem_bytes(g.dtype);
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(ra.q), b0 = reinterpret_cast<uintptr_t>(ra.q_out);
      if (a0 < b0 + bytes && b0 < a0 + bytes)
        return fail(SPK_ERR_INVALID_ARG, "q_out overlaps q without being q");
    }
  }
  if (rp) {
    rp->q = static_cast<const char*>(ra.q);
    rp->q_out = static_cast<char*>(ra.q_out);
    rp->pos = ra.pos;
    rp->head_dim = g.head_dim;
    rp->rot_pairs = int32_t(total);
    int i = 0;
    for (int a = 0; a < 3; ++a) {
      const int n = r->sections[a];
      for (int j = 0; j < n; ++j, ++i) {
        rp->axis[i] = int8_t(a);
        rp->inv_freq[i] = std::pow(r->theta, -double(j) / double(n));
      }
    }
  }
  return SPK_OK;
}

int append_impl(spk_cache* c, int stream, int block, const void* k, const void* v, const RopeArgs* ra,
                void* cuda_stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if ((rc = check_stream(c, stream))) return rc;
  const spk_config& g = c->cfg;
  if (block < 0 || block >= g.num_blocks) return fail(SPK_ERR_INVALID_ARG, "block %d out of range [0, %d)", block, g.num_blocks);
  if (c->dry) {
    if (k || v) return fail(SPK_ERR_INVALID_ARG, "bookkeeping-only cache takes k = v = NULL");
  } else if (!k || !v) {
    return fail(SPK_ERR_INVALID_ARG, "k and v must be device pointers");
  } else if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) {
    return fail(SPK_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  }
  AppendRopeParams rp{};
  if (ra && (rc = check_rope(c, *ra, &rp))) return rc;
  StreamState& s = c->st[stream];
  if (block == 0) {
    if ((rc = allocate_frame(c, s))) return rc;
    c->plan_valid = false;
  } else {
    if (s.frame_count == 0) return fail(SPK_ERR_BAD_STATE, "append of block %d before block 0 of a frame", block);
    if (s.appended[block]) return fail(SPK_ERR_BAD_STATE, "block %d appended twice in one frame (missing block 0?)", block);
  }
  s.appended[block] = 1;
  if (c->dry) return ok();
  AppendParams p{};
  const int e = elem_bytes(g.dtype);
  p.pool = static_cast<char*>(c->pools[block]);
  p.k = static_cast<const char*>(k);
  p.v = static_cast<const char*>(v);
  p.row_bytes = int64_t(g.num_heads) * g.head_dim * e;
  p.half_bytes = int64_t(g.page_size) * p.row_bytes;
  p.page_bytes = 2 * p.half_bytes;
  p.T = c->T;
  p.P = g.patches_per_frame;
  p.patch_page = s.cur_patch;
  for (int j = 0; j < g.specials_per_frame; ++j) {
    p.special_page[j] = s.cur_spage[j];
    p.special_slot[j] = s.cur_sslot[j];
  }
  cudaError_t err;
  if (ra) {
    rp.a = p;
    err = launch_append_rope(rp, e, static_cast<cudaStream_t>(cuda_stream));
  } else {
    err = launch_append(p, e, static_cast<cudaStream_t>(cuda_stream));
  }
  if (err != cudaSuccess) return cuda_fail(err, "append kernel launch");
  return ok();
}

}  // namespace

extern "C" {

int spk_append_frame(spk_cache* c, int stream, int block, const void* k, const void* v, void* cuda_stream) {
  return append_impl(c, stream, block, k, v, nullptr, cuda_stream);
}

int spk_append_frame_rope(spk_cache* c, int stream, int block, const void* k, const void* v, const void* q,
                          void* q_out, const int32_t* positions, const spk_rope* rope, void* cuda_stream) {
  const RopeArgs ra{q, q_out, positions, rope};
  return append_impl(c, stream, block, k, v, &ra, cuda_stream);
}

int spk_evict_frames(spk_cache* c, int stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if ((rc = check_stream(c, stream))) return rc;
  StreamState& s = c->st[stream];
  while (!s.defer_eviction && int64_t(s.live.size()) > c->cfg.sliding_window) {
    s.free_patch.push_back(s.live.front());
    s.live.pop_front();
  }
  c->plan_valid = false;
  return ok();
}

int spk_set_defer_eviction(spk_cache* c, int stream, int on) {
  int rc = check_cache(c);
  if (rc) return rc;
  if ((rc = check_stream(c, stream))) return rc;
  c->st[stream].defer_eviction = on != 0;
  return ok();
}

int spk_rollback_frame(spk_cache* c, int stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if ((rc = check_stream(c, stream))) return rc;
  const spk_config& g = c->cfg;
  StreamState& s = c->st[stream];
  StreamState::Undo& u = s.undo;
  if (!u.valid) return fail(SPK_ERR_BAD_STATE, "stream %d: no frame to roll back since its last append", stream);
  const bool held = u.in_scale ? (!s.scale.empty() && s.scale.back() == u.pid)
                               : (!s.live.empty() && s.live.back() == u.pid);
  if (!held)
    return fail(SPK_ERR_BAD_STATE, "stream %d: the newest frame's patch page was already evicted "
                "(defer eviction to keep frames that may be rolled back)", stream);
  if (u.in_scale) s.scale.pop_back();
  else s.live.pop_back();
  s.free_patch.push_front(u.pid);
  for (auto it = u.opened.rbegin(); it != u.opened.rend(); ++it) {
    s.special_pages.pop_back();
    s.special_free.push_front(*it);
  }
  s.special_tokens -= g.specials_per_frame;
  s.frame_count -= 1;
  s.cur_patch = u.prev_patch;
  s.cur_spage = u.prev_spage;
  s.cur_sslot = u.prev_sslot;
  s.appended = u.prev_appended;
  u.valid = false;
  c->plan_valid = false;
  return ok();
}

int spk_plan_queries(spk_cache* c, int query_frames, void* workspace, void* cuda_stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (c->dry && workspace) return fail(SPK_ERR_INVALID_ARG, "bookkeeping-only cache takes workspace = NULL");
  if (!c->dry && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return fail(SPK_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  const int max_qf = std::max(1, c->cfg.max_query_frames);
  if (query_frames < 1 || query_frames > max_qf)
    return fail(SPK_ERR_INVALID_ARG, "query_frames %d outside [1, %d] (spk_config.max_query_frames)", query_frames,
                max_qf);
  for (int s = 0; s < c->cfg.num_streams; ++s)
    if (c->st[s].frame_count < query_frames)
      return fail(SPK_ERR_BAD_STATE, "stream %d holds %lld frames, fewer than the %d query frames", s,
                  (long long)c->st[s].frame_count, query_frames);
  c->plan_valid = false;
  c->Tq = query_frames * c->T;
  if ((rc = build_plan(c))) return rc;
  if (!c->dry && (rc = upload_plan(c, workspace, static_cast<cudaStream_t>(cuda_stream)))) return rc;
  c->plan_ws = workspace;
  c->plan_valid = true;
  return ok();
}

int spk_plan(spk_cache* c, void* workspace, void* cuda_stream) { return spk_plan_queries(c, 1, workspace, cuda_stream); }

}  // extern "C"

namespace {

// Parameters of block's attention launch over the current plan, with the split-KV
// partials at part_o / part_lse.
AttnParams attention_params(const spk_cache* c, int block, const void* q, void* out, char* ws, float* part_o,
                            float* part_lse) {
  const spk_config& g = c->cfg;
  const WorkspaceLayout& L = c->ws;
  AttnParams p{};
  p.pool = c->pools[block];
  p.q = q;
  p.out = out;
  p.chunks = reinterpret_cast<const ChunkDesc*>(ws + L.chunks);
  p.works = reinterpret_cast<const WorkDesc*>(ws + L.works);
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.status = reinterpret_cast<int32_t*>(ws + L.status);
  p.row_stride = int64_t(g.num_heads) * g.head_dim;
  p.half_stride = int64_t(g.page_size) * p.row_stride;
  p.page_stride = 2 * p.half_stride;
  p.T = c->Tq;
  p.H = g.num_heads;
  p.D = g.head_dim;
  p.ps = g.page_size;
  p.num_splits = c->info.num_splits;
  p.ntiles = (c->Tq + kTileRows - 1) / kTileRows;
  {
    const TileShape ts = attention_bf16_tiles(c->Tq, g.head_dim);
    p.main_tiles = ts.main_tiles;
    p.tail_rows = ts.tail_rows;
    p.ngroups = ts.ngroups;
  }
  p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(g.head_dim)));
  p.wait_limit_ns = c->wait_limit_ns;
  return p;
}

// Launch the attention kernel, then, when a stream has several KV splits, the merge
// of their partials (not in score-dump mode, which writes no output).
int launch_attention(const spk_cache* c, int block, const AttnParams& p, char* ws, cudaStream_t stream) {
  const spk_config& g = c->cfg;
  cudaError_t e = g.dtype == SPK_BF16 ? launch_attention_bf16(p, &c->maps[block], stream)
                                      : launch_attention_f32(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  if (c->info.merge_needed && !p.dump_scores) {
    MergeParams m{};
    m.part_o = p.part_o;
    m.part_lse = p.part_lse;
    m.streams = reinterpret_cast<const StreamDesc*>(ws + c->ws.streams);
    m.out = p.out;
    m.B = g.num_streams;
    m.T = c->Tq;
    m.H = g.num_heads;
    m.D = g.head_dim;
    e = launch_merge(m, g.dtype, stream);
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  }
  return SPK_OK;
}

int run_attention_impl(spk_cache* c, int block, const void* q, void* out, void* workspace, void* cuda_stream,
                       float* dump_scores, unsigned long long* trace = nullptr, int32_t trace_cap = 0) {
  int rc = check_cache(c);
  if (rc) return rc;
  const spk_config& g = c->cfg;
  if (c->dry) return fail(SPK_ERR_INVALID_ARG, "bookkeeping-only cache cannot run attention");
  if (block < 0 || block >= g.num_blocks) return fail(SPK_ERR_INVALID_ARG, "block %d out of range", block);
  if (!q || !workspace || (!out && !dump_scores)) return fail(SPK_ERR_INVALID_ARG, "q, out and workspace must be device pointers");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(SPK_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (dump_scores && g.dtype != SPK_BF16) return fail(SPK_ERR_INVALID_ARG, "score dump exists for the bf16 kernel only");
  if (!c->plan_valid) return fail(SPK_ERR_BAD_STATE, "no current plan: call spk_plan after append/evict");
  if (workspace != c->plan_ws) return fail(SPK_ERR_INVALID_ARG, "workspace differs from the one given to spk_plan");
  for (int s = 0; s < g.num_streams; ++s)
    if (!c->st[s].appended[block])
      return fail(SPK_ERR_BAD_STATE, "block %d of stream %d not appended in the current frame", block, s);
  const WorkspaceLayout& L = c->ws;
  char* ws = static_cast<char*>(workspace);
  AttnParams p = attention_params(c, block, q, out, ws, reinterpret_cast<float*>(ws + L.part_o),
                                  reinterpret_cast<float*>(ws + L.part_lse));
  p.dump_scores = dump_scores;
  p.trace = trace;
  p.trace_cap = trace_cap;
  return launch_attention(c, block, p, ws, static_cast<cudaStream_t>(cuda_stream));
}

}  // namespace

extern "C" {

int spk_run_attention(spk_cache* c, int block, const void* q, void* out, void* workspace, void* cuda_stream) {
  return run_attention_impl(c, block, q, out, workspace, cuda_stream, nullptr);
}

int spk_debug_dump_scores(spk_cache* c, int block, const void* q, float* dst, void* workspace, void* cuda_stream) {
  if (!dst) return fail(SPK_ERR_INVALID_ARG, "dst is NULL");
  return run_attention_impl(c, block, q, nullptr, workspace, cuda_stream, dst);
}

int spk_debug_trace_attention(spk_cache* c, int block, const void* q, void* out, void* workspace,
                              uint64_t* trace, int32_t capacity, void* cuda_stream) {
  if (!trace || capacity < 1) return fail(SPK_ERR_INVALID_ARG, "trace buffer is NULL or empty");
  if (c && c->cfg.dtype != SPK_BF16) return fail(SPK_ERR_INVALID_ARG, "trace exists for the bf16 kernel only");
  return run_attention_impl(c, block, q, out, workspace, cuda_stream, nullptr,
                            reinterpret_cast<unsigned long long*>(trace), capacity);
}

int spk_run_attention_static_scratch(spk_cache* c, int block, const void* q, void* out, void* workspace,
                                     void* cuda_stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  const spk_config& g = c->cfg;
  if (c->dry) return fail(SPK_ERR_INVALID_ARG, "bookkeeping-only cache cannot run attention");
  if (block < 0 || block >= g.num_blocks) return fail(SPK_ERR_INVALID_ARG, "block %d out of range", block);
  if (!q || !out || !workspace) return fail(SPK_ERR_INVALID_ARG, "q, out and workspace must be device pointers");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(SPK_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (!c->plan_valid) return fail(SPK_ERR_BAD_STATE, "no current plan: call spk_plan after append/evict");
  if (workspace != c->plan_ws) return fail(SPK_ERR_INVALID_ARG, "workspace differs from the one given to spk_plan");
  for (int s = 0; s < g.num_streams; ++s)
    if (!c->st[s].appended[block])
      return fail(SPK_ERR_BAD_STATE, "block %d of stream %d not appended in the current frame", block, s);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != c->device)
    return fail(SPK_ERR_INVALID_ARG, "device %d is current but the cache lives on device %d", dev, c->device);
  // partials of every split: fp32 O, then fp32 lse (split_scratch_bytes)
  const size_t o_bytes = split_scratch_o_bytes(c);
  const size_t need = split_scratch_bytes(c);
  if (need > static_scratch_bytes())
    return fail(SPK_ERR_INVALID_ARG,
                "this plan needs %zu bytes of split scratch but the static array holds %zu; "
                "use fewer KV splits (spk_config.splits_per_stream)",
                need, static_scratch_bytes());
  void* scratch = c->static_scratch;
  char* ws = static_cast<char*>(workspace);
  const AttnParams p = attention_params(c, block, q, out, ws, static_cast<float*>(scratch),
                                        reinterpret_cast<float*>(static_cast<char*>(scratch) + o_bytes));
  rc = launch_attention(c, block, p, ws, static_cast<cudaStream_t>(cuda_stream));
  if (rc) return rc;
  return ok();
}

int spk_read_kv(spk_cache* c, int block, int page_id, void* dst, void* cuda_stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  const spk_config& g = c->cfg;
  if (c->dry) return fail(SPK_ERR_INVALID_ARG, "bookkeeping-only cache has no pools");
  if (block < 0 || block >= g.num_blocks) return fail(SPK_ERR_INVALID_ARG, "block %d out of range", block);
  const int64_t pages = int64_t(g.num_streams) * (int64_t(g.max_patch_pages) + g.max_special_pages);
  if (page_id < 0 || page_id >= pages) return fail(SPK_ERR_INVALID_ARG, "page %d out of range [0, %lld)", page_id, (long long)pages);
  if (!dst) return fail(SPK_ERR_INVALID_ARG, "dst is NULL");
  const size_t page_bytes = 2 * size_t(g.page_size) * g.num_heads * g.head_dim * elem_bytes(g.dtype);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaMemcpyAsync(dst, static_cast<char*>(c->pools[block]) + size_t(page_id) * page_bytes, page_bytes,
                                  cudaMemcpyDefault, stream);
  if (e != cudaSuccess) return cuda_fail(e, "read_kv copy");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "read_kv sync");
  return ok();
}

int spk_get_plan_host(const spk_cache* c, int32_t* indices, int32_t capacity, int32_t* kv_indptr, int32_t* last_page_len,
                      int32_t* num_patch_pages, int32_t* qo_indptr, int32_t* nnz) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!c->plan_valid) return fail(SPK_ERR_BAD_STATE, "no current plan");
  if (!nnz) return fail(SPK_ERR_INVALID_ARG, "nnz is NULL");
  *nnz = int32_t(c->indices.size());
  const int B = c->cfg.num_streams;
  if (kv_indptr) std::copy(c->kv_indptr.begin(), c->kv_indptr.end(), kv_indptr);
  if (last_page_len) std::copy(c->lpl.begin(), c->lpl.end(), last_page_len);
  if (num_patch_pages) std::copy(c->npp.begin(), c->npp.end(), num_patch_pages);
  if (qo_indptr) std::copy(c->qo.begin(), c->qo.begin() + B + 1, qo_indptr);
  if (indices) {
    if (capacity < *nnz) return fail(SPK_ERR_INVALID_ARG, "indices capacity %d < %d", capacity, *nnz);
    std::copy(c->indices.begin(), c->indices.end(), indices);
  }
  return ok();
}

int spk_get_plan_info(const spk_cache* c, spk_plan_info* info) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!c->plan_valid) return fail(SPK_ERR_BAD_STATE, "no current plan");
  if (!info) return fail(SPK_ERR_INVALID_ARG, "info is NULL");
  *info = c->info;
  return ok();
}

int spk_get_frame_targets(const spk_cache* c, int stream, int32_t* patch_page, int32_t* special_pages,
                          int32_t* special_slots) {
  int rc = check_cache(c);
  if (rc) return rc;
  if ((rc = check_stream(c, stream))) return rc;
  const StreamState& s = c->st[stream];
  if (s.frame_count == 0) return fail(SPK_ERR_BAD_STATE, "stream %d holds no frame", stream);
  if (patch_page) *patch_page = s.cur_patch;
  if (special_pages) std::copy(s.cur_spage.begin(), s.cur_spage.end(), special_pages);
  if (special_slots) std::copy(s.cur_sslot.begin(), s.cur_sslot.end(), special_slots);
  return ok();
}

int spk_get_stats(const spk_cache* c, int stream, spk_stats* out) {
  int rc = check_cache(c);
  if (rc) return rc;
  if ((rc = check_stream(c, stream))) return rc;
  if (!out) return fail(SPK_ERR_INVALID_ARG, "stats is NULL");
  const StreamState& s = c->st[stream];
  out->frame_count = s.frame_count;
  out->scale_pages = int64_t(s.scale.size());
  out->live_pages = int64_t(s.live.size());
  out->free_pages = int64_t(s.free_patch.size());
  out->special_tokens = s.special_tokens;
  return ok();
}

int spk_read_device_status(void* workspace, void* cuda_stream, int32_t* code) {
  if (!workspace || !code) return fail(SPK_ERR_INVALID_ARG, "workspace and code must be non-NULL");
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "status sync");
  int32_t v = 0;
  e = cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *code = v;
  if (v != kStatusOk) {
    e = cudaMemset(workspace, 0, 8);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return fail(SPK_ERR_DEVICE_TIMEOUT, "a device-side wait ran past its limit (code %d)", v);
  }
  return ok();
}

int spk_selftest_wait_timeout(void* workspace, int64_t limit_ns, void* cuda_stream) {
  if (!workspace) return fail(SPK_ERR_INVALID_ARG, "workspace is NULL");
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return fail(SPK_ERR_INVALID_ARG, "limit_ns must be in [1e3, 1e10]");
  cudaError_t e = launch_selftest_wait(static_cast<int32_t*>(workspace), (long long)limit_ns,
                                       static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return ok();
}

}  // extern "C"
