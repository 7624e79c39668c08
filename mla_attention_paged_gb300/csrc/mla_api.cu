// mla_api.cu -- host side of the libmla C ABI (include/mla.h): argument validation, the
// memoised decode plan (split count + workspace size, computed at run time and cached as
// the TokenSpeed talk "构建面向 Agentic 推理的下一代 LLM 推理引擎", section
// "Kernel：让 MLA 真正跑满 GPU", describes), TMA tensor-map encoding and kernel launches.
// No device memory is allocated here and no call synchronises the stream, except
// mla_get_status which exists to read the device status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <limits>
#include <queue>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/mla.h"
#include "mla_internal.h"

namespace mla {

// Per-device status word written by the kernels (bit 0 timeout, bit 1 device argument).
__device__ unsigned int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;

unsigned* status_ptr() {
  static std::mutex mu;
  static unsigned* ptrs[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// Tiled tensor map (128-byte swizzle unless given).  dims/strides innermost first; strides
// in bytes for dims 1..rank-1.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides[i];
  }
  CUresult r = fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool page_size_ok(int P) { return P == 8 || P == 16 || P == 32 || P == 64 || P == 128 || P == 256; }

thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;

// Inside stream capture an event must be recorded as an external node to be observable
// when the graph runs.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  return cudaEventRecord(ev, s);
}

std::mutex g_plan_mu;
std::unordered_map<std::string, mla_decode_plan_t> g_plan_cache;

// Cost model of the planner, in units of one 64-key tile of one CTA: a CTA costs its tiles
// plus a fixed part (start-up until its first tile has landed, and the epilogue), and a
// plan with more than one split pays kCombineTiles for the combine kernel.  The fixed part
// in tile units depends on the pool format: an e4m3 tile holds half the bytes of a bf16 or
// int8 one and streams in about half the time, while the start-up (Q load and split, the
// first tiles' latency) and the epilogue take about as long.
constexpr long long kCombineTiles = 2;
long long cta_fixed_tiles(int kv_dtype) { return kv_dtype == MLA_KV_E4M3 ? 10 : 3; }

// Launch order of a multi-wave plan: split by split (every request's split s before any
// split s + 1, so that short remainders go last) for one row group; request by request
// for several, whose row groups share each tile through L2 and so run best side by side
// on one request's keys.
bool split_major_order(int groups) { return groups == 1; }

// Estimated duration of a decode call whose splits are ct tiles long: the partial kernel's
// CTAs, in the grid's launch order (group fastest, then split_major_order's), are
// dispatched each onto the SM that frees first; CTAs of splits a request does not have
// exit at once and cost nothing.  Plus the combine, when some request is split.
// `bound`: the caller only needs costs up to it; once the estimate is known to exceed it,
// some value above it is returned without finishing the schedule.
long long plan_cost(const std::vector<int>& tiles, int groups, int ct, int sms, long long fixed,
                    long long bound = std::numeric_limits<long long>::max()) {
  int max_splits = 1;
  long long n_ctas = 0, longest = 0, work = 0;
  for (int t : tiles) {
    const int ns = (t + ct - 1) / ct;
    max_splits = std::max(max_splits, ns);
    n_ctas += static_cast<long long>(ns) * groups;
    longest = std::max<long long>(longest, std::min(t, ct));
    work += (static_cast<long long>(t) + static_cast<long long>(ns) * fixed) * groups;
  }
  const long long combine = max_splits > 1 ? kCombineTiles : 0;
  long long span;
  if (n_ctas <= sms) {
    span = longest + fixed;  // one wave: the longest CTA
  } else {
    // no schedule is shorter than its longest CTA or than the work spread over every SM
    const long long lower = std::max(longest + fixed, (work + sms - 1) / sms) + combine;
    if (lower > bound) return lower;
    std::priority_queue<long long, std::vector<long long>, std::greater<long long>> free_at;
    for (int i = 0; i < sms; ++i) free_at.push(0);
    span = 0;
    auto dispatch = [&](int t, int s) {
      const long long cost = std::min<long long>(ct, t - static_cast<long long>(s) * ct) + fixed;
      for (int g = 0; g < groups; ++g) {
        const long long start = free_at.top();
        free_at.pop();
        free_at.push(start + cost);
        span = std::max(span, start + cost);
      }
      return span + combine <= bound;  // (the span only grows)
    };
    bool go = true;
    if (split_major_order(groups)) {
      for (int s = 0; go && s < max_splits; ++s)
        for (size_t i = 0; go && i < tiles.size(); ++i)
          if (s * static_cast<long long>(ct) < tiles[i]) go = dispatch(tiles[i], s);
    } else {
      for (size_t i = 0; go && i < tiles.size(); ++i)
        for (int s = 0; go && s * static_cast<long long>(ct) < tiles[i]; ++s) go = dispatch(tiles[i], s);
    }
  }
  return span + combine;
}

// Keys-per-split chunk in whole 64-key tiles (at least 4 tiles, or the whole of the
// longest request when it is shorter).  Candidates: the smallest chunk for which the
// partial kernel needs no more CTAs than the GPU has SMs (one wave; when the unsplit call
// already fits), the longest request cut into 1-4 splits (1-32 with several row groups
// that the others leave badly balanced, below), and, for calls of one row group,
// the chunks that share all tiles evenly over one or two waves of SMs (the one-wave one and
// up to 8 tiles more).  (A batch of equal requests that one wave leaves a few SMs short of,
// e.g. 16 x 1024 tiles on 152 SMs as 144 CTAs of 114, then runs as 144 CTAs of 108 plus 16
// remainders of 52, the remainders launched last and paired up on the SMs that free first;
// with an e4m3 pool's larger fixed cost, 109 and remainders of 43.)  The candidate with the
// lowest plan_cost wins, the one with fewer splits on a tie, so a split is only taken when
// the model says it shortens the call.
int choose_chunk_tiles(const std::vector<int>& lens, int groups, int sms, long long fixed) {
  std::vector<int> tiles;
  tiles.reserve(lens.size());
  int max_tiles = 1;
  for (int L : lens) {
    tiles.push_back((L + kTileKeys - 1) / kTileKeys);
    max_tiles = std::max(max_tiles, tiles.back());
  }
  auto ctas = [&](int ct) {
    long long n = 0;
    for (int t : tiles) n += (t + ct - 1) / ct;
    return n * groups;
  };
  // smallest chunk: 4 tiles; fewer (down to one) only where the longest request still needs
  // at most 32 splits, one round of the combine (which stages up to 32 splits at a time)
  const int lo = std::min(4, std::max(1, (max_tiles + 31) / 32));
  std::vector<int> cands;
  for (int k = 1; k <= 4; ++k) {
    const int ct = (max_tiles + k - 1) / k;
    if (ct >= lo) cands.push_back(ct);
  }
  if (ctas(max_tiles) <= sms) {
    int a = lo, b = max_tiles;
    while (a < b) {
      const int mid = (a + b) / 2;
      if (ctas(mid) <= sms)
        b = mid;
      else
        a = mid + 1;
    }
    cands.push_back(a);
  }
  if (groups == 1) {
    long long total = 0;
    for (int t : tiles) total += t;
    for (int waves = 1; waves <= 2; ++waves) {
      const long long base = (total + static_cast<long long>(waves) * sms - 1) / (static_cast<long long>(waves) * sms);
      // one wave: also up to 8 tiles longer, which shortens the remainders that run two to
      // an SM (a larger fixed cost per CTA wants shorter remainders)
      for (int d = 0; d <= (waves == 1 ? 8 : 0); ++d) {
        const long long ct = base + d;
        if (ct >= lo && ct < max_tiles) cands.push_back(static_cast<int>(ct));
      }
    }
  }
  // A candidate wins with a lower cost, or an equal one and fewer splits (a longer chunk),
  // so costs above the best so far need not be finished.
  int best = max_tiles;
  long long best_cost = plan_cost(tiles, groups, max_tiles, sms, fixed);
  auto consider = [&](int ct) {
    const long long c = plan_cost(tiles, groups, ct, sms, fixed, best_cost);
    if (c < best_cost || (c == best_cost && ct > best)) {
      best = ct;
      best_cost = c;
    }
  };
  for (int ct : cands) consider(ct);
  // Several row groups (tensor-bound; each tile shared through L2) whose best plan so far
  // leaves the SMs idle more than a tenth of it (its cost above 1.1 x the work spread over
  // every SM, e.g. a ragged batch cut into one wave): also the longest request in 5-32
  // splits, whose shorter CTAs even the load out over several waves.
  if (groups > 1) {
    long long work = 0;
    for (int t : tiles) work += (static_cast<long long>(t) + fixed) * groups;
    const long long spread = (work + sms - 1) / sms;
    if (10 * best_cost > 11 * spread) {
      for (int k = 5; k <= 32; ++k) {
        const int ct = (max_tiles + k - 1) / k;
        if (ct >= lo) consider(ct);
      }
    }
  }
  return best;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int mla_version(void) { return 101; }

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_DEVICE_ARG: return "MLA_ERR_DEVICE_ARG";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_decode_plan(int batch, const int32_t* seq_lens_host, int q_len, int num_heads, int page_size,
                    int max_pages_per_seq, int64_t num_pages, int kv_dtype, int num_sms,
                    mla_decode_plan_t* plan_out) {
  if (!seq_lens_host || !plan_out || batch < 1 || q_len < 1 || num_heads < 1 || max_pages_per_seq < 1 ||
      num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_E4M3 && kv_dtype != MLA_KV_INT8 && kv_dtype != MLA_KV_INT8_PAGE)
    return MLA_ERR_INVALID_ARG;
  // q_len beyond a few drafts is the prefill of q_len new tokens over a paged prefix in
  // absorbed form (the same computation: new token t sees keys 0 .. L - q_len + t)
  if (q_len > 8192 || !page_size_ok(page_size) || static_cast<int64_t>(q_len) * num_heads > 131072)
    return MLA_ERR_UNSUPPORTED;
  if (batch > 65535) return MLA_ERR_UNSUPPORTED;
  std::vector<int> lens(seq_lens_host, seq_lens_host + batch);
  int max_len = 0;
  for (int L : lens) {
    if (L < q_len || static_cast<int64_t>(L) > static_cast<int64_t>(max_pages_per_seq) * page_size)
      return MLA_ERR_INVALID_ARG;
    max_len = std::max(max_len, L);
  }
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
  }
  std::string key;
  key.reserve(64 + 4 * lens.size());
  char head[160];
  snprintf(head, sizeof head, "%d,%d,%d,%d,%d,%lld,%d,%d|", batch, q_len, num_heads, page_size, max_pages_per_seq,
           static_cast<long long>(num_pages), kv_dtype, num_sms);
  key += head;
  key.append(reinterpret_cast<const char*>(lens.data()), lens.size() * sizeof(int));
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = g_plan_cache.find(key);
    if (it != g_plan_cache.end()) {
      *plan_out = it->second;
      return MLA_OK;
    }
  }
  mla_decode_plan_t pl;
  memset(&pl, 0, sizeof pl);
  pl.batch = batch;
  pl.q_len = q_len;
  pl.num_heads = num_heads;
  pl.page_size = page_size;
  pl.max_pages_per_seq = max_pages_per_seq;
  pl.kv_dtype = kv_dtype;
  pl.num_pages = num_pages;
  pl.num_sms = num_sms;
  pl.rows = q_len * num_heads;
  pl.head_groups = (pl.rows + kGroupRows - 1) / kGroupRows;
  const int ct = choose_chunk_tiles(lens, pl.head_groups, num_sms, cta_fixed_tiles(kv_dtype));
  pl.chunk_tokens = ct * kTileKeys;
  pl.max_seq_len = max_len;
  pl.max_splits = (max_len + pl.chunk_tokens - 1) / pl.chunk_tokens;
  if (pl.max_splits > 65535) return MLA_ERR_UNSUPPORTED;
  {
    // more CTAs with work than SMs, one row group: launch split by split, as the cost model assumed
    long long n_ctas = 0;
    for (int L : lens) n_ctas += (L + pl.chunk_tokens - 1) / pl.chunk_tokens;
    pl.split_major = (n_ctas * pl.head_groups > num_sms && split_major_order(pl.head_groups)) ? 1 : 0;
  }
  if (pl.max_splits > 1) {
    const size_t parts = static_cast<size_t>(batch) * pl.max_splits * pl.rows;
    pl.workspace_bytes = 256 + parts * kValueDim * sizeof(__nv_bfloat16) + parts * sizeof(float);
  } else {
    pl.workspace_bytes = 0;
  }
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    if (g_plan_cache.size() > 4096) g_plan_cache.clear();
    g_plan_cache.emplace(key, pl);
  }
  *plan_out = pl;
  return MLA_OK;
}

}  // extern "C"

namespace {

constexpr int kStagePartial = 1;
constexpr int kStageCombine = 2;

// The two stages of a decode call.  The partial stage needs q, the pages and the page table;
// the combine stage reads only the lengths, the workspace and writes out/lse.
int decode_stages(const mla_decode_plan_t* plan, const void* q, const void* kv_pages, const float* page_scales,
                  const int32_t* page_table,
                  const int32_t* seq_lens, int q_len, int num_heads, float scale, float kv_scale, void* out,
                  float* lse, void* workspace, size_t workspace_bytes, void* stream, int stages) {
  const bool partial = (stages & kStagePartial) != 0;
  if (!plan || !seq_lens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (partial && (!q || !kv_pages || !page_table)) return MLA_ERR_INVALID_ARG;
  // a pool with a scale per page needs the scales; no other pool takes them
  if (partial && (plan->kv_dtype == MLA_KV_INT8_PAGE) != (page_scales != nullptr)) return MLA_ERR_INVALID_ARG;
  if (page_scales && !aligned(page_scales, 4)) return MLA_ERR_INVALID_ARG;
  if (q_len != plan->q_len || num_heads != plan->num_heads || plan->rows != q_len * num_heads)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
  if (partial && (!aligned(q, 16) || !aligned(kv_pages, 16))) return MLA_ERR_INVALID_ARG;
  if (partial && (!(scale > 0.f) || !(kv_scale > 0.f))) return MLA_ERR_INVALID_ARG;
  if (plan->workspace_bytes > 0) {
    if (!workspace) return MLA_ERR_INVALID_ARG;
    if (workspace_bytes < plan->workspace_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  }
  unsigned* status = status_ptr();
  if (!status) return MLA_ERR_CUDA;

  const uint64_t row_bytes = kLatentDim * 2;
  // Latent rows are viewed as [rows][9 blocks][64 columns] (block stride 128 bytes), so one
  // 3-D box {64 columns, n rows, 9 blocks} lands a whole row range as the nine 128-byte
  // swizzled column blocks the MMAs read, in a single TMA instruction.
  CUtensorMap tm_q, tm_kv;
  memset(&tm_q, 0, sizeof tm_q);
  if (partial) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(plan->batch) * plan->rows, kLatentDim / 64};
    const uint64_t strides[2] = {row_bytes, 128};
    const uint32_t box[3] = {64, static_cast<uint32_t>(kGroupRows), kLatentDim / 64};
    if (!make_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box)) return MLA_ERR_CUDA;
  }
  memset(&tm_kv, 0, sizeof tm_kv);
  if (partial && plan->kv_dtype == MLA_KV_E4M3) {
    // e4m3 codes, 576 bytes per row, viewed as [rows][9 blocks][64 bytes] with 64-byte
    // swizzle: one box lands a 64-key tile as the K-major layout the 8-bit MMAs read.
    const uint64_t rows = static_cast<uint64_t>(plan->num_pages) * plan->page_size;
    if (plan->page_size >= kTileKeys) {
      const uint64_t dims[3] = {64, rows, kLatentDim / 64};
      const uint64_t strides[2] = {static_cast<uint64_t>(kLatentDim), 64};
      const uint32_t box[3] = {64, static_cast<uint32_t>(kTileKeys), kLatentDim / 64};
      if (!make_map(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv_pages, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
        return MLA_ERR_CUDA;
    } else {  // smaller pages: one 2-D box per (page, column block)
      const uint64_t dims[2] = {static_cast<uint64_t>(kLatentDim), rows};
      const uint64_t strides[1] = {static_cast<uint64_t>(kLatentDim)};
      const uint32_t box[2] = {64, static_cast<uint32_t>(plan->page_size)};
      if (!make_map(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv_pages, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
        return MLA_ERR_CUDA;
    }
  }
  if (partial && plan->kv_dtype == MLA_KV_BF16) {  // int8 pages are read row by row by the decode warps
    const uint64_t rows = static_cast<uint64_t>(plan->num_pages) * plan->page_size;
    if (plan->page_size >= kTileKeys) {  // a 64-key tile is one row range of one page
      const uint64_t dims[3] = {64, rows, kLatentDim / 64};
      const uint64_t strides[2] = {row_bytes, 128};
      const uint32_t box[3] = {64, static_cast<uint32_t>(kTileKeys), kLatentDim / 64};
      if (!make_map(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_pages, dims, strides, box)) return MLA_ERR_CUDA;
    } else {  // smaller pages: one 2-D box per (page, column block)
      const uint64_t dims[2] = {static_cast<uint64_t>(kLatentDim), rows};
      const uint64_t strides[1] = {row_bytes};
      const uint32_t box[2] = {64, static_cast<uint32_t>(plan->page_size)};
      if (!make_map(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_pages, dims, strides, box)) return MLA_ERR_CUDA;
    }
  }
  DecodeParams p;
  memset(&p, 0, sizeof p);
  p.B = plan->batch;
  p.T = q_len;
  p.H = num_heads;
  p.R = plan->rows;
  p.page_size = plan->page_size;
  p.max_pages = plan->max_pages_per_seq;
  p.chunk = plan->chunk_tokens;
  p.max_splits = plan->max_splits;
  p.max_seq = plan->max_seq_len;
  p.split_major = plan->split_major;
  p.kv_dtype = plan->kv_dtype;
  p.num_pages = plan->num_pages;
  const bool kv8 = plan->kv_dtype != MLA_KV_BF16;
  p.scale_log2 = scale * 1.4426950408889634f * (kv8 ? kv_scale : 1.f);
  p.v_scale = kv8 ? kv_scale : 1.f;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.kv_pool = static_cast<const uint8_t*>(kv_pages);
  p.page_scales = page_scales;
  p.inv_ref_scale = 1.f / kv_scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  if (plan->max_splits > 1) {
    const size_t parts = static_cast<size_t>(plan->batch) * plan->max_splits * plan->rows;
    p.ws_o = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(workspace) + 256);
    p.ws_lse = reinterpret_cast<float*>(p.ws_o + parts * kValueDim);
  }
  p.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (partial) {
    if (g_prof_start && record_event(g_prof_start, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (launch_decode_partial(p, tm_q, tm_kv, plan->head_groups, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (g_prof_stop && record_event(g_prof_stop, s) != cudaSuccess) return MLA_ERR_CUDA;
  }
  if ((stages & kStageCombine) && plan->max_splits > 1) {
    if (launch_decode_combine(p, s) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode(const mla_decode_plan_t* plan, const void* q, const void* kv_pages, const int32_t* page_table,
               const int32_t* seq_lens, int q_len, int num_heads, float scale, float kv_scale, void* out,
               float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_stages(plan, q, kv_pages, nullptr, page_table, seq_lens, q_len, num_heads, scale, kv_scale, out,
                       lse, workspace, workspace_bytes, stream, kStagePartial | kStageCombine);
}

int mla_decode_int8_paged(const mla_decode_plan_t* plan, const void* q, const void* kv_pages, const float* page_scales,
                          const int32_t* page_table, const int32_t* seq_lens, int q_len, int num_heads, float scale,
                          float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!plan || plan->kv_dtype != MLA_KV_INT8_PAGE || !page_scales) return MLA_ERR_INVALID_ARG;
  return decode_stages(plan, q, kv_pages, page_scales, page_table, seq_lens, q_len, num_heads, scale, kv_scale, out,
                       lse, workspace, workspace_bytes, stream, kStagePartial | kStageCombine);
}

int mla_decode_partial(const mla_decode_plan_t* plan, const void* q, const void* kv_pages,
                       const int32_t* page_table, const int32_t* seq_lens, int q_len, int num_heads, float scale,
                       float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return decode_stages(plan, q, kv_pages, nullptr, page_table, seq_lens, q_len, num_heads, scale, kv_scale, out,
                       lse, workspace, workspace_bytes, stream, kStagePartial);
}

int mla_decode_combine(const mla_decode_plan_t* plan, const int32_t* seq_lens, int q_len, int num_heads,
                       void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_stages(plan, nullptr, nullptr, nullptr, nullptr, seq_lens, q_len, num_heads, 1.f, 1.f, out, lse,
                       workspace, workspace_bytes, stream, kStageCombine);
}

int mla_prefill_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_kv, const int32_t* prefix_lens, int batch, int num_heads,
                       int max_seqlen_q, int total_q, int total_kv, float scale, void* out, float* lse,
                       void* stream) {
  if (batch < 1 || batch > 65535 || max_seqlen_q < 0 || total_q < 0 || total_kv < 0) return MLA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > 256) return MLA_ERR_UNSUPPORTED;
  if (!(scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (total_q == 0 || max_seqlen_q == 0) return MLA_OK;  // no new tokens: nothing to compute
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_kv || !prefix_lens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (total_kv < 1) return MLA_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  if (!status) return MLA_ERR_CUDA;
  const uint64_t H = static_cast<uint64_t>(num_heads);
  // q/k/v rows are viewed as [token][column block][64 columns] per head, 4-D
  // (columns, token, block, head): one box {64 columns, n tokens, all blocks, 1 head}
  // lands every 128-byte swizzled column block of a tile in a single TMA instruction.
  CUtensorMap tm_q, tm_k, tm_v;
  {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(total_q), 3, H};
    const uint64_t strides[3] = {H * 192 * 2, 128, 192 * 2};
    const uint32_t box[4] = {64, 128, 3, 1};
    if (!make_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(total_kv), 3, H};
    const uint64_t strides[3] = {H * 192 * 2, 128, 192 * 2};
    const uint32_t box[4] = {64, 128, 3, 1};
    if (!make_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(total_kv), 2, H};
    const uint64_t strides[3] = {H * 128 * 2, 128, 128 * 2};
    const uint32_t box[4] = {64, 128, 2, 1};
    if (!make_map(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dims, strides, box)) return MLA_ERR_CUDA;
  }
  PrefillParams p;
  memset(&p, 0, sizeof p);
  p.B = batch;
  p.H = num_heads;
  p.max_q_blocks = (max_seqlen_q + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.prefix_lens = prefix_lens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.max_seqlen_q = max_seqlen_q;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g_prof_start && record_event(g_prof_start, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_prefill(p, tm_q, tm_k, tm_v, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (g_prof_stop && record_event(g_prof_stop, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_prefill_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                      const int32_t* cu_seqlens_q, const int32_t* kv_lens, int batch, int num_heads, int page_size,
                      int max_pages_per_seq, int64_t num_pages, int max_seqlen_q, int total_q, float scale,
                      void* out, float* lse, void* stream) {
  if (batch < 1 || batch > 65535 || max_seqlen_q < 0 || total_q < 0 || max_pages_per_seq < 1 || num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > 256) return MLA_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128 && page_size != 256)
    return MLA_ERR_UNSUPPORTED;
  if (num_pages * page_size >= (int64_t(1) << 31)) return MLA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  if (!(scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (total_q == 0 || max_seqlen_q == 0) return MLA_OK;  // no new tokens: nothing to compute
  if (!q || !k_pages || !v_pages || !page_table || !cu_seqlens_q || !kv_lens || !out || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  unsigned* status = status_ptr();
  if (!status) return MLA_ERR_CUDA;
  const uint64_t H = static_cast<uint64_t>(num_heads);
  const uint64_t rows = static_cast<uint64_t>(num_pages) * page_size;
  // The pools are [num_pages * page_size rows][H][192 | 128]: the same 4-D view as the
  // contiguous prefill.  Pages of 128 or 256 keys take one box per 128-key tile; smaller
  // pages one box per (page, 64-column block).
  const uint32_t box_rows = static_cast<uint32_t>(page_size < 128 ? page_size : 128);
  const bool whole = page_size >= 128;
  CUtensorMap tm_q, tm_k, tm_v;
  {
    const uint64_t dims[4] = {64, static_cast<uint64_t>(total_q), 3, H};
    const uint64_t strides[3] = {H * 192 * 2, 128, 192 * 2};
    const uint32_t box[4] = {64, 128, 3, 1};
    if (!make_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {64, rows, 3, H};
    const uint64_t strides[3] = {H * 192 * 2, 128, 192 * 2};
    const uint32_t box[4] = {64, box_rows, whole ? 3u : 1u, 1};
    if (!make_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k_pages, dims, strides, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {64, rows, 2, H};
    const uint64_t strides[3] = {H * 128 * 2, 128, 128 * 2};
    const uint32_t box[4] = {64, box_rows, whole ? 2u : 1u, 1};
    if (!make_map(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v_pages, dims, strides, box)) return MLA_ERR_CUDA;
  }
  PrefillParams p;
  memset(&p, 0, sizeof p);
  p.B = batch;
  p.H = num_heads;
  p.max_q_blocks = (max_seqlen_q + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.cu_q = cu_seqlens_q;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.max_seqlen_q = max_seqlen_q;
  p.total_q = total_q;
  p.total_kv = static_cast<int>(rows);
  p.status = status;
  p.page_table = page_table;
  p.kv_lens = kv_lens;
  p.page_size = page_size;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g_prof_start && record_event(g_prof_start, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_prefill(p, tm_q, tm_k, tm_v, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (g_prof_stop && record_event(g_prof_stop, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_set_profile_events(void* start_event, void* stop_event) {
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return MLA_OK;
}

int mla_profile_elapsed_ms(void* start_event, void* stop_event, float* ms_out) {
  if (!start_event || !stop_event || !ms_out) return MLA_ERR_INVALID_ARG;
  if (cudaEventElapsedTime(ms_out, static_cast<cudaEvent_t>(start_event), static_cast<cudaEvent_t>(stop_event)) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_selftest_wait_timeout(void* stream) {
  unsigned* status = status_ptr();
  if (!status) return MLA_ERR_CUDA;
  if (launch_selftest_timeout(status, static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_get_status(void* stream) {
  unsigned* status = status_ptr();
  if (!status) return MLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, status, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof host, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  if (host & kStatusTimeout) return MLA_ERR_TIMEOUT;
  if (host & kStatusDeviceArg) return MLA_ERR_DEVICE_ARG;
  return MLA_OK;
}

}  // extern "C"
