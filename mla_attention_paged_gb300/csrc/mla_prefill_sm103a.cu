// mla_prefill_sm103a.cu -- ragged (no padding) causal MLA prefill on top of a cached
// prefix, sm_103a.  K/V come either as contiguous per-request rows or from a paged cache
// (per-head k/v pages behind a page table; the same kernel, a different producer).
//
// What it computes: request b has p_b cached prefix tokens followed by n_b new tokens; for
// new token i and head h,
//   out[i,h,:] = sum_{j <= p_b + i} softmax_j(scale * q[i,h,:] . k[j,h,:]) * v[j,h,:]
// with q/k 192 wide (128 no-rope + 64 rope) and v 128 wide.  TokenSpeed pages:
// "构建面向 Agentic 推理的下一代 LLM 推理引擎" (AICon talk), section "Kernel：让 MLA 真正跑满
// GPU", last paragraph (agent prefill hits a cached prefix >90% of the time and appends a
// few hundred tokens, so Q and KV lengths differ and the batch is variable-length without
// padding); launch-blog repost "英偉達力薦，小團隊兩個月開源一款「光速級」智能體推理引擎",
// section "TokenSpeed 性能預覽" (prefill with a long prefix KV cache, tuned softmax).
//
// Design on sm_103a (one CTA per (128-row query block, head, request), one CTA per SM,
// 352 threads: softmax warps 0-7, producer warp 8, BMM1 warp 9, BMM2 warp 10):
//  * Producer warp: TMA (128-byte swizzled, 4-D maps over (columns, token, column block,
//    head), one box per operand tile) loads the query block once and streams 128-key K (192
//    wide) and V (128 wide) tiles of the same head through two separate 2-stage mbarrier
//    rings: a K stage is refilled as soon as its BMM1 is done, a V stage once its BMM2 is,
//    so the K loads run ahead of the softmax instead of waiting for the whole tile.
//  * Two MMA warps (uniform control flow, one elected thread issues): the BMM1 warp puts
//    S = Q . K^T (M=128 rows, N=128 keys, K=192) into one of two TMEM S buffers; the BMM2
//    warp adds O += P . V (M=128, N=128, K=128) with P read straight from TMEM (the A
//    operand) and V MN-major from shared memory.  Issuing an MMA stalls while the tensor
//    pipe is busy, so with one issuer a ready BMM2 waited behind the next BMM1's 12 MMAs.
//  * Softmax warps (8: two per TMEM lane quadrant, each row = TMEM lane split between a
//    warp for keys 0-63 and one for keys 64-127 of every tile, which swap their partial
//    row maxima through shared memory): causal mask offset by the prefix only on tiles
//    that cross the diagonal, running max in the log2 domain with a lazy rescale of the
//    thread's half of its O row (only when the max grows by more than 2^8), exp2 on the
//    MUFU unit; P (bf16) is written back into the first 64 columns of the tile's own S
//    buffer, so it never touches shared memory.
//  * Epilogue: O / l to bf16 and the natural-log LSE, straight from TMEM (each half of a
//    row writes its 64 value columns; the row sum is the two halves' partial sums).
//  * Key-range split: a (request, head, q block) of at least kMinSplitTiles key tiles runs
//    as two CTAs over the first and second half of its tiles, so that the grid's CTAs are
//    small enough to even out over the SMs (a few hundred to ~750 tiles each, 3-4 per SM
//    otherwise, left SMs idle ~10 % of the call at its end).  Each half writes its
//    normalised partial and LSE (the first half into out / lse, the second into a scratch
//    slot), fences, and counts itself on the pair's counter; the half that arrives second
//    merges the two (weights exp(lse_i - max)) into out / lse and clears the counter.
//    Neither half ever waits for the other.
// Every wait is bounded; on expiry the CTA records a timeout in the status word, drains
// its in-flight copies and MMAs, frees TMEM and returns.
#include "mla_internal.h"
#include "sm103a_ptx.cuh"

namespace mla {

// Scratch of the key-range split: the second half's partial output (bf16, 128 rows x 128
// value columns) and LSE per slot, and each slot's arrival counter (cleared before every
// launch).
constexpr int kSplitSlots = 1024;
__device__ uint4 g_split_o[kSplitSlots * 128 * 128 * 2 / 16];
__device__ float g_split_lse[kSplitSlots * 128];
__device__ int g_split_count[kSplitSlots];

namespace {

constexpr int kDqk = 192;
constexpr int kDv = 128;
constexpr int kBM = 128;     // query rows per CTA
constexpr int kBN = 128;     // keys per tile
constexpr int kStages = 2;
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant, one per half of the key tile
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;   // issues BMM1 (and owns TMEM)
constexpr int kBmm2Warp = kSoftmaxWarps + 2;  // issues BMM2
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);

constexpr int kMinSplitTiles = 8;     // key tiles from which a q block is split in two
constexpr int kMaxSplitPairs = kSplitSlots;  // q blocks past the scratch slots are not split

constexpr int kQBlockBytes = kBM * 128;                // 16 KB per 64-column block
constexpr int kQBytes = (kDqk / 64) * kQBlockBytes;    // 48 KB
constexpr int kKVBlockBytes = kBN * 128;               // 16 KB
constexpr int kKBytes = (kDqk / 64) * kKVBlockBytes;   // 48 KB
constexpr int kVBytes = (kDv / 64) * kKVBlockBytes;    // 32 KB

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;               // K ring: 2 x 48 KB
constexpr int kOffV = kOffK + kStages * kKBytes;     // V ring: 2 x 32 KB
constexpr int kOffCtrl = kOffV + kStages * kVBytes;

struct PrefillCtrl {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t k_empty[kStages];   // BMM1 of the tile in this K stage has completed
  uint64_t v_full[kStages];
  uint64_t v_empty[kStages];   // BMM2 of the tile in this V stage has completed
  uint64_t s_full[2];
  uint64_t s_consumed[2];  // BMM2 has read the P held in this S buffer
  uint64_t p_full;
  uint64_t o_done;
  uint64_t mma_drain;
  uint64_t mma_drain2;     // the BMM2 warp's MMAs
  uint32_t tmem_base;
  int abort_flag;
  int split_arrival;       // key-range split: 0 if this half finished first, 1 if second
  float row_max[2][kBM];   // per half of the key tile: this tile's partial row maxima
  float row_sum[2][kBM];   // per half: partial row sums (epilogue)
};
constexpr int kSmemBytes = kOffCtrl + 4096 + 1024;
static_assert(sizeof(PrefillCtrl) <= 4096, "control block");

constexpr uint32_t kTmemCols = 512;  // O at 0..127, S/P buffers at 128..255 and 256..383
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 128;
constexpr float kRescaleThreshold = 8.0f;

// D[tmem] (+)= A[tmem] * B[smem desc]: the A operand (M rows x 16 K elements, bf16 packed
// two per 32-bit column, row = lane) is read from Tensor Memory.
__device__ __forceinline__ void umma_ts_bf16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kPaged: K/V rows of request b come from a paged cache (row j of the request is row j % P
// of page page_table[b][j / P] of the pools) instead of contiguous rows at cu_kv[b].
template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PrefillCtrl* ctrl = reinterpret_cast<PrefillCtrl*>(smem + kOffCtrl);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  // Longest work first: blockIdx.z is the rank of the request by its key count (descending,
  // ties by index) and blockIdx.x / 2 counts q blocks down from the last one, so the
  // in-order dispatch of the grid starts the longest CTAs first and the shorter ones fill
  // in behind them (per-CTA work spans a few hundred to a few thousand tiles across
  // requests).  blockIdx.x % 2 is the half of a split key range.
  __shared__ int s_req;
  int b = blockIdx.z;
  if (p.B <= kThreads) {
    if (threadIdx.x < p.B) {
      const int t = threadIdx.x;
      const int len_t = kPaged ? p.kv_lens[t] : p.cu_kv[t + 1] - p.cu_kv[t];
      int rank = 0;
      for (int u = 0; u < p.B; ++u) {
        const int len_u = kPaged ? p.kv_lens[u] : p.cu_kv[u + 1] - p.cu_kv[u];
        rank += (len_u > len_t || (len_u == len_t && u < t)) ? 1 : 0;
      }
      if (rank == static_cast<int>(blockIdx.z)) s_req = t;
    }
    __syncthreads();
    b = s_req;
  }
  const int n_qb = static_cast<int>(gridDim.x >> 1);
  const int qb = n_qb - 1 - static_cast<int>(blockIdx.x >> 1);
  const int part = static_cast<int>(blockIdx.x & 1u);

  const int q_start = p.cu_q[b];
  const int n_b = p.cu_q[b + 1] - q_start;
  // Device-side argument checks, before any load or store: the request's rows lie inside
  // q/out/lse and k/v (paged: its length fits its page-table row), its kv length is prefix
  // + new tokens, and its new tokens fit the grid the host sized from max_seqlen_q (rows
  // beyond it would be left unwritten).
  const int kv_start = kPaged ? 0 : p.cu_kv[b];
  const int kv_total = kPaged ? p.kv_lens[b] : p.cu_kv[b + 1] - kv_start;
  const int pre = kPaged ? kv_total - n_b : p.prefix_lens[b];
  const bool bad = n_b < 0 || pre < 0 || kv_total != pre + n_b || n_b > p.max_seqlen_q || q_start < 0 ||
                   kv_start < 0 || static_cast<int64_t>(q_start) + n_b > p.total_q ||
                   (kPaged ? static_cast<int64_t>(kv_total) > static_cast<int64_t>(p.max_pages) * p.page_size
                           : static_cast<int64_t>(kv_start) + kv_total > p.total_kv);
  if (bad) {
    if (threadIdx.x == 0 && qb == 0 && h == 0 && part == 0) atomicOr(p.status, kStatusDeviceArg);
    return;
  }
  const int row_begin = qb * kBM;
  if (row_begin >= n_b) return;
  const int rows = min(kBM, n_b - row_begin);
  const int kv_len = pre + row_begin + rows;  // keys any row of this block can see
  const int ntiles = (kv_len + kBN - 1) / kBN;
  const int diag_tile = (pre + row_begin) / kBN;  // first tile that may need the causal mask
  // key-range split: this CTA takes tiles [t_lo, t_lo + nloc) of the q block's ntiles
  const int slot = (static_cast<int>(blockIdx.z) * p.H + h) * n_qb + (n_qb - 1 - qb);
  const bool split = ntiles >= kMinSplitTiles && slot < kMaxSplitPairs;
  if (part == 1 && !split) return;  // (CTA-uniform, before any set-up)
  const int t_lo = (split && part == 1) ? ntiles / 2 : 0;
  const int nloc = split ? (part == 0 ? ntiles / 2 : ntiles - ntiles / 2) : ntiles;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctrl->k_full[s], 1);
      mbar_init(&ctrl->k_empty[s], 1);
      mbar_init(&ctrl->v_full[s], 1);
      mbar_init(&ctrl->v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->s_consumed[i], 1);
    }
    mbar_init(&ctrl->p_full, kSoftmaxThreads);
    mbar_init(&ctrl->o_done, 1);
    mbar_init(&ctrl->mma_drain, 1);
    mbar_init(&ctrl->mma_drain2, 1);
    ctrl->abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    // contiguous K/V: lane 0 streams the K ring, lane 1 the V ring (independent waits in
    // divergent lanes)
    if constexpr (!kPaged) {
      if (lane < 2) {
        const bool is_k = lane == 0;
        const uint64_t pol_kv = policy_evict_last();  // re-read by the other query blocks of this head
        if (is_k) {
          mbar_arrive_expect_tx(&ctrl->q_full, kQBytes);
          // one box: 128 rows x all three 64-column blocks of head h
          tma_load_4d(smem + kOffQ, &tm_q, &ctrl->q_full, 0, q_start + row_begin, 0, h, policy_evict_first());
        }
        uint64_t* full = is_k ? ctrl->k_full : ctrl->v_full;
        uint64_t* empty = is_k ? ctrl->k_empty : ctrl->v_empty;
        int last_issued[kStages] = {-1, -1};
        bool ok = true;
        for (int j = 0; j < nloc; ++j) {
          const int s = j % kStages;
          if (j >= kStages) {
            ok = mbar_wait(&empty[s], ((j / kStages) - 1) & 1, abort_flag);
            if (!ok) break;
          }
          const int row = kv_start + (t_lo + j) * kBN;
          if (is_k) {
            mbar_arrive_expect_tx(&full[s], kKBytes);
            tma_load_4d(smem + kOffK + s * kKBytes, &tm_k, &full[s], 0, row, 0, h, pol_kv);  // 128 rows x 3 blocks
          } else {
            mbar_arrive_expect_tx(&full[s], kVBytes);
            tma_load_4d(smem + kOffV + s * kVBytes, &tm_v, &full[s], 0, row, 0, h, pol_kv);  // 128 rows x 2 blocks
          }
          last_issued[s] = j;
        }
        if (!ok) {
          if (is_k) drain_wait(&ctrl->q_full, 0);
          for (int s = 0; s < kStages; ++s)
            if (last_issued[s] >= 0) drain_wait(&full[s], (last_issued[s] / kStages) & 1);
        }
      }
    } else {
      // Paged: lanes 0-15 stream the K ring, lanes 16-31 the V ring.  A tile of 128 keys is
      // one box per operand when a page holds 128 or 256 keys, else one box per (page,
      // 64-column block) of its 128 / P pages; the group's lanes take those boxes round-robin,
      // so that they are issued in parallel.  The group's first lane waits for the stage and
      // arms its barrier.  Page ids of the next tile are read before that wait.  An id
      // outside the pool, or a page past the request's end, becomes -1: its boxes lie before
      // the first row and TMA fills them with zeros (an id outside the pool is reported).
      const bool is_k = lane < 16;
      const int gl = lane & 15;
      const int leader = is_k ? 0 : 16;
      const unsigned gmask = is_k ? 0x0000FFFFu : 0xFFFF0000u;
      const uint64_t pol_kv = policy_evict_last();  // re-read by the other query blocks of this head
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctrl->q_full, kQBytes);
        tma_load_4d(smem + kOffQ, &tm_q, &ctrl->q_full, 0, q_start + row_begin, 0, h, policy_evict_first());
      }
      uint64_t* full = is_k ? ctrl->k_full : ctrl->v_full;
      uint64_t* empty = is_k ? ctrl->k_empty : ctrl->v_empty;
      const int P = p.page_size;
      const int npt = P >= kBN ? 1 : kBN / P;          // pages per tile: 1, 2, 4 or 8
      const int nblk = is_k ? kDqk / 64 : kDv / 64;     // boxes per page when P < 128
      const int nbox = P >= kBN ? 1 : npt * nblk;       // boxes per tile: at most 24, two per lane
      const int pages_b = (kv_total + P - 1) / P;
      const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
      const unsigned n_pages = static_cast<unsigned>(min(p.num_pages, static_cast<int64_t>(0x7fffffff)));
      bool bad_pid = false;
      auto page_id = [&](int jt, int bx) -> int {  // page of box bx of (absolute) tile jt, or -1
        const int pg = jt * kBN / P + (P >= kBN ? 0 : bx / nblk);
        int v = -1;
        if (bx < nbox && jt < t_lo + nloc && pg < pages_b) {
          v = __ldg(pt + pg);
          if (static_cast<unsigned>(v) >= n_pages) {
            bad_pid = true;
            v = -1;
          }
        }
        return v;
      };
      const CUtensorMap* map = is_k ? &tm_k : &tm_v;
      int last_issued[kStages] = {-1, -1};
      bool ok = true;
      int cur0 = page_id(t_lo, gl), cur1 = page_id(t_lo, gl + 16);
      for (int j = 0; j < nloc; ++j) {
        const int s = j % kStages;
        const int nxt0 = page_id(t_lo + j + 1, gl), nxt1 = page_id(t_lo + j + 1, gl + 16);
        if (j >= kStages) {
          bool w = true;
          if (gl == 0) w = mbar_wait(&empty[s], ((j / kStages) - 1) & 1, abort_flag);
          ok = __shfl_sync(gmask, w, leader);
          if (!ok) break;
        }
        uint8_t* dst = smem + (is_k ? kOffK + s * kKBytes : kOffV + s * kVBytes);
        if (gl == 0) mbar_arrive_expect_tx(&full[s], is_k ? kKBytes : kVBytes);
        __syncwarp(gmask);  // the barrier is armed before any of the group's copies can land
        if (P >= kBN) {
          if (gl == 0) tma_load_4d(dst, map, &full[s], 0, cur0 * P + ((t_lo + j) * kBN) % P, 0, h, pol_kv);
        } else {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int bx = gl + 16 * k;
            if (bx < nbox) {
              const int pp = bx / nblk, blk = bx % nblk;
              tma_load_4d(dst + blk * kKVBlockBytes + pp * P * 128, map, &full[s], 0, (k ? cur1 : cur0) * P, blk, h,
                          pol_kv);
            }
          }
        }
        last_issued[s] = j;
        cur0 = nxt0;
        cur1 = nxt1;
      }
      if (__any_sync(gmask, bad_pid) && gl == 0) atomicOr(p.status, kStatusDeviceArg);
      if (!ok && gl == 0) {
        if (is_k) drain_wait(&ctrl->q_full, 0);
        for (int s = 0; s < kStages; ++s)
          if (last_issued[s] >= 0) drain_wait(&full[s], (last_issued[s] / kStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ BMM1 issuer (whole warp,
    // uniform control flow; one elected thread issues the MMAs and their commits).  Issuing
    // blocks while the tensor pipe is busy, so BMM2 has a warp of its own: neither GEMM
    // waits behind the other's issue loop.
    const uint32_t idesc1 = make_idesc_bf16(kBM, kBN, false, false);
    const uint64_t q_desc = make_smem_desc(smem_u32(smem + kOffQ), 16, 1024);
    bool ok = mbar_wait(&ctrl->q_full, 0, abort_flag);
    // BMM1(j) once K(j) has landed and BMM2(j-2) has read the P in its S buffer (j counts
    // this CTA's tiles)
    for (int j = 0; j < nloc; ++j) {
      const int s = j % kStages, sb = j & 1;
      if (ok) ok = mbar_wait(&ctrl->k_full[s], (j / kStages) & 1, abort_flag);
      if (ok && j >= 2) ok = mbar_wait(&ctrl->s_consumed[sb], ((j - 2) >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint64_t k_desc = make_smem_desc(smem_u32(smem + kOffK + s * kKBytes), 16, 1024);
      if (elect_one()) {
#pragma unroll
        for (int c = 0; c < kDqk / 64; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tmem + kTmemS + sb * 128, q_desc + static_cast<uint64_t>((c * kQBlockBytes + k * 32) >> 4),
                      k_desc + static_cast<uint64_t>((c * kKVBlockBytes + k * 32) >> 4), idesc1, (c | k) != 0);
        }
        umma_commit(&ctrl->s_full[sb]);
        umma_commit(&ctrl->k_empty[s]);
      }
      __syncwarp();
    }
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain);
      drain_wait(&ctrl->mma_drain, 0);
    }
    __syncwarp();
  } else if (warp == kBmm2Warp) {
    // ------------------------------------------------------------------ BMM2 issuer: O += P . V
    // as soon as P(j) and V(j) are ready (it frees a V stage and an S buffer)
    const uint32_t idesc2 = make_idesc_bf16(kBM, kDv, false, true);
    bool ok = true;
    for (int j = 0; j < nloc; ++j) {
      const int s = j % kStages, sb = j & 1;
      if (ok) ok = mbar_wait(&ctrl->p_full, j & 1, abort_flag);
      if (ok) ok = mbar_wait(&ctrl->v_full[s], (j / kStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      // P: 128 rows x 16 keys per MMA, 8 TMEM columns apart.  V: 16 keys (two 8-key groups,
      // SBO apart) x 128 value columns (two 64-column blocks, LBO apart), MN-major.
      const uint64_t v_desc = make_smem_desc(smem_u32(smem + kOffV + s * kVBytes), kKVBlockBytes, 1024);
      const uint32_t p_tmem = tmem + kTmemS + sb * 128;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts_bf16(tmem + kTmemO, p_tmem + kk * 8, v_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc2,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&ctrl->o_done);
        umma_commit(&ctrl->v_empty[s]);
        umma_commit(&ctrl->s_consumed[sb]);
      }
      __syncwarp();
    }
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain2);
      drain_wait(&ctrl->mma_drain2, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-7)
    // Warp w serves TMEM lane quadrant w%4 (query rows 32(w%4) .. +31) and half hf = w/4 of
    // every key tile (keys 64hf .. 64hf+63); the two warps of a quadrant swap their partial
    // row maxima through shared memory (a 64-thread named barrier per quadrant) so that both
    // halves scale P by the same running maximum.
    const int quad = warp & 3;
    const int hf = warp >> 2;
    const int r = quad * 32 + lane;            // query row within the block = TMEM lane
    const bool row_active = r < rows;
    const int vis_last = pre + row_begin + r;  // last visible key of this row
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int pair_bar = 2 + quad;
    float m_used = -INFINITY;
    float l_sum = 0.f;  // this half's share of the row sum
    bool failed = false;
    for (int j = 0; j < nloc; ++j) {
      const int sb = j & 1;
      const int k0 = (t_lo + j) * kBN + 64 * hf;  // absolute key of this half's first column
      const uint32_t s_tmem = tmem + lane_base + kTmemS + sb * 128;
      bool fail = !mbar_wait(&ctrl->s_full[sb], (j >> 1) & 1, abort_flag);
      fail = __any_sync(0xffffffffu, fail);
      bool need_rescale = false;
      float alpha = 1.f;
      uint32_t sr[64];
      int lim = -1;
      if (!fail) {
        tc_fence_after();
        tmem_ld32(s_tmem + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(s_tmem + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld_wait();
        lim = (t_lo + j >= diag_tile) ? (row_active ? vis_last - k0 : -1) : (row_active ? 63 : -1);
        float mx = -INFINITY;
        if (lim >= 63) {
#pragma unroll
          for (int i = 0; i < 64; ++i) mx = fmaxf(mx, __uint_as_float(sr[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i <= lim) mx = fmaxf(mx, __uint_as_float(sr[i]));
        }
        ctrl->row_max[hf][r] = mx;
      }
      // both halves have loaded their S columns (P below overwrites columns 0..63) and
      // published their partial maxima
      named_bar_sync(pair_bar, 64);
      if (!fail) {
        const float mx = fmaxf(ctrl->row_max[0][r], ctrl->row_max[1][r]);
        const float mt = mx * p.scale_log2;
        if (m_used == -INFINITY) {
          m_used = mt;
        } else if (mt > m_used + kRescaleThreshold) {
          alpha = ex2_approx(m_used - mt);
          need_rescale = true;
          l_sum *= alpha;
          m_used = mt;
        }
        const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
        uint32_t packed[32];
        float l0 = 0.f, l1 = 0.f;
        if (lim >= 63) {
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[i]), p.scale_log2, neg_m));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[i + 1]), p.scale_log2, neg_m));
            l0 += p0;
            l1 += p1;
            packed[i >> 1] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float p0 = (i <= lim) ? ex2_approx(fmaf(__uint_as_float(sr[i]), p.scale_log2, neg_m)) : 0.f;
            const float p1 = (i + 1 <= lim) ? ex2_approx(fmaf(__uint_as_float(sr[i + 1]), p.scale_log2, neg_m)) : 0.f;
            l0 += p0;
            l1 += p1;
            packed[i >> 1] = pack_bf16x2(p0, p1);
          }
        }
        l_sum += l0 + l1;
        // P (bf16 pairs) of this half over columns 32hf .. 32hf+31 of the tile's S buffer
        tmem_st32(s_tmem + 32 * hf, packed);
      }
      if (!fail && j >= 1) {
        // O may only be rescaled once BMM2(j-1) has finished accumulating into it
        fail = !mbar_wait(&ctrl->o_done, (j - 1) & 1, abort_flag);
        fail = __any_sync(0xffffffffu, fail);
      }
      if (!fail && __any_sync(0xffffffffu, need_rescale) && j >= 1) {
        // rescale this thread's half of its O row (TMEM lane r, columns 64hf .. 64hf+63)
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          const uint32_t addr = tmem + lane_base + kTmemO + 64 * hf + c * 32;
          tmem_ld32(addr, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(addr, v);
        }
      }
      tmem_st_wait();
      if (bar_or(1, kSoftmaxThreads, fail || (*abort_flag != 0))) {
        failed = true;
        break;
      }
      tc_fence_before();
      mbar_arrive(&ctrl->p_full);
    }
    if (!failed) failed = !mbar_wait(&ctrl->o_done, (nloc - 1) & 1, abort_flag);
    if (!failed) ctrl->row_sum[hf][r] = l_sum;
    if (!bar_or(1, kSoftmaxThreads, failed || (*abort_flag != 0))) {
      tc_fence_after();
      const float l_tot = ctrl->row_sum[0][r] + ctrl->row_sum[1][r];
      const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
      const int64_t tok = static_cast<int64_t>(q_start) + row_begin + r;
      const float lse_own = (l_tot > 0.f) ? (m_used + __log2f(l_tot)) * 0.69314718055994530942f : -INFINITY;
      // this thread's 64 value columns of its row: in out, or (second half of a split) in
      // the slot's scratch row
      uint4* const out_row = reinterpret_cast<uint4*>(p.out + (tok * p.H + h) * kDv + 64 * hf);
      uint4* const scratch_row = g_split_o + (static_cast<int64_t>(slot) * kBM + r) * (kDv * 2 / 16) + hf * 8;
      uint4* const dst = (split && part == 1) ? scratch_row : out_row;
      float o[64];  // normalised O of this thread's columns (kept for a merge)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kTmemO + 64 * hf + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[32 * c + i] = __uint_as_float(v[i]) * inv;
        if (row_active) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* f = &o[32 * c + 8 * i];
            dst[4 * c + i] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                        pack_bf16x2(f[6], f[7]));
          }
        }
      }
      if (row_active && hf == 0) {
        if (split && part == 1)
          g_split_lse[slot * kBM + r] = lse_own;
        else
          p.lse[tok * p.H + h] = lse_own;
      }
      if (split) {
        // publish this half's partial, then count it; the half that counts second merges
        __threadfence();
        named_bar_sync(1, kSoftmaxThreads);
        if (threadIdx.x == 0) ctrl->split_arrival = atomicAdd(&g_split_count[slot], 1);
        named_bar_sync(1, kSoftmaxThreads);
        if (ctrl->split_arrival == 1) {
          __threadfence();
          if (row_active) {
            // The same arithmetic whichever half arrives second: both halves' bf16 partials
            // (this half's as it wrote them), combined first half first.
            const float lse_oth = (part == 1) ? __ldcg(p.lse + tok * p.H + h) : __ldcg(g_split_lse + slot * kBM + r);
            const uint4* const oth = (part == 1) ? out_row : scratch_row;
            const float lse0 = part == 0 ? lse_own : lse_oth;
            const float lse1 = part == 0 ? lse_oth : lse_own;
            const float m = fmaxf(lse0, lse1);
            const float w0 = (lse0 == -INFINITY) ? 0.f : __expf(lse0 - m);
            const float w1 = (lse1 == -INFINITY) ? 0.f : __expf(lse1 - m);
            const float tot = w0 + w1;
            const float a0 = (tot > 0.f) ? w0 / tot : 0.f;
            const float a1 = (tot > 0.f) ? w1 / tot : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 u = __ldcg(oth + i);
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
              uint32_t pk[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
                const float own_x = __bfloat162float(__float2bfloat16_rn(o[8 * i + 2 * k]));
                const float own_y = __bfloat162float(__float2bfloat16_rn(o[8 * i + 2 * k + 1]));
                const float x0 = part == 0 ? own_x : f.x, x1 = part == 0 ? f.x : own_x;
                const float y0 = part == 0 ? own_y : f.y, y1 = part == 0 ? f.y : own_y;
                pk[k] = pack_bf16x2(__fmaf_rn(a1, x1, __fmul_rn(a0, x0)), __fmaf_rn(a1, y1, __fmul_rn(a0, y0)));
              }
              out_row[i] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            if (hf == 0) p.lse[tok * p.H + h] = (tot > 0.f) ? m + __logf(tot) : -INFINITY;
          }
          if (threadIdx.x == 0) g_split_count[slot] = 0;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && ctrl->abort_flag) atomicOr(p.status, kStatusTimeout);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, cudaStream_t stream) {
  // the shared-memory limit is a per-device attribute: set it once per device, thread and instance
  static thread_local int configured_device[2] = {-1, -1};
  const bool paged = p.page_table != nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device[paged] != dev) {
    e = paged ? cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)
              : cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device[paged] = dev;
  }
  if (p.max_q_blocks < 1) return cudaSuccess;
  // the split counters start at zero (the merging half clears its own; a launch that gave
  // up part-way may not have)
  static thread_local int count_device = -1;
  static thread_local void* count_ptr = nullptr;
  if (count_device != dev) {
    e = cudaGetSymbolAddress(&count_ptr, g_split_count);
    if (e != cudaSuccess) return e;
    count_device = dev;
  }
  const long long slots = static_cast<long long>(p.B) * p.H * p.max_q_blocks;
  e = cudaMemsetAsync(count_ptr, 0, sizeof(int) * static_cast<size_t>(slots < kSplitSlots ? slots : kSplitSlots),
                      stream);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.max_q_blocks, p.H, p.B);
  if (paged)
    prefill_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(tm_q, tm_k, tm_v, p);
  else
    prefill_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(tm_q, tm_k, tm_v, p);
  return cudaGetLastError();
}

}  // namespace mla
