// mla_decode_sm103a.cu -- absorbed MLA decode over a paged latent KV cache (bf16 or int8
// pool), sm_103a.  (An e4m3 pool runs decode_partial_e4m3_kernel, mla_decode_e4m3_sm103a.cu.)
//
// What it computes (per request b, draft t, head h; keys j = 0 .. L_b - T + t):
//   out[b,t,h,:] = sum_j softmax_j(scale * q[b,t,h,:] . k_j) * k_j[:512]
// where k_j is the 576-wide latent row j of request b, found through the page table (an
// int8 pool is decoded exactly to f16 and its per-tensor scale folded into the softmax
// scale and the output).  With T beyond a few drafts the same computation is the
// prefill of T new tokens over a paged prefix in absorbed form.  TokenSpeed pages: "构建面向 Agentic 推理的下一代 LLM 推理引擎"
// (AICon talk), section "Kernel：让 MLA 真正跑满 GPU" (latent state shared by all heads,
// fold factor, split-KV partial + reduction stages, TMEM accumulators, KV bandwidth as the
// limit even with 8-bit KV); launch-blog repost "英偉達力薦，小團隊兩個月開源一款「光速級」
// 智能體推理引擎", section "TokenSpeed 性能預覽" (query-sequence axis folded into the head
// axis to fill the first matmul's M tile).
//
// Design on sm_103a (one CTA per (64-row group, split, request); one CTA per SM):
//  * Fold: the T*H query rows of a request are one matrix with row m = t*H + h; a CTA
//    takes 64 consecutive rows, so all heads and drafts share each latent tile load.
//  * Producer warp: bf16 pools are gathered by TMA (one 3-D box per 64-key tile: 64 rows x
//    nine 128-byte-swizzled column blocks) from the pages named by the page table, into a
//    2-stage ring.  For int8 pools, six decode warps (4 and 6-10) read each tile's rows
//    from the page pool into registers, wait for the stage, and write them as f16 into the
//    same swizzled layout (exact decode: int8 codes as themselves); the BMM1 warp prefetches
//    rows into L2 a few tiles ahead of them.  The int8 GEMMs run on f16 operands (Q
//    converted once per CTA, P in f16), issued by two warps (BMM1 by warp 5, BMM2 by the
//    last warp), each waiting on its own inputs; one polling warp for both left each GEMM
//    waiting behind the other's issue.  (The bf16 path keeps one issuer for both: split,
//    it measured slower there.)
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kv8_decode.cuh"
#include "mla_internal.h"
#include "sm103a_ptx.cuh"

namespace mla {
namespace {

constexpr int kDimBlocks = kLatentDim / 64;          // 9 blocks of 64 columns (128 bytes)
constexpr int kBlockBytes = 64 * 128;                // 64 rows x 128 bytes, swizzled
constexpr int kTileBytes = kDimBlocks * kBlockBytes; // 73728: one bf16 64-key latent tile
constexpr int kStages = 2;
constexpr int kPrefetchTiles = 3;  // int8 pools: tiles ahead of the decode that are prefetched into L2
// Warps 0-3 softmax/epilogue, 5 MMA; bf16: warp 4 producer (192 threads); int8 pools:
// warps 4 and 6-10 decode (352 threads), each lane holding four rows' codes of its tile.
constexpr int kDecodeWarps = 6;
constexpr int kDequantThreads = 32 * kDecodeWarps;
// int8: softmax warps 0-3, decode warp 4, BMM1 warp 5, decode warps 6 .. 4 + kDecodeWarps,
// BMM2 warp 5 + kDecodeWarps
__host__ __device__ constexpr int threads_for(bool fp8) { return fp8 ? 32 * (6 + kDecodeWarps) : 192; }
constexpr int kBmm2WarpInt8 = 5 + kDecodeWarps;
static_assert(threads_for(true) / 32 - 1 == kBmm2WarpInt8, "the last int8 warp is the BMM2 issuer");
static_assert(1 + (kBmm2WarpInt8 - 6) == kDecodeWarps, "decode warps: 4 and 6 .. kBmm2WarpInt8 - 1");

// Shared memory map: Q | stage0 | stage1 | P | ctrl.  A stage holds one 64-key tile as nine
// 128-byte-swizzled column blocks: bf16 as loaded by TMA, or (int8 pools) f16 as decoded
// by the dequant warps from rows they read straight from global memory.
constexpr int kOffQ = 0;
constexpr int kOffStages = kOffQ + kTileBytes;
constexpr int kOffP = kOffStages + kStages * kTileBytes;
constexpr int kOffCtrl = kOffP + kBlockBytes;

struct DecodeCtrl {
  uint64_t q_full;
  uint64_t kv_full[kStages];   // tile landed (bf16: TMA bytes; int8: dequant threads)
  uint64_t kv_empty[kStages];  // BMM2 of the tile in this stage completed
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t q_ready;            // int8 pools: Q converted to f16 in place
  uint64_t mma_drain;
  uint64_t mma_drain2;         // int8: the BMM2 warp's MMAs
  uint32_t tmem_base;
  int abort_flag;
  int rescale_flag[4];
  alignas(16) float alpha[kGroupRows];
  alignas(16) float row_scale[kGroupRows];
  // int8 pools with a scale per page: each key's scale relative to kv_scale, per stage
  alignas(16) float key_scale[kStages][kTileKeys];
};
constexpr int kCtrlBytes = 2048;
constexpr int kSmemBytes = kOffCtrl + kCtrlBytes + 1024;  // + control block + alignment slack
static_assert(sizeof(DecodeCtrl) <= kCtrlBytes, "control block");
static_assert(kSmemBytes <= 232448, "shared memory per block");

// Values of the CTA's abort flag: a bounded wait ran out, or a device argument check failed.
constexpr int kAbortTimeout = 1;
constexpr int kAbortBadArg = 2;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;   // S buffers at columns 256 and 320; O^T chunks at 0,64,128,192
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// kKv: pool format (kKvBf16, kKvInt8 or kKvInt8Page; kInt8 below selects the decode warps
// and f16 GEMMs of the int8 paths, kPageScales the per-key scales of kKvInt8Page).
// kSplitMajor: the grid's launch order (a compile-time choice: a run-time select of the
// block-index mapping measured 1.4 % slower on 128-head decode).
template <int kKv, bool kSplitMajor>
__global__ void __launch_bounds__(threads_for(kKv != kKvBf16), 1)
decode_partial_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                      const DecodeParams p) {
  constexpr bool kInt8 = kKv == kKvInt8 || kKv == kKvInt8Page;
  constexpr bool kPageScales = kKv == kKvInt8Page;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DecodeCtrl* ctrl = reinterpret_cast<DecodeCtrl*>(smem + kOffCtrl);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = blockIdx.x;
  // grid (row groups, requests, splits) for a multi-wave plan: the hardware starts CTAs in
  // linear block order, so every request's first split is dispatched before any second
  // split; (row groups, splits, requests) otherwise
  const int b = kSplitMajor ? blockIdx.y : blockIdx.z;
  const int split = kSplitMajor ? blockIdx.z : blockIdx.y;

  // Set-up that reads no input of this call: barriers, TMEM, descriptor prefetch.  The
  // kernel is launched as a programmatic dependent of the stream's previous kernel, so this
  // part may overlap that kernel's tail; griddepcontrol.wait below then holds every thread
  // until that kernel has completed and its writes are visible.
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    mbar_init(&ctrl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctrl->kv_full[s], kInt8 ? kDequantThreads : 1);
      mbar_init(&ctrl->kv_empty[s], kInt8 ? 2 : 1);  // int8: BMM1 and BMM2 come from two warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->s_free[i], 128);
    }
    mbar_init(&ctrl->p_full, 128);
    mbar_init(&ctrl->o_done, 1);
    mbar_init(&ctrl->q_ready, kDequantThreads);
    mbar_init(&ctrl->mma_drain, 1);
    mbar_init(&ctrl->mma_drain2, 1);
    ctrl->abort_flag = 0;
    for (int w = 0; w < 4; ++w) ctrl->rescale_flag[w] = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0 && !kInt8) tma_prefetch_desc(&tm_kv);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int L = p.seq_lens[b];
  const bool bad_len = L < p.T || L > p.max_seq || L > p.max_pages * p.page_size;
  if (bad_len && threadIdx.x == 0 && split == 0 && group == 0) atomicOr(p.status, kStatusDeviceArg);
  const int kv_start = split * p.chunk;
  if (bad_len || kv_start >= L) {  // (CTA-uniform) a bad length, or this request needs fewer splits
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);  // no tensor-core work was issued
    return;
  }
  const int kv_end = min(L, kv_start + p.chunk);
  const int ntiles = (kv_end - kv_start + kTileKeys - 1) / kTileKeys;
  const int nsplit_b = (L + p.chunk - 1) / p.chunk;
  const int row0 = group * kGroupRows;
  const int nrows = min(kGroupRows, p.R - row0);
  const int nq = (nrows + 15) & ~15;  // BMM2 N (multiple of 16)
  if (threadIdx.x == 0) {
    // Q: nine 64-column blocks of the 64 folded rows
    mbar_arrive_expect_tx(&ctrl->q_full, kTileBytes);
    tma_load_3d(smem + kOffQ, &tm_q, &ctrl->q_full, 0, b * p.R + row0, 0, policy_evict_last());
  }
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == 4 && !kInt8) {
    // ------------------------------------------------------------------ producer (bf16)
    const int P = p.page_size;
    const int sub = P < kTileKeys ? kTileKeys / P : 1;  // pages per tile
    const int box_rows = P < kTileKeys ? P : kTileKeys;
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
    const int first_page = kv_start / P;
    const int last_page = (kv_end - 1) / P;
    int batch_base = first_page;
    int cur = (first_page + lane <= last_page) ? __ldg(pt + first_page + lane) : 0;
    int nxt = (first_page + 32 + lane <= last_page) ? __ldg(pt + first_page + 32 + lane) : 0;
    const uint64_t pol_kv = policy_evict_first();
    const unsigned n_pages = static_cast<unsigned>(min(p.num_pages, static_cast<int64_t>(0x7fffffff)));
    bool bad_pid = false;
    int last_issued[kStages] = {-1, -1};
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kStages;
      const int k0 = kv_start + j * kTileKeys;
      const int pg0 = k0 / P;
      const int tile_end = min(k0 + kTileKeys, L);
      const int npg = (P < kTileKeys) ? ((tile_end - 1) / P - pg0 + 1) : 1;
      int pids[8];
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const int pi = pg0 + pp;
        if (pp < sub) {
          while (pi - batch_base >= 32) {  // advance the page-id window (warp-uniform)
            batch_base += 32;
            cur = nxt;
            const int nb = batch_base + 32 + lane;
            nxt = (nb <= last_page) ? __ldg(pt + nb) : 0;
          }
          pids[pp] = __shfl_sync(0xffffffffu, cur, (pi - batch_base) & 31);
        } else {
          pids[pp] = 0;
        }
      }
      // A page id outside the pool is replaced by -1 (reported after the loop): its box
      // then lies wholly before the first row, and TMA fills it with zeros instead of reading.
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const bool outside = pp < npg && static_cast<unsigned>(pids[pp]) >= n_pages;
        bad_pid |= outside;
        pids[pp] = outside ? -1 : pids[pp];
      }
      // The page ids above are resolved before waiting for the stage, so that only the
      // copies are left once it frees up (resolving them after the wait was measured to
      // delay each tile's copies by ~1.5k cycles).
      if (j >= kStages) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&ctrl->kv_empty[s], ((j / kStages) - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, w, 0);
        if (!ok) break;
      }
      if (lane == 0) {
        const int row_in_page = (P > kTileKeys) ? (k0 % P) : 0;
        {
          uint8_t* stage = smem + kOffStages + s * kTileBytes;
          mbar_arrive_expect_tx(&ctrl->kv_full[s], static_cast<uint32_t>(npg * box_rows * 128 * kDimBlocks));
          if (P >= kTileKeys) {  // one 3-D box: 64 rows x all 9 column blocks
            tma_load_3d(stage, &tm_kv, &ctrl->kv_full[s], 0, pids[0] * P + row_in_page, 0, pol_kv);
          } else {
            for (int pp = 0; pp < npg; ++pp) {
              const int y = pids[pp] * P;
              for (int c = 0; c < kDimBlocks; ++c)
                tma_load_2d(stage + c * kBlockBytes + pp * box_rows * 128, &tm_kv, &ctrl->kv_full[s], c * 64, y,
                            pol_kv);
            }
          }
        }
      }
      last_issued[s] = j;
      __syncwarp();
    }
    if (bad_pid && lane == 0) atomicOr(p.status, kStatusDeviceArg);
    if (!ok && lane == 0) {
      // drain copies still in flight before the CTA exits
      drain_wait(&ctrl->q_full, 0);
      for (int s = 0; s < kStages; ++s)
        if (last_issued[s] >= 0) drain_wait(&ctrl->kv_full[s], (last_issued[s] / kStages) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer (whole warp,
    // uniform control flow; one elected thread issues each GEMM's MMAs and their commit)
    // the int8 path multiplies f16 operands (Q converted once, K/V decoded to f16, P in f16)
    const uint32_t idesc1 = kInt8 ? make_idesc_f16(64, 64, false, false) : make_idesc_bf16(64, 64, false, false);
    const uint32_t idesc2 = kInt8 ? make_idesc_f16(128, nq, true, false) : make_idesc_bf16(128, nq, true, false);
    // Descriptors are built once; each MMA advances the start-address field by a
    // compile-time offset (addresses stay below 256 KB, so no carry leaves the field).
    const uint64_t q_desc = make_smem_desc(smem_u32(smem + kOffQ), 16, 1024);
    const uint64_t p_desc = make_smem_desc(smem_u32(smem + kOffP), 16, 1024);
    auto poll = [&](uint64_t* bar, uint32_t parity) -> bool {
      uint32_t v = 0;
      if (lane == 0) v = mbar_test_wait(bar, parity) ? 1u : 0u;
      return __shfl_sync(0xffffffffu, v, 0) != 0;
    };
    // int8 pools: lanes < sub (pages per tile) prefetch their page of tile n1 + 1 + kPrefetchTiles
    // into L2 each time BMM1(n1) is issued, with the page id looked up one BMM1 earlier.
    const int P = p.page_size;
    const int sub = P < kTileKeys ? kTileKeys / P : 1;
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
    auto page_of = [&](int jt) -> int {  // page index of this lane's page of tile jt, or -1
      const int k = kv_start + jt * kTileKeys + lane * P;
      return (lane < sub && jt < ntiles && k < kv_end) ? k / P : -1;
    };
    const unsigned n_pages = static_cast<unsigned>(min(p.num_pages, static_cast<int64_t>(0x7fffffff)));
    auto prefetch = [&](int jt, int pid) {
      if (static_cast<unsigned>(pid) >= n_pages) return;  // none, or outside the pool (the decode warps report it)
      const int k = kv_start + jt * kTileKeys + lane * P;
      const int rows = min(min(P, kTileKeys), kv_end - k);
      prefetch_l2_bulk(p.kv_pool + (static_cast<int64_t>(pid) * P + k % P) * kLatentDim,
                       static_cast<uint32_t>(rows * kLatentDim));
    };
    int pf_pid = -1;
    if (kInt8) {
      for (int jt = 1; jt <= kPrefetchTiles; ++jt) {
        const int pg = page_of(jt);
        if (pg >= 0) prefetch(jt, __ldg(pt + pg));
      }
      const int pg = page_of(1 + kPrefetchTiles);
      pf_pid = (pg >= 0) ? __ldg(pt + pg) : -1;
      __syncwarp();
    }
    bool ok = kInt8 ? mbar_wait(&ctrl->q_ready, 0, abort_flag) : mbar_wait(&ctrl->q_full, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if constexpr (kInt8) {
      // int8 pools: this warp issues BMM1 only (BMM2 has its own warp): BMM1(n1) once tile
      // n1 has been decoded and its S buffer is free.  Its commit on the stage's empty
      // barrier is the first of two (the BMM2 warp's is the other).
      for (int n1 = 0; ok && n1 < ntiles; ++n1) {
        const int s = n1 % kStages, sb = n1 & 1;
        bool w = mbar_wait(&ctrl->kv_full[s], (n1 / kStages) & 1, abort_flag);
        if (w && n1 >= 2) w = mbar_wait(&ctrl->s_free[sb], ((n1 - 2) >> 1) & 1, abort_flag);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        const uint64_t k_desc = make_smem_desc(smem_u32(smem + kOffStages + s * kTileBytes), 16, 1024);
        const uint32_t d = tmem + kTmemS + sb * 64;
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < kDimBlocks; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t off = static_cast<uint64_t>((c * kBlockBytes + k * 32) >> 4);
              umma_bf16(d, q_desc + off, k_desc + off, idesc1, (c | k) != 0);
            }
          }
          umma_commit(&ctrl->s_full[sb]);
          umma_commit(&ctrl->kv_empty[s]);
        }
        __syncwarp();
        prefetch(n1 + 1 + kPrefetchTiles, pf_pid);
        const int pg = page_of(n1 + 2 + kPrefetchTiles);
        pf_pid = (pg >= 0) ? __ldg(pt + pg) : -1;
        __syncwarp();
      }
      ok = false;  // (the loop below is the bf16 path's)
    }
    // Issue whichever GEMM is ready: BMM2(n2) first (it frees a stage), else BMM1(n1) for a
    // tile whose data has landed and whose S buffer is free.  BMM1 runs at most two tiles
    // ahead of BMM2 (double-buffered S).
    int n1 = 0, n2 = 0;
    unsigned long long idle_since = 0;
    while (ok && n2 < ntiles) {
      bool progressed = false;
      if (n2 < n1 && poll(&ctrl->p_full, n2 & 1)) {
        tc_fence_after();
        const int s = n2 % kStages;
        const uint32_t kv_base = smem_u32(smem + kOffStages + s * kTileBytes);
        // V^T: 128 value columns (two 64-column blocks, LBO apart) x 16 keys (two 8-key
        // groups, SBO apart), MN-major.  P^T: rows x 16 keys, K-major.
        const uint64_t v_desc = make_smem_desc(kv_base, kBlockBytes, 1024);
        if (elect_one()) {
#pragma unroll
          for (int qc = 0; qc < 4; ++qc) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t voff = static_cast<uint64_t>((2 * qc * kBlockBytes + kk * 2048) >> 4);
              const uint64_t poff = static_cast<uint64_t>((kk * 32) >> 4);
              umma_bf16(tmem + qc * 64, v_desc + voff, p_desc + poff, idesc2, (n2 > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(&ctrl->o_done);
          umma_commit(&ctrl->kv_empty[s]);
        }
        __syncwarp();
        ++n2;
        progressed = true;
      } else if (n1 < ntiles && n1 < n2 + 2) {
        const int s = n1 % kStages, sb = n1 & 1;
        const bool data = poll(&ctrl->kv_full[s], (n1 / kStages) & 1);
        if (data && (n1 < 2 || poll(&ctrl->s_free[sb], ((n1 - 2) >> 1) & 1))) {
          tc_fence_after();
          const uint64_t k_desc = make_smem_desc(smem_u32(smem + kOffStages + s * kTileBytes), 16, 1024);
          const uint32_t d = tmem + kTmemS + sb * 64;
          if (elect_one()) {
#pragma unroll
            for (int c = 0; c < kDimBlocks; ++c) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t off = static_cast<uint64_t>((c * kBlockBytes + k * 32) >> 4);
                umma_bf16(d, q_desc + off, k_desc + off, idesc1, (c | k) != 0);
              }
            }
            umma_commit(&ctrl->s_full[sb]);
          }
          __syncwarp();
          if (kInt8) {
            prefetch(n1 + 1 + kPrefetchTiles, pf_pid);
            const int pg = page_of(n1 + 2 + kPrefetchTiles);
            pf_pid = (pg >= 0) ? __ldg(pt + pg) : -1;
            __syncwarp();
          }
          ++n1;
          progressed = true;
        }
      }
      if (progressed) {
        idle_since = 0;
      } else {
        uint32_t give_up = 0;
        if (lane == 0) {
          const unsigned long long now = global_timer_ns();
          if (idle_since == 0) {
            idle_since = now;
          } else if (*abort_flag) {
            give_up = 1;
          } else if (now - idle_since > kWaitLimitNs) {
            *abort_flag = kAbortTimeout;
            give_up = 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, give_up, 0) == 0;
      }
    }
    // every MMA issued so far completes before TMEM is released
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain);
      drain_wait(&ctrl->mma_drain, 0);
    }
    __syncwarp();
  } else if (kInt8 && warp == kBmm2WarpInt8) {
    // ------------------------------------------------------------------ int8 pools: BMM2 issuer
    // O^T += V^T . P^T once the softmax has written P(n2); V from the decoded stage (waited
    // for here too, so that this warp orders its reads after the decode warps' writes).
    const uint32_t idesc2 = make_idesc_f16(128, nq, true, false);
    const uint64_t p_desc = make_smem_desc(smem_u32(smem + kOffP), 16, 1024);
    bool ok = true;
    for (int n2 = 0; ok && n2 < ntiles; ++n2) {
      const int s = n2 % kStages;
      bool w = mbar_wait(&ctrl->p_full, n2 & 1, abort_flag);
      if (w) w = mbar_wait(&ctrl->kv_full[s], (n2 / kStages) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      const uint64_t v_desc = make_smem_desc(smem_u32(smem + kOffStages + s * kTileBytes), kBlockBytes, 1024);
      if (elect_one()) {
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t voff = static_cast<uint64_t>((2 * qc * kBlockBytes + kk * 2048) >> 4);
            const uint64_t poff = static_cast<uint64_t>((kk * 32) >> 4);
            umma_bf16(tmem + qc * 64, v_desc + voff, p_desc + poff, idesc2, (n2 > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&ctrl->o_done);
        umma_commit(&ctrl->kv_empty[s]);
      }
      __syncwarp();
    }
    // every MMA this warp issued completes before TMEM is released
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain2);
      drain_wait(&ctrl->mma_drain2, 0);
    }
    __syncwarp();
  } else if (kInt8 && warp >= 4) {
    // ------------------------------------------------------------------ int8 dequant (warps 4, 6-10):
    // Q to f16 in place once; then, per tile, each lane reads its rows' int8 bytes straight
    // from the page pool into registers (issued before waiting for the stage, so the reads
    // overlap the previous tile's GEMMs), waits for the stage, and writes them as f16 into
    // the swizzled tile.  Lane dl of decode warp dw (0..5) owns rows 32 (dw / 3) + dl/4 + 8i
    // (i < 4) and 16-byte chunk dl % 4 of column blocks dw % 3, + 3 and + 6.  (The MMA warp prefetches
    // the rows into L2 kPrefetchTiles tiles ahead.)
    const int dw = (warp == 4) ? 0 : warp - 5;
    const int dl = lane;
    const int td = dw * 32 + dl;
    const int bg = dw % 3;                        // column blocks bg, bg + 3, bg + 6
    const int rbase0 = 32 * (dw / 3) + (dl >> 2);  // first owned row; then every 8th, four in all
    const int P = p.page_size;
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
    // Every page id this split reads (rows kv_start .. kv_end - 1) is checked once, before
    // any row is read; the loads are issued here and overlap the Q conversion.  An id
    // outside the pool stops the CTA (reported as a device argument error below).  The
    // check stays out of the tile loop, whose loads it would otherwise delay.
    bool bad_id = false;
    {
      const unsigned n_pages = static_cast<unsigned>(min(p.num_pages, static_cast<int64_t>(0x7fffffff)));
      for (int pg = kv_start / P + td; pg <= (kv_end - 1) / P; pg += kDequantThreads) {
        const unsigned pid = static_cast<unsigned>(__ldg(pt + pg));
        bad_id |= pid >= n_pages;
        if (kPageScales && pid < n_pages) {
          // a page's scale relative to kv_scale must be finite and in [0, 255], so that
          // P times it stays within f16's range
          const float rel = __ldg(p.page_scales + pid) * p.inv_ref_scale;
          bad_id |= !(rel >= 0.f && rel <= 255.f);
        }
      }
    }
    bool ok = mbar_wait(&ctrl->q_full, 0, abort_flag);
    if (ok) {
      const uint32_t q_s = smem_u32(smem + kOffQ);
      for (int c = td; c < kTileBytes / 16; c += kDequantThreads) {
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(q_s + c * 16));
        st_shared_v4(q_s + c * 16, bf16x2_to_f16x2(w0), bf16x2_to_f16x2(w1), bf16x2_to_f16x2(w2),
                     bf16x2_to_f16x2(w3));
      }
      fence_proxy_async_smem();
      mbar_arrive(&ctrl->q_ready);
    }
    if (bar_or(2, kDequantThreads, bad_id)) {
      if (td == 0) {
        atomicOr(p.status, kStatusDeviceArg);
        *abort_flag = kAbortBadArg;  // the other roles leave their loops at their next wait
      }
      ok = false;
    }
    // page id of each owned row of tile j (0 past the request end: the row is not read)
    auto row_pids = [&](int j, int (&pid)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = kv_start + j * kTileKeys + rbase0 + 8 * i;
        pid[i] = (k < L) ? __ldg(pt + k / P) : 0;
      }
    };
    int pid_cur[4];
    row_pids(0, pid_cur);
    // per-page scales: eight lanes of each of decode warps 0 and 3 hold the scale (relative
    // to kv_scale) of each of their 32 rows of a tile, loaded one tile ahead; rows past the
    // request end get 0
    const bool scale_lane = kPageScales && bg == 0 && (dl & 3) == 0;
    auto row_rels = [&](int j, const int (&pid)[4], float (&rel)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = kv_start + j * kTileKeys + rbase0 + 8 * i;
        rel[i] = (scale_lane && k < L) ? __ldg(p.page_scales + pid[i]) * p.inv_ref_scale : 0.f;
      }
    };
    float rel_cur[4];
    if (kPageScales) row_rels(0, pid_cur, rel_cur);
    for (int j = 0; ok && j < ntiles; ++j) {
      const int s = j % kStages;
      const int k0 = kv_start + j * kTileKeys;
      uint4 w[3][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = k0 + rbase0 + 8 * i;
        const uint8_t* row = p.kv_pool + (static_cast<int64_t>(pid_cur[i]) * P + k % P) * kLatentDim + (dl & 3) * 16;
        const bool valid = k < L;
#pragma unroll
        for (int m = 0; m < 3; ++m)
          w[m][i] = valid ? __ldg(reinterpret_cast<const uint4*>(row + (bg + 3 * m) * 64)) : make_uint4(0u, 0u, 0u, 0u);
      }
      int pid_nxt[4];
      float rel_nxt[4];
      if (j + 1 < ntiles) {
        row_pids(j + 1, pid_nxt);
        if (kPageScales) row_rels(j + 1, pid_nxt, rel_nxt);
      }
      // the stage is free once BMM2(j - 2) has completed
      if (j >= kStages) ok = mbar_wait(&ctrl->kv_empty[s], ((j / kStages) - 1) & 1, abort_flag);
      if (!ok) break;
      if (scale_lane) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ctrl->key_scale[s][rbase0 + 8 * i] = rel_cur[i];
      }
      const uint32_t st = smem_u32(smem + kOffStages + s * kTileBytes) + (dl & 3) * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = rbase0 + 8 * i;
        const uint32_t rbase = st + row * 128;
        const int sw = (row & 7) << 4;
#pragma unroll
        for (int m = 0; m < 3; ++m) store_f16_chunk_int8(rbase + (bg + 3 * m) * kBlockBytes, sw, w[m][i]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&ctrl->kv_full[s]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pid_cur[i] = pid_nxt[i];
        if (kPageScales) rel_cur[i] = rel_nxt[i];
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    // BMM1 runs with M = 64: folded row r lives in TMEM lane 32*(r/16) + r%16, so warp w
    // owns rows 16w .. 16w+15.  Each row is split between lanes i and i+16 of its warp:
    // lane i takes keys 0-31 of every tile, lane i+16 keys 32-63.
    const int half = lane >> 4;
    const bool row_lane = half == 0;  // the lane that writes per-row results
    const int r = warp * 16 + (lane & 15);
    const bool row_active = r < nrows;
    const int t = (row0 + r) / p.H;
    const int lim_abs = L - p.T + t;  // last visible key of this row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_used = -INFINITY;
    float l_sum = 0.f;
    bool failed = false;
    // (int8 codes are decoded to their exact values: the scales apply as they are)
    const float scale_log2 = p.scale_log2;
    const float v_scale = p.v_scale;

    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      const int k0 = kv_start + j * kTileKeys;
      bool need_rescale = false;
      float alpha = 1.f;
      uint32_t packed[16];
      bool fail = !mbar_wait(&ctrl->s_full[sb], (j >> 1) & 1, abort_flag);
      fail = __any_sync(0xffffffffu, fail);
      if (!fail) {
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld16x32bx2_32(tmem + lane_base + kTmemS + sb * 64, sr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&ctrl->s_free[sb]);
        // keys i <= lim of this lane's 32-key half are visible
        const int lim = row_active ? (min(kv_end - 1, lim_abs) - k0 - 32 * half) : -1;
        if constexpr (kPageScales) {
          // the keys' scales relative to kv_scale (written by the decode warps before they
          // released the tile: waiting on that release orders their writes before the reads)
          fail = __any_sync(0xffffffffu, !mbar_wait(&ctrl->kv_full[j % kStages], (j / kStages) & 1, abort_flag));
          float ks[32];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 f = *reinterpret_cast<const float4*>(&ctrl->key_scale[j % kStages][32 * half + i]);
            ks[i] = f.x;
            ks[i + 1] = f.y;
            ks[i + 2] = f.z;
            ks[i + 3] = f.w;
          }
          online_softmax_step<32, true, true, true>(sr, lim, scale_log2, kRescaleThreshold, m_used, l_sum, packed,
                                                    alpha, need_rescale, ks);
        } else {
          // the int8 path multiplies P in f16 (P <= 2^8 here, where f16 keeps more bits than bf16)
          online_softmax_step<32, true, kInt8>(sr, lim, scale_log2, kRescaleThreshold, m_used, l_sum, packed,
                                              alpha, need_rescale);
        }
      }
      if (!fail && j >= 1) {
        fail = !mbar_wait(&ctrl->o_done, (j - 1) & 1, abort_flag);
        fail = __any_sync(0xffffffffu, fail);
      }
      if (!fail) {
        // this lane's half of P row r (32 keys = four 16-byte chunks) into the
        // 128-byte-swizzled K-major block
        const uint32_t row_addr = smem_u32(smem + kOffP) + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = 4 * half + c;
          st_shared_v4(row_addr + ((chunk ^ (r & 7)) << 4), packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                       packed[4 * c + 3]);
        }
        if (row_lane) ctrl->alpha[r] = alpha;
        const bool any = __any_sync(0xffffffffu, need_rescale);
        if (lane == 0) ctrl->rescale_flag[warp] = any ? 1 : 0;
      }
      fence_proxy_async_smem();
      if (bar_or(1, 128, fail || (*abort_flag != 0))) {
        failed = true;
        break;
      }
      if (!kInt8) {
        // zero value rows past the request's end in the last tile (stale or unloaded rows
        // would otherwise meet P = 0 in BMM2 and could carry NaN/Inf bit patterns)
        const int valid_rows = L - k0;
        if (valid_rows < kTileKeys) {
          uint8_t* stage = smem + kOffStages + (j % kStages) * kTileBytes;
          const int nzero = (kTileKeys - valid_rows) * 8;  // 16-byte chunks per block
          for (int idx = threadIdx.x; idx < nzero * 8; idx += 128) {
            const int blk = idx / nzero;
            const int rem = idx % nzero;
            const int row = valid_rows + rem / 8;
            st_shared_v4(smem_u32(stage + blk * kBlockBytes + row * 128 + (rem % 8) * 16), 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
      }
      if (ctrl->rescale_flag[0] | ctrl->rescale_flag[1] | ctrl->rescale_flag[2] | ctrl->rescale_flag[3]) {
        // O^T[dim, row] *= alpha[row] for all 512 value columns; this thread owns TMEM lane
        // (warp*32 + lane) of each 128-column chunk.
        tc_fence_after();
        if constexpr (kInt8) {
          // (the int8 kernels run at a lower register cap: rows 32hh .. 32hh+31 at a time,
          // so that only their 32 factors are held in registers)
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            float al[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 f = *reinterpret_cast<const float4*>(&ctrl->alpha[hh * 32 + i]);
              al[i] = f.x;
              al[i + 1] = f.y;
              al[i + 2] = f.z;
              al[i + 3] = f.w;
            }
#pragma unroll 1
            for (int qc = 0; qc < 4; ++qc) {
              uint32_t v[32];
              const uint32_t addr = tmem + lane_base + qc * 64 + hh * 32;
              tmem_ld32(addr, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * al[i]);
              tmem_st32(addr, v);
            }
          }
        } else {
#pragma unroll 1
          for (int qc = 0; qc < 4; ++qc) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t v[32];
              const uint32_t addr = tmem + lane_base + qc * 64 + hh * 32;
              tmem_ld32(addr, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * ctrl->alpha[hh * 32 + i]);
              tmem_st32(addr, v);
            }
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&ctrl->p_full);
    }

    if (!failed) {
      failed = !mbar_wait(&ctrl->o_done, (ntiles - 1) & 1, abort_flag);
    }
    if (bar_or(1, 128, failed || (*abort_flag != 0))) {
      failed = true;
    } else {
      tc_fence_after();
      const bool final_out = (nsplit_b == 1);
      l_sum += __shfl_xor_sync(0xffffffffu, l_sum, 16);  // the two halves' partial row sums
      if (row_lane) {
        const float lse2 = (l_sum > 0.f) ? (m_used + __log2f(l_sum)) : -INFINITY;
        const float lse_nat = lse2 * 0.69314718055994530942f;
        ctrl->row_scale[r] = (l_sum > 0.f) ? (v_scale / l_sum) : 0.f;
        if (row_active) {
          const int64_t grow = static_cast<int64_t>(b) * p.R + row0 + r;
          if (final_out)
            p.lse[grow] = lse_nat;
          else
            p.ws_lse[(static_cast<int64_t>(b) * p.max_splits + split) * p.R + row0 + r] = lse_nat;
        }
      }
      named_bar_sync(1, 128);
      // Normalised O (bf16) is transposed through shared memory (the KV stage area is free
      // once the last BMM2 has completed) so that global stores are whole 16-byte row
      // chunks.  Split partials are kept in bf16 too: they are averaged by the combine and
      // rounded to the bf16 output anyway, and half the bytes is half the extra traffic.
      // The 64 row scales go to registers first: shared-memory loads interleaved with the
      // staging stores below would each have to wait for the stores before them.
      const uint32_t stage_s = smem_u32(smem + kOffStages);  // [64][512] bf16
      if constexpr (kInt8) {
        // (the int8 kernels run at a lower register cap: rows 32hh .. 32hh+31 at a time,
        // their 32 scales in registers)
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float rs[32];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 f = *reinterpret_cast<const float4*>(&ctrl->row_scale[hh * 32 + i]);
            rs[i] = f.x;
            rs[i + 1] = f.y;
            rs[i + 2] = f.z;
            rs[i + 3] = f.w;
          }
#pragma unroll 1
          for (int qc = 0; qc < 4; ++qc) {
            const int dim = qc * 128 + warp * 32 + lane;
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + qc * 64 + hh * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(v[i]) * rs[i]);
              asm volatile("st.shared.b16 [%0], %1;" ::"r"(stage_s + ((hh * 32 + i) * kValueDim + dim) * 2),
                           "h"(*reinterpret_cast<const uint16_t*>(&o)));
            }
          }
        }
      } else {
        float rs[kGroupRows];
#pragma unroll
        for (int i = 0; i < kGroupRows; i += 4) {
          const float4 f = *reinterpret_cast<const float4*>(&ctrl->row_scale[i]);
          rs[i] = f.x;
          rs[i + 1] = f.y;
          rs[i + 2] = f.z;
          rs[i + 3] = f.w;
        }
#pragma unroll 1
        for (int qc = 0; qc < 4; ++qc) {
          const int dim = qc * 128 + warp * 32 + lane;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + qc * 64 + hh * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int rr = hh * 32 + i;
              const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(v[i]) * rs[rr]);
              asm volatile("st.shared.b16 [%0], %1;" ::"r"(stage_s + (rr * kValueDim + dim) * 2),
                           "h"(*reinterpret_cast<const uint16_t*>(&o)));
            }
          }
        }
      }
      __nv_bfloat16* stage_h = reinterpret_cast<__nv_bfloat16*>(smem + kOffStages);
      named_bar_sync(1, 128);
      constexpr int kChunksPerRow = kValueDim * 2 / 16;
      __nv_bfloat16* dst = final_out
                               ? p.out + (static_cast<int64_t>(b) * p.R + row0) * kValueDim
                               : p.ws_o + ((static_cast<int64_t>(b) * p.max_splits + split) * p.R + row0) * kValueDim;
      for (int c = threadIdx.x; c < nrows * kChunksPerRow; c += 128) {
        const int rr = c / kChunksPerRow, cc = c % kChunksPerRow;
        const uint4 v = *reinterpret_cast<const uint4*>(stage_h + rr * kValueDim + cc * 8);
        *reinterpret_cast<uint4*>(dst + rr * kValueDim + cc * 8) = v;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && ctrl->abort_flag == kAbortTimeout) atomicOr(p.status, kStatusTimeout);
  // every store of this CTA is issued: the combine grid may be scheduled now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------------------------------
// Combine: out[b, row] = sum_s exp(lse_s - lse) * O_s,  lse = log sum_s exp(lse_s).
// One 128-thread CTA per (request, kCombineRows folded rows).  One thread copies the rows'
// partials of a batch of splits (each a contiguous 1 KB per row) into shared memory with
// bulk copies, so that the TMA engine rather than per-thread loads moves them; meanwhile
// each warp loads its row's log-sum-exps and reduces the weights with shuffles.  Thread t
// then accumulates value columns 8(t%64)..8(t%64)+7 of row t/64 from shared memory.  A
// running maximum rescales earlier batches when a request has more than kCombineBatch
// splits.
// --------------------------------------------------------------------------------------
constexpr int kCombineRows = 2;
constexpr int kCombineThreads = 64 * kCombineRows;
constexpr int kCombineBatch = 32;  // splits staged per round (lane l holds split s0 + l)
constexpr int kCombineRowBytes = kValueDim * 2;

__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t cs[];  // [split][row][512] bf16
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int row0 = blockIdx.x * kCombineRows;
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nr = min(kCombineRows, p.R - row0);
  const int r = tid / 64;   // row of this thread within the CTA
  const int c8 = tid % 64;  // value columns 8*c8 .. 8*c8+7
  const bool active = r < nr;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent of the stream's previous kernel (the partial
  // kernel inside mla_decode): wait for it to complete before reading any input, the
  // lengths included, since a caller's own kernel between the two stages may write them.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int L = p.seq_lens[b];
  if (L < p.T || L > p.max_seq) return;  // (CTA-uniform; the partial kernel reported it)
  const int ns = (L + p.chunk - 1) / p.chunk;
  if (ns <= 1) return;
  const int64_t base = static_cast<int64_t>(b) * p.max_splits;
  const float* lse_s = p.ws_lse + base * p.R + row0 + (active ? r : 0);
  float m_run = -INFINITY, w_run = 0.f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  bool ok = true;
  uint32_t phase = 0;
  for (int s0 = 0; s0 < ns && ok; s0 += kCombineBatch) {
    const int nb = min(kCombineBatch, ns - s0);
    if (tid == 0) {
      mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(nb * nr * kCombineRowBytes));
      const uint64_t pol = policy_evict_first();
      for (int s = 0; s < nb; ++s)
        bulk_load(cs + s * nr * kCombineRowBytes, p.ws_o + ((base + s0 + s) * p.R + row0) * kValueDim,
                  static_cast<uint32_t>(nr * kCombineRowBytes), &bar, pol);
    }
    const float l = (lane < nb) ? __ldg(lse_s + static_cast<int64_t>(s0 + lane) * p.R) : -INFINITY;
    float bm = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    const float m_new = fmaxf(m_run, bm);
    if (m_new != -INFINITY) {
      const float c = __expf(m_run - m_new);  // 0 while nothing has been accumulated
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= c;
      w_run *= c;
      m_run = m_new;
    }
    const float w = (m_new == -INFINITY) ? 0.f : __expf(l - m_new);
    float ws = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    w_run += ws;
    ok = mbar_wait(&bar, phase, &abort_flag);
    phase ^= 1u;
    if (ok) {
      const uint32_t src = smem_u32(cs) + (active ? r : 0) * kCombineRowBytes + c8 * 16;
      for (int s = 0; s < nb; ++s) {
        const float ws_s = __shfl_sync(0xffffffffu, w, s);
        uint32_t v0, v1, v2, v3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                     : "r"(src + s * nr * kCombineRowBytes));
        const uint32_t vv[4] = {v0, v1, v2, v3};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vv[i]));
          acc[2 * i] += ws_s * f.x;
          acc[2 * i + 1] += ws_s * f.y;
        }
      }
    }
    ok = __syncthreads_and(ok) != 0;  // the staging area is reused by the next batch
  }
  if (!ok) {
    if (tid == 0) {
      atomicOr(p.status, kStatusTimeout);
      drain_wait(&bar, phase ^ 1u);  // copies still in flight land before the CTA exits
    }
    return;
  }
  if (active) {
    const float inv = w_run > 0.f ? 1.f / w_run : 0.f;
    uint4 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    const int64_t orow = static_cast<int64_t>(b) * p.R + row0 + r;
    *reinterpret_cast<uint4*>(p.out + orow * kValueDim + c8 * 8) = pk;
    if (c8 == 0) p.lse[orow] = (w_run > 0.f) ? (m_run + __logf(w_run)) : -INFINITY;
  }
}

// Watchdog self-test: wait on an mbarrier that nothing ever arrives on, through the same
// bounded wait the kernels above use; the wait must give up and record a timeout.
__global__ void selftest_timeout_kernel(unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0, &abort_flag);
  __syncthreads();
  if (threadIdx.x == 0 && (!ok || abort_flag)) atomicOr(status, kStatusTimeout);
}

template <int kKv>
cudaError_t launch_partial_impl(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                int head_groups, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(decode_partial_kernel<kKv, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_partial_kernel<kKv, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // programmatic dependent launch: the kernel's set-up may overlap the previous kernel,
  // whose completion it awaits (griddepcontrol.wait) before reading any input
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.split_major ? dim3(head_groups, p.B, p.max_splits) : dim3(head_groups, p.max_splits, p.B);
  cfg.blockDim = dim3(threads_for(kKv != kKvBf16));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.split_major ? cudaLaunchKernelEx(&cfg, decode_partial_kernel<kKv, true>, tm_q, tm_kv, p)
                       : cudaLaunchKernelEx(&cfg, decode_partial_kernel<kKv, false>, tm_q, tm_kv, p);
}

}  // namespace

cudaError_t launch_decode_partial(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                  int head_groups, cudaStream_t stream) {
  switch (p.kv_dtype) {
    case kKvE4m3: return launch_decode_partial_e4m3(p, tm_q, tm_kv, head_groups, stream);
    case kKvInt8: return launch_partial_impl<kKvInt8>(p, tm_q, tm_kv, head_groups, stream);
    case kKvInt8Page: return launch_partial_impl<kKvInt8Page>(p, tm_q, tm_kv, head_groups, stream);
    default:
      // at most 32 folded rows: Q fits in tensor memory, and shared memory takes three tiles
      if (p.R <= 32) return launch_decode_partial_narrow(p, tm_q, tm_kv, stream);
      return launch_partial_impl<kKvBf16>(p, tm_q, tm_kv, head_groups, stream);
  }
}

cudaError_t launch_selftest_timeout(unsigned* status, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const dim3 grid((p.R + kCombineRows - 1) / kCombineRows, p.B);
  const int smem = min(p.max_splits, kCombineBatch) * kCombineRows * kCombineRowBytes;
  // the shared-memory limit is a per-device attribute: set it once per device and thread
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(decode_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCombineBatch * kCombineRows * kCombineRowBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, p);
}

}  // namespace mla
