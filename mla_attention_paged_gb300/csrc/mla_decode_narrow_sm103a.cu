// mla_decode_narrow_sm103a.cu -- absorbed MLA decode over a paged bf16 latent cache for
// narrow requests (q_len * heads <= 32 folded rows, e.g. 16 heads with one or two drafts),
// sm_103a.
//
// It computes exactly what decode_partial_kernel<bf16> (mla_decode_sm103a.cu) computes and
// writes the same outputs (final rows and LSE, or split partials for the combine):
//   out[b,t,h,:] = sum_j softmax_j(scale * q[b,t,h,:] . k_j) * k_j[:512]
// over keys j = 0 .. L_b - T + t of request b.  TokenSpeed pages: "构建面向 Agentic 推理的下一代
// LLM 推理引擎" (AICon talk), section "Kernel：让 MLA 真正跑满 GPU" (fold factor, split-KV
// partials, TMEM accumulators, KV bandwidth as the limit); launch-blog repost, section
// "TokenSpeed 性能预览" (query-sequence axis folded into the head axis).
//
// What changes against the general kernel, and why.  That kernel keeps the folded Q tile in
// shared memory (72 KB), which leaves room for two 72 KB key tiles: a stage stays busy from
// its copy until the BMM2 that reads it completes, so two stages pace the loop at about
// half that lifetime, above a tile's share of HBM bandwidth.  Here Q lives in tensor
// memory as the A operand of BMM1 (M = 128; folded row r in lane 32*(r/16) + r%16, so S
// has the M = 64 layout the softmax reads, other lanes zero), and shared memory holds
// three key tiles.  Tensor memory then holds O^T (4 x 32 columns: at most 32 rows), one S
// buffer (64) and Q (288 of 512 columns).  Q is copied by TMA into the third stage and
// moved into tensor memory by the softmax warps before that stage's first tile is loaded.
//
// Roles (192 threads): warps 0-3 softmax and epilogue, warp 4 TMA producer, warp 5 MMA
// issuer.
#include "mla_internal.h"
#include "sm103a_ptx.cuh"

namespace mla {
namespace {

constexpr int kDimBlocks = kLatentDim / 64;           // 9 blocks of 64 columns (128 bytes)
constexpr int kBlockBytes = 64 * 128;                 // 64 rows x 128 bytes, swizzled
constexpr int kTileBytes = kDimBlocks * kBlockBytes;  // 73728: one 64-key latent tile
constexpr int kStages = 3;
constexpr int kQStage = 2;      // Q lands here; it is free for tile kQStage once Q is in TMEM
constexpr int kNarrowRows = 32; // folded rows per request this kernel handles (at most)
constexpr int kThreads = 192;

// Shared memory map: stage0 | stage1 | stage2 | P | ctrl
constexpr int kOffStages = 0;
constexpr int kOffP = kOffStages + kStages * kTileBytes;  // P: 32 rows x 64 keys, swizzled
constexpr int kOffCtrl = kOffP + kNarrowRows * 128;

struct NarrowCtrl {
  uint64_t q_full;             // Q landed in stage kQStage
  uint64_t q_ready;            // Q copied into TMEM (softmax warps)
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];  // BMM2 of the tile in this stage completed
  uint64_t s_full;
  uint64_t s_free;
  uint64_t p_full;
  uint64_t o_done;
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
  int rescale_flag[2];
  alignas(16) float alpha[kNarrowRows];
  alignas(16) float row_scale[kNarrowRows];
};
constexpr int kCtrlBytes = 1024;
constexpr int kSmemBytes = kOffCtrl + kCtrlBytes + 1024;  // + control block + alignment slack
static_assert(sizeof(NarrowCtrl) <= kCtrlBytes, "control block");
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kOffP % 1024 == 0, "swizzled P tile alignment");

constexpr int kAbortTimeout = 1;

// Tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O^T chunk qc (value dims 128qc .. 128qc+127 x rows) at 32qc
constexpr uint32_t kTmemS = 128;  // S: 64 keys
constexpr uint32_t kTmemQ = 192;  // Q: column block c (64 dims) at 192 + 32c, 288 columns
static_assert(kTmemQ + kDimBlocks * 32 <= kTmemCols, "TMEM budget");
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__global__ void __launch_bounds__(kThreads, 1)
decode_partial_narrow_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                             const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  NarrowCtrl* ctrl = reinterpret_cast<NarrowCtrl*>(smem + kOffCtrl);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // grid (row groups, requests, splits) for a multi-wave plan: the hardware starts CTAs in
  // linear block order, so every request's first split is dispatched before any second
  // split; (row groups, splits, requests) otherwise
  const int b = p.split_major ? blockIdx.y : blockIdx.z;
  const int split = p.split_major ? blockIdx.z : blockIdx.y;

  // Set-up that reads no input of this call (overlaps the previous kernel's tail under
  // programmatic dependent launch; griddepcontrol.wait then orders every input read).
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    mbar_init(&ctrl->q_full, 1);
    mbar_init(&ctrl->q_ready, 128);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctrl->kv_full[s], 1);
      mbar_init(&ctrl->kv_empty[s], 1);
    }
    mbar_init(&ctrl->s_full, 1);
    mbar_init(&ctrl->s_free, 128);
    mbar_init(&ctrl->p_full, 128);
    mbar_init(&ctrl->o_done, 1);
    mbar_init(&ctrl->mma_drain, 1);
    ctrl->abort_flag = 0;
    ctrl->rescale_flag[0] = ctrl->rescale_flag[1] = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) tma_prefetch_desc(&tm_kv);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int L = p.seq_lens[b];
  const bool bad_len = L < p.T || L > p.max_seq || L > p.max_pages * p.page_size;
  if (bad_len && threadIdx.x == 0 && split == 0) atomicOr(p.status, kStatusDeviceArg);
  const int kv_start = split * p.chunk;
  if (bad_len || kv_start >= L) {  // (CTA-uniform) a bad length, or this request needs fewer splits
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int kv_end = min(L, kv_start + p.chunk);
  const int ntiles = (kv_end - kv_start + kTileKeys - 1) / kTileKeys;
  const int nsplit_b = (L + p.chunk - 1) / p.chunk;
  const int nrows = min(kNarrowRows, p.R);
  const int nq = (nrows + 15) & ~15;  // BMM2 N (16 or 32)
  if (threadIdx.x == 0) {
    // Q: the 64-row box from this request's first row (rows past its R are not used)
    mbar_arrive_expect_tx(&ctrl->q_full, kTileBytes);
    tma_load_3d(smem + kOffStages + kQStage * kTileBytes, &tm_q, &ctrl->q_full, 0, b * p.R, 0,
                policy_evict_last());
  }
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
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
    int last_issued[kStages] = {-1, -1, -1};
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
      // A page id outside the pool becomes -1 (reported after the loop): its box then lies
      // wholly before the first row, and TMA fills it with zeros instead of reading.
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const bool outside = pp < npg && static_cast<unsigned>(pids[pp]) >= n_pages;
        bad_pid |= outside;
        pids[pp] = outside ? -1 : pids[pp];
      }
      if (j == kQStage || j >= kStages) {
        // the stage is free once Q has left it (first use of stage kQStage) or once the
        // BMM2 of the tile before in this stage has completed
        bool w = true;
        if (lane == 0)
          w = (j < kStages) ? mbar_wait(&ctrl->q_ready, 0, abort_flag)
                            : mbar_wait(&ctrl->kv_empty[s], ((j / kStages) - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, w, 0);
        if (!ok) break;
      }
      if (lane == 0) {
        const int row_in_page = (P > kTileKeys) ? (k0 % P) : 0;
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
    const uint32_t idesc1 = make_idesc_bf16(128, 64, false, false);
    const uint32_t idesc2 = make_idesc_bf16(128, nq, true, false);
    const uint64_t p_desc = make_smem_desc(smem_u32(smem + kOffP), 16, 1024);
    auto poll = [&](uint64_t* bar, uint32_t parity) -> bool {
      uint32_t v = 0;
      if (lane == 0) v = mbar_test_wait(bar, parity) ? 1u : 0u;
      return __shfl_sync(0xffffffffu, v, 0) != 0;
    };
    bool ok = mbar_wait(&ctrl->q_ready, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    // BMM2(n2) first when P is ready (it frees a stage), else BMM1(n1) once its tile has
    // landed and the softmax has read the previous S (one S buffer).
    int n1 = 0, n2 = 0;
    unsigned long long idle_since = 0;
    while (ok && n2 < ntiles) {
      bool progressed = false;
      if (n2 < n1 && poll(&ctrl->p_full, n2 & 1)) {
        tc_fence_after();
        const int s = n2 % kStages;
        // V^T: 128 value columns (two 64-column blocks, LBO apart) x 16 keys (two 8-key
        // groups, SBO apart), MN-major.  P^T: rows x 16 keys, K-major.
        const uint64_t v_desc = make_smem_desc(smem_u32(smem + kOffStages + s * kTileBytes), kBlockBytes, 1024);
        if (elect_one()) {
#pragma unroll
          for (int qc = 0; qc < 4; ++qc) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t voff = static_cast<uint64_t>((2 * qc * kBlockBytes + kk * 2048) >> 4);
              const uint64_t poff = static_cast<uint64_t>((kk * 32) >> 4);
              umma_bf16(tmem + kTmemO + qc * 32, v_desc + voff, p_desc + poff, idesc2, (n2 > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(&ctrl->o_done);
          umma_commit(&ctrl->kv_empty[s]);
        }
        __syncwarp();
        ++n2;
        progressed = true;
      } else if (n1 < ntiles && n1 < n2 + 2) {
        const int s = n1 % kStages;
        const bool data = poll(&ctrl->kv_full[s], (n1 / kStages) & 1);
        if (data && (n1 == 0 || poll(&ctrl->s_free, (n1 - 1) & 1))) {
          tc_fence_after();
          const uint64_t k_desc = make_smem_desc(smem_u32(smem + kOffStages + s * kTileBytes), 16, 1024);
          if (elect_one()) {
            // S[row, key] = sum over 576 dims: A = Q from TMEM (8 columns per 16 dims),
            // B = the key tile, K-major
#pragma unroll
            for (int c = 0; c < kDimBlocks; ++c) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t off = static_cast<uint64_t>((c * kBlockBytes + k * 32) >> 4);
                umma_bf16_ts(tmem + kTmemS, tmem + kTmemQ + c * 32 + k * 8, k_desc + off, idesc1, (c | k) != 0);
              }
            }
            umma_commit(&ctrl->s_full);
          }
          __syncwarp();
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
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    // Folded row r lives in TMEM lane 32*(r/16) + r%16, so warps 0 and 1 own rows 0-15 and
    // 16-31; warps 2 and 3 hold no rows but share the O^T rescale and the epilogue (each
    // warp reaches only its own 32-lane quarter of TMEM).  A row is split between lanes i
    // and i+16 of its warp: lane i takes keys 0-31 of every tile, lane i+16 keys 32-63.
    const int half = lane >> 4;
    const bool row_lane = half == 0;
    const int r = warp * 16 + (lane & 15);
    const bool owns_rows = warp < kNarrowRows / 16;  // (warp-uniform)
    const bool row_active = r < nrows;
    const int t = r / p.H;
    const int lim_abs = L - p.T + t;  // last visible key of this row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_used = -INFINITY;
    float l_sum = 0.f;

    // Q into TMEM: this thread writes its own lane (32*warp + lane) of the 288 Q columns,
    // the folded row's 576 values (lanes of no row, and rows past R, get zeros).
    bool failed = !mbar_wait(&ctrl->q_full, 0, abort_flag);
    if (!__any_sync(0xffffffffu, failed)) {
      const bool q_row = owns_rows && row_lane && row_active;
      const uint32_t q_s = smem_u32(smem + kOffStages + kQStage * kTileBytes) + r * 128;
#pragma unroll 1
      for (int c = 0; c < kDimBlocks; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
          if (q_row)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(q_s + c * kBlockBytes + ((k ^ (r & 7)) << 4)));
          v[4 * k] = w0;
          v[4 * k + 1] = w1;
          v[4 * k + 2] = w2;
          v[4 * k + 3] = w3;
        }
        tmem_st32(tmem + lane_base + kTmemQ + c * 32, v);
      }
      tmem_st_wait();
    }
    failed = bar_or(1, 128, failed || (*abort_flag != 0));
    if (!failed) {
      tc_fence_before();
      mbar_arrive(&ctrl->q_ready);
    }
    const float scale_log2 = p.scale_log2;

    for (int j = 0; !failed && j < ntiles; ++j) {
      const int k0 = kv_start + j * kTileKeys;
      bool need_rescale = false;
      float alpha = 1.f;
      uint32_t packed[16];
      bool fail = !mbar_wait(&ctrl->s_full, j & 1, abort_flag);
      fail = __any_sync(0xffffffffu, fail);
      if (!fail) {
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld16x32bx2_32(tmem + lane_base + kTmemS, sr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&ctrl->s_free);
        // keys i <= lim of this lane's 32-key half are visible
        const int lim = (owns_rows && row_active) ? (min(kv_end - 1, lim_abs) - k0 - 32 * half) : -1;
        online_softmax_step<32, true>(sr, lim, scale_log2, kRescaleThreshold, m_used, l_sum, packed, alpha,
                                      need_rescale);
      }
      if (!fail && j >= 1) {
        fail = !mbar_wait(&ctrl->o_done, (j - 1) & 1, abort_flag);
        fail = __any_sync(0xffffffffu, fail);
      }
      if (!fail && owns_rows) {
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
      {
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
      if (ctrl->rescale_flag[0] | ctrl->rescale_flag[1]) {
        // O^T[dim, row] *= alpha[row] for all 512 value columns; this thread owns TMEM lane
        // (warp*32 + lane) of each 32-column chunk.
        tc_fence_after();
        float al[kNarrowRows];
#pragma unroll
        for (int i = 0; i < kNarrowRows; i += 4) {
          const float4 f = *reinterpret_cast<const float4*>(&ctrl->alpha[i]);
          al[i] = f.x;
          al[i + 1] = f.y;
          al[i + 2] = f.z;
          al[i + 3] = f.w;
        }
#pragma unroll 1
        for (int qc = 0; qc < 4; ++qc) {
          uint32_t v[32];
          const uint32_t addr = tmem + lane_base + kTmemO + qc * 32;
          tmem_ld32(addr, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * al[i]);
          tmem_st32(addr, v);
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
      if (owns_rows && row_lane) {
        const float lse2 = (l_sum > 0.f) ? (m_used + __log2f(l_sum)) : -INFINITY;
        const float lse_nat = lse2 * 0.69314718055994530942f;
        ctrl->row_scale[r] = (l_sum > 0.f) ? (p.v_scale / l_sum) : 0.f;
        if (row_active) {
          const int64_t grow = static_cast<int64_t>(b) * p.R + r;
          if (final_out)
            p.lse[grow] = lse_nat;
          else
            p.ws_lse[(static_cast<int64_t>(b) * p.max_splits + split) * p.R + r] = lse_nat;
        }
      }
      named_bar_sync(1, 128);
      // Normalised O (bf16) is transposed through shared memory (stage 0 is free once the
      // last BMM2 has completed) so that global stores are whole 16-byte row chunks.
      const uint32_t stage_s = smem_u32(smem + kOffStages);  // [32][512] bf16
      float rs[kNarrowRows];
#pragma unroll
      for (int i = 0; i < kNarrowRows; i += 4) {
        const float4 f = *reinterpret_cast<const float4*>(&ctrl->row_scale[i]);
        rs[i] = f.x;
        rs[i + 1] = f.y;
        rs[i + 2] = f.z;
        rs[i + 3] = f.w;
      }
#pragma unroll 1
      for (int qc = 0; qc < 4; ++qc) {
        const int dim = qc * 128 + warp * 32 + lane;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kTmemO + qc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(v[i]) * rs[i]);
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(stage_s + (i * kValueDim + dim) * 2),
                       "h"(*reinterpret_cast<const uint16_t*>(&o)));
        }
      }
      const __nv_bfloat16* stage_h = reinterpret_cast<const __nv_bfloat16*>(smem + kOffStages);
      named_bar_sync(1, 128);
      constexpr int kChunksPerRow = kValueDim * 2 / 16;
      __nv_bfloat16* dst = final_out ? p.out + static_cast<int64_t>(b) * p.R * kValueDim
                                     : p.ws_o + (static_cast<int64_t>(b) * p.max_splits + split) * p.R * kValueDim;
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

}  // namespace

cudaError_t launch_decode_partial_narrow(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                         cudaStream_t stream) {
  if (p.R > kNarrowRows || p.kv_dtype != kKvBf16) return cudaErrorInvalidValue;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(decode_partial_narrow_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // programmatic dependent launch, as for the general kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.split_major ? dim3(1, p.B, p.max_splits) : dim3(1, p.max_splits, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_partial_narrow_kernel, tm_q, tm_kv, p);
}

}  // namespace mla
