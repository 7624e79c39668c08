// mla_decode_e4m3_sm103a.cu -- absorbed MLA decode over an FP8 (e4m3fn) paged latent KV
// cache, sm_103a.
//
// What it computes is the decode of mla_decode_sm103a.cu (per request b, draft t, head h,
// keys j = 0 .. L_b - T + t: out = sum_j softmax_j(scale * q . k_j) * k_j[:512]) with the
// latent rows stored as e4m3 codes times one per-tensor kv_scale.  TokenSpeed pages: "构建面向
// Agentic 推理的下一代 LLM 推理引擎" (AICon talk), section "Kernel：让 MLA 真正跑满 GPU" (latent
// state shared by all heads, split-KV partial + reduction stages, 8-bit KV still
// bandwidth-bound); launch-blog repost "英偉達力薦，小團隊兩個月開源一款「光速級」智能體推理引擎",
// section "TokenSpeed 性能預覽" (query-sequence axis folded into the head axis).
//
// Design on sm_103a (one CTA per (64-row group, split, request); one CTA per SM; 352
// threads: softmax warps 0-7, producer warp 8, BMM1 warp 9, BMM2 warp 10).  Both GEMMs run on
// the 8-bit codes as they arrive (kind::f8f6f4); nothing is decoded to a wider type:
//  * The raw e4m3 tile (64 keys x 576 codes, 36 KB) arrives by TMA (64-byte swizzle) in a
//    5-stage ring.  (Five stages cover the load latency: an L2 prefetch ahead of the ring,
//    which an earlier 4-stage ring needed, now only delayed the producer's loads.)
//  * Q keeps its bf16 value: each query row, scaled by a power of two 2^s that brings its
//    largest element into [128, 256), is split into q_hi = e4m3(q 2^s) and
//    q_lo = e4m3(q 2^s - q_hi), an 8-bit significand in two 4-bit halves.  This is exact
//    for every element within 2^9 of the row's largest |q|; smaller elements fall under
//    e4m3's subnormal floor (2^-9 at that scale) and carry an absolute error of at most
//    2^-17 of the row's largest |q|.
//  * BMM1 (M = 128, N = 64 keys, K = 576): the A operand stacks q_hi and q_lo, 8 rows of
//    each in turn, so that row r's hi and lo partial scores land in TMEM lanes i and i + 8
//    (i = 16 (r / 8) + r % 8).  The 16x256b load shape hands both lanes' values for the
//    same columns to one thread, which adds them.  One pass of full-rate MMAs reads the K
//    tile once.  The split's column blocks 0-7 sit in TMEM (the A operand from tensor
//    memory: stacked row = lane, four codes per 32-bit column), the rope block 8 in shared
//    memory; the stacked Q is then not re-read from shared memory on every tile.
//  * BMM2 (O^T += V^T . P^T, M = 128 value columns, N = rows, K = 64 keys) takes V straight
//    from the raw stage as an MN-major e4m3 operand.  P is split in two 8-bit parts: the
//    softmax forms P 2^6 (at most 2^8, because the running max moves once a tile's max
//    exceeds it by more than 2 in the log2 domain) and writes p_hi = e4m3(P 2^6) and
//    p_lo = e5m2(P 2^6 - p_hi); two MMA passes (e4m3 x e4m3, e4m3 x e5m2) add both.  Their
//    sum carries P 2^6 to within 2^-8 relative from 2^-6 up (e4m3's normal range) and to
//    within 2^-14 absolute below.  p_lo is e5m2 for its range: a P below e4m3's subnormal
//    floor (2^-9 of 2^6, i.e. 2^-15 of the running max) would flush to zero, and behind one
//    dominant key a long tail of such keys is a mass that O would lose; e5m2 keeps every
//    key down to 2^-22 of the running max.  The output is normalised by the sum of
//    p_hi + p_lo (the values the MMAs use), the LSE taken from the fp32 P.
//  * A raw stage is released when BMM1 and BMM2 of its tile have both completed.  Rows of
//    the request's last tile past its end are zeroed in the stage before BMM2 reads them
//    (stale codes there could be NaN, and 0 * NaN is NaN).
//  * BMM1 and BMM2 are issued by two warps, each waiting on its own inputs: issuing blocks
//    while the tensor pipe is busy.
//  * P is double-buffered by tile parity: the softmax of tile j waits only for BMM2 of tile
//    j-2 (which read its buffer).
//  * TMEM: O^T (256 columns) | two S buffers (2 x 64) | split blocks 0-7 (128).  Shared
//    memory: the split's rope block (8 KB) | raw ring (5 x 36 KB) | two P buffers (p_hi |
//    p_lo, 2 x 8 KB) | control.  The bf16 Q tile lands by TMA on ring stages 1-2 and is
//    split from there before their first load; the epilogue stages the bf16 output in
//    stages 0-1.
//  * Softmax and epilogue: eight warps, two per TMEM lane quadrant, so that two warps share
//    each scheduler (one alone left most of its cycles to latency).  They ping-pong: the
//    two warps of a quadrant take alternate tiles, each owning the quadrant's 16 rows; a
//    row's 64 keys are spread over four adjacent threads (16 each), which combine their
//    maxima by shuffles.  A tile's running max is handed to the other warp through a named
//    barrier as soon as it is known, so each warp has two tile periods for its per-tile
//    waits and hand-offs.  P is formed and split in f16x2 arithmetic; lazy rescale; bf16
//    output or split partial for the combine kernel (a programmatic dependent launch).
// Every wait is bounded; on expiry the CTA records a timeout in the status word, drains
// its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda_fp16.h>

#include "mla_internal.h"
#include "sm103a_ptx.cuh"

namespace mla {
namespace {

constexpr int kBlocks = kLatentDim / 64;           // 9 column blocks of 64
constexpr int kStages = 5;                         // raw ring depth
constexpr int kRawBlock = 64 * 64;                 // 64 keys x 64 one-byte codes (64-byte swizzle)
constexpr int kRawTile = kBlocks * kRawBlock;      // 36864
constexpr int kQRBytes = 128 * 64;                 // the split's rope block: 128 stacked rows x 64 codes
constexpr int kF16Block = 64 * 128;                // 64 rows x 64 16-bit columns (128-byte swizzle)
constexpr int kQBf16Bytes = kBlocks * kF16Block;   // 73728
constexpr int kPPart = 64 * 64;                    // p_hi (e4m3) or p_lo (e5m2): 64 rows x 64 keys
constexpr int kPBuf = 2 * kPPart;                  // one P buffer: p_hi | p_lo
constexpr int kOffQR = 0;
constexpr int kOffRaw = kQRBytes;                  // raw ring
constexpr int kOffP = kOffRaw + kStages * kRawTile;  // two P buffers (tile parity)
constexpr int kOffCtrl = kOffP + 2 * kPBuf;
constexpr int kOffQBf16 = kOffRaw + kRawTile;      // the bf16 Q tile lands on ring stages 1-2
constexpr int kOffOStage = kOffRaw;                // [64][512] bf16 output staging (stages 0-1)
static_assert(kQBf16Bytes == 2 * kRawTile, "bf16 Q staging spans ring stages 1-2 exactly");
static_assert(kGroupRows * kValueDim * 2 <= 2 * kRawTile, "output staging fits ring stages 0-1");

constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant, alternating tiles
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kBmm1Warp = kSoftmaxWarps + 1;
constexpr int kBmm2Warp = kSoftmaxWarps + 2;
constexpr int kThreads = 32 * (kBmm2Warp + 1);
constexpr int kQThreadsPerRow = kSoftmaxThreads / kGroupRows;  // 4 adjacent threads per Q row
static_assert(kQThreadsPerRow == 4, "Q split threads per row");

struct Ctrl {
  uint64_t q_full;             // bf16 Q tile landed (TMA)
  uint64_t q_ready;            // stacked q_hi / q_lo written (softmax threads)
  uint64_t raw_full[kStages];  // raw tile landed (TMA)
  uint64_t raw_empty[kStages]; // BMM1 and BMM2 of the tile done (two commits)
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];          // P buffer written (softmax threads), by tile parity
  uint64_t o_done[2];          // BMM2 of the tile done (commit), by tile parity
  uint64_t mma_drain;
  uint64_t mma_drain2;         // the BMM2 warp's MMAs
  uint32_t tmem_base;
  int abort_flag;
  // by tile parity: written before a tile's closing barrier and read after it, while the
  // next tile's writes may already run (it waits only for the BMM2 two tiles back)
  alignas(16) int rescale_flag[2][kSoftmaxWarps];
  alignas(16) float alpha[2][kGroupRows];
  alignas(16) float q_mult[kGroupRows];     // 2^s of each row's Q split
  alignas(16) float row_scale[kGroupRows];
  // ping-pong softmax: the running max each tile hands to the other parity's warps (by
  // sender parity), a stop mark per (sender parity, quadrant), and each parity's final
  // (reference max, row sum, row sum of the split values) per row
  alignas(16) float tok_m[2][kGroupRows];
  int tok_stop[2][4];
  alignas(16) float fin[2][3][kGroupRows];
  alignas(16) float q_unscale[kGroupRows];  // 2^-s of each row's Q split
};
constexpr int kCtrlBytes = 4096;
constexpr int kSmemBytes = kOffCtrl + kCtrlBytes + 1024;  // + control block + alignment slack
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");
static_assert(kSmemBytes <= 232448, "shared memory per block");

constexpr int kAbortTimeout = 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;  // S buffers at columns 256 and 320; O^T chunks at 0,64,128,192
// Column blocks 0-7 of the stacked split (BMM1's A operand): 128 lanes (stacked rows) x 512
// codes, four per 32-bit column, at columns 384-511.  (The rope block, 8, stays in shared
// memory: with two S buffers and O^T there is no room for it.)
constexpr uint32_t kTmemQ = 384;
// The running max (log2 domain) moves once a tile's max exceeds it by more than this, and
// P is formed times 2^kPShift: P 2^kPShift <= 2^(threshold + shift) = 256 < 448 (e4m3 max),
// and e4m3's subnormal floor (2^-9) sits 2^-15 below a P of 1.
constexpr float kRescaleThreshold = 2.0f;
constexpr float kPShift = 6.0f;

// Two floats -> two e4m3 codes (round to nearest even, saturating), `lo` in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e4m3 codes (low byte first) -> their exact values as floats.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(codes));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}

__device__ __forceinline__ uint32_t f16x2_to_e5m2x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(codes));
  return h2;
}

__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint32_t codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e5m2x2 %0, c;\n\t}" : "=r"(h2) : "r"(codes));
  return h2;
}

// P 2^kPShift for this thread's 16 keys of its row, eight pairs: x[2i], x[2i+1] are the
// keys 8i and 8i + 1 past the thread's first key (visible while <= lim; kAll: all of them).
// Each pair is split into two e4m3 hi and two e5m2 lo codes (low byte first) through f16: the f16
// value keeps 11 bits, and hi, the residual (exact in f16: hi is within a factor of 2 of
// the value, or zero) and lo are formed there.  l_sum accumulates the fp32 P 2^kPShift (for
// the LSE), l_use the hi + lo values the MMAs take (for the output's normalisation, so that
// the split's rounding of a dominant key cancels in O / l).
template <bool kAll>
__device__ __forceinline__ void p_split16(const float (&x)[16], int lim, float scale_log2, float off, float& l_sum,
                                          float& l_use, uint32_t (&phi)[8], uint32_t (&plo)[8]) {
  float ls = 0.f, lu = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float p0 = (kAll || 8 * i <= lim) ? ex2_approx(fmaf(x[2 * i], scale_log2, off)) : 0.f;
    const float p1 = (kAll || 8 * i + 1 <= lim) ? ex2_approx(fmaf(x[2 * i + 1], scale_log2, off)) : 0.f;
    ls += p0 + p1;
    const uint32_t ph = pack_f16x2(p0, p1);
    phi[i] = f16x2_to_e4m3x2(ph);
    const uint32_t hb = e4m3x2_to_f16x2(phi[i]);
    uint32_t d, sum;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(ph), "r"(hb));
    plo[i] = f16x2_to_e5m2x2(d);
    const uint32_t lb = e5m2x2_to_f16x2(plo[i]);
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(sum) : "r"(hb), "r"(lb));
    const float2 uf = __half22float2(*reinterpret_cast<const __half2*>(&sum));
    lu += uf.x + uf.y;
  }
  l_sum += ls;
  l_use += lu;
}

// kMayIdle: q_len * heads is not a multiple of 64, so a row group may hold 48 rows or fewer
// and a softmax warp may own no row; such warps then skip their S reads and P writes.  (A
// compile-time choice: the check alone measured 1.2 % slower on full 64-row groups.)
template <bool kMayIdle>
__global__ void __launch_bounds__(kThreads, 1)
decode_partial_e4m3_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                           const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kOffCtrl);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = blockIdx.x;
  // grid (row groups, requests, splits) for a multi-wave plan: the hardware starts CTAs in
  // linear block order, so every request's first split is dispatched before any second
  // split; (row groups, splits, requests) otherwise
  const int b = p.split_major ? blockIdx.y : blockIdx.z;
  const int split = p.split_major ? blockIdx.z : blockIdx.y;

  // Set-up that reads no input of this call (overlaps the previous kernel's tail: this is a
  // programmatic dependent launch; griddepcontrol.wait below orders every input read).
  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    mbar_init(&ctrl->q_ready, kSoftmaxWarps);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctrl->raw_full[s], 1);
      mbar_init(&ctrl->raw_empty[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->s_full[s], 1);
      mbar_init(&ctrl->s_free[s], kSoftmaxWarps / 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->p_full[s], kSoftmaxWarps / 2);
      mbar_init(&ctrl->o_done[s], 1);
    }
    mbar_init(&ctrl->mma_drain, 1);
    mbar_init(&ctrl->mma_drain2, 1);
    ctrl->abort_flag = 0;
    for (int w = 0; w < kSoftmaxWarps; ++w) ctrl->rescale_flag[0][w] = ctrl->rescale_flag[1][w] = 0;
    for (int q = 0; q < 4; ++q) ctrl->tok_stop[0][q] = ctrl->tok_stop[1][q] = 0;
    fence_mbarrier_init();
  }
  if (warp == kBmm1Warp) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
  }
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
    if (warp == kBmm1Warp) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int kv_end = min(L, kv_start + p.chunk);
  const int ntiles = (kv_end - kv_start + kTileKeys - 1) / kTileKeys;
  const int nsplit_b = (L + p.chunk - 1) / p.chunk;
  const int row0 = group * kGroupRows;
  const int nrows = min(kGroupRows, p.R - row0);
  const int nq = (nrows + 15) & ~15;  // BMM2 N (multiple of 16)
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer: Q, then raw tiles
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
    int last_issued[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last_issued[s] = -1;
    bool ok = true;
    bool q_waited = false;
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctrl->q_full, kQBf16Bytes);
      tma_load_3d(smem + kOffQBf16, &tm_q, &ctrl->q_full, 0, b * p.R + row0, 0, policy_evict_last());
    }
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
      if (s >= 1 && !q_waited) {  // stages 1-2 hold the bf16 Q tile until it has been split
        bool w = true;
        if (lane == 0) w = mbar_wait(&ctrl->q_ready, 0, abort_flag);
        ok = __shfl_sync(0xffffffffu, w, 0);
        q_waited = true;
        if (!ok) break;
      }
      if (j >= kStages) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&ctrl->raw_empty[s], ((j / kStages) - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, w, 0);
        if (!ok) break;
      }
      if (lane == 0) {
        uint8_t* stage = smem + kOffRaw + s * kRawTile;
        mbar_arrive_expect_tx(&ctrl->raw_full[s], static_cast<uint32_t>(npg * box_rows * 64 * kBlocks));
        if (P >= kTileKeys) {  // one 3-D box: 64 rows x all 9 column blocks
          tma_load_3d(stage, &tm_kv, &ctrl->raw_full[s], 0, pids[0] * P + ((P > kTileKeys) ? (k0 % P) : 0), 0,
                      pol_kv);
        } else {  // one 2-D box per (page, column block)
          for (int pp = 0; pp < npg; ++pp)
            for (int c = 0; c < kBlocks; ++c)
              tma_load_2d(stage + c * kRawBlock + pp * box_rows * 64, &tm_kv, &ctrl->raw_full[s], c * 64,
                          pids[pp] * P, pol_kv);
        }
      }
      last_issued[s] = j;
      __syncwarp();
    }
    if (bad_pid && lane == 0) atomicOr(p.status, kStatusDeviceArg);
    if (!ok && lane == 0) {
      drain_wait(&ctrl->q_full, 0);
      for (int s = 0; s < kStages; ++s)
        if (last_issued[s] >= 0) drain_wait(&ctrl->raw_full[s], (last_issued[s] / kStages) & 1);
    }
  } else if (warp == kBmm1Warp) {
    // ------------------------------------------------------------------ BMM1 issuer (whole warp,
    // uniform control flow; one elected thread issues the MMAs and their commits)
    const uint32_t idesc1 = make_idesc_e4m3(128, 64);
    const uint64_t qr_desc = make_smem_desc_sw64(smem_u32(smem + kOffQR));
    bool ok = mbar_wait(&ctrl->q_ready, 0, abort_flag);
    // BMM1(j) as soon as raw tile j has landed and its S buffer is free
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kStages, sb = j & 1;
      if (ok) ok = mbar_wait(&ctrl->raw_full[s], (j / kStages) & 1, abort_flag);
      if (ok && j >= 2) ok = mbar_wait(&ctrl->s_free[sb], ((j - 2) >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint64_t k_desc = make_smem_desc_sw64(smem_u32(smem + kOffRaw + s * kRawTile));
      const uint32_t d = tmem + kTmemS + sb * 64;
      if (elect_one()) {
        // S_hi / S_lo (stacked rows) = [q_hi; q_lo] . k: 9 blocks x 2 K-steps of 32 codes,
        // A from TMEM for blocks 0-7 (8 columns per K-step), from shared memory for block 8
#pragma unroll
        for (int c = 0; c < kBlocks - 1; ++c) {
#pragma unroll
          for (int k = 0; k < 2; ++k)
            umma_f8_ts(d, tmem + kTmemQ + c * 16 + k * 8, k_desc + static_cast<uint64_t>((c * kRawBlock + k * 32) >> 4),
                       idesc1, (c | k) != 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
          umma_f8(d, qr_desc + static_cast<uint64_t>((k * 32) >> 4),
                  k_desc + static_cast<uint64_t>(((kBlocks - 1) * kRawBlock + k * 32) >> 4), idesc1, 1u);
        umma_commit(&ctrl->s_full[sb]);
        umma_commit(&ctrl->raw_empty[s]);
      }
      __syncwarp();
    }
    // every MMA this warp issued completes before TMEM is released
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain);
      drain_wait(&ctrl->mma_drain, 0);
    }
    __syncwarp();
  } else if (warp == kBmm2Warp) {
    // ------------------------------------------------------------------ BMM2 issuer
    // O^T[value col, row] += V^T . P^T: A = V^T, MN-major straight from the raw stage (two
    // 64-column blocks of 4 KB per 128-column chunk, 8-key groups 512 bytes apart); B = p_hi
    // (e4m3) then p_lo (e5m2), K-major rows of 64 keys.
    const uint32_t idesc2_hi = make_idesc_f8(128, nq, kF8E4M3, kF8E4M3, true, false);
    const uint32_t idesc2_lo = make_idesc_f8(128, nq, kF8E4M3, kF8E5M2, true, false);
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kStages, pb = j & 1;
      if (ok) ok = mbar_wait(&ctrl->p_full[pb], (j >> 1) & 1, abort_flag);
      if (ok) ok = mbar_wait(&ctrl->raw_full[s], (j / kStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint64_t v_desc = make_smem_desc_sw64(smem_u32(smem + kOffRaw + s * kRawTile), kRawBlock, 512);
      const uint64_t phi_desc = make_smem_desc_sw64(smem_u32(smem + kOffP + pb * kPBuf));
      const uint64_t plo_desc = make_smem_desc_sw64(smem_u32(smem + kOffP + pb * kPBuf + kPPart));
      if (elect_one()) {
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t voff = static_cast<uint64_t>((2 * qc * kRawBlock + kk * 2048) >> 4);
            const uint64_t poff = static_cast<uint64_t>((kk * 32) >> 4);
            umma_f8(tmem + qc * 64, v_desc + voff, phi_desc + poff, idesc2_hi, (j > 0 || kk > 0) ? 1u : 0u);
            umma_f8(tmem + qc * 64, v_desc + voff, plo_desc + poff, idesc2_lo, 1u);
          }
        }
        umma_commit(&ctrl->o_done[pb]);
        umma_commit(&ctrl->raw_empty[s]);
      }
      __syncwarp();
    }
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain2);
      drain_wait(&ctrl->mma_drain2, 0);
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-7)
    // Q split, in two passes over the bf16 tile (ring stages 1-2).  First, row r's largest
    // |q| (threads 4r .. 4r+3, each over bf16 chunks 2h, 2h+1 of every 64-column block) sets
    // its power-of-two scale, and the same threads write the rope block's q_hi / q_lo
    // (e4m3 chunk h) to shared memory: q_hi of row r as stacked row 16 (r / 8) + r % 8,
    // q_lo 8 rows further.  Then each thread writes one stacked row's codes of four column
    // blocks into TMEM (its lane quadrant's lane = the stacked row; blocks 4kh .. 4kh+3):
    // lane i holds row 16 quad + 8 (i / 16) + i % 8, its q_hi for i % 16 < 8, else its q_lo.
    bool failed = bar_or(1, kSoftmaxThreads, !mbar_wait(&ctrl->q_full, 0, abort_flag));
    const uint32_t qb0 = smem_u32(smem + kOffQBf16);
    if (!failed) {
      const int r = threadIdx.x >> 2, h = threadIdx.x & 3;
      const uint32_t qb = qb0 + r * 128;
      float mx = 0.f;
      for (int c = 0; c < kBlocks; ++c) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t w[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(qb + c * kF16Block + (((2 * h + jj) ^ (r & 7)) << 4)));
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      int sh = 0;  // the row's power-of-two scale: its largest |q| lands in [128, 256)
      if (mx > 0.f) sh = min(126, max(-120, 7 - (static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127)));
      const float mult = __uint_as_float(static_cast<uint32_t>(sh + 127) << 23);
      if (h == 0) {
        ctrl->q_unscale[r] = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
        ctrl->q_mult[r] = mult;
      }
      const int m_hi = 16 * (r >> 3) + (r & 7);  // stacked row of q_hi (q_lo: m_hi + 8)
      const uint32_t qhi = smem_u32(smem + kOffQR) + m_hi * 64;
      const uint32_t qlo = qhi + 8 * 64;
      const uint32_t e_off = (h ^ ((m_hi >> 1) & 3)) << 4;  // chunk h under both rows' 64-byte swizzle
      constexpr int c = kBlocks - 1;  // the rope block
      uint32_t w[8];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "r"(qb + c * kF16Block + (((2 * h) ^ (r & 7)) << 4)));
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                   : "r"(qb + c * kF16Block + (((2 * h + 1) ^ (r & 7)) << 4)));
      uint32_t hi4[4], lo4[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        // four values: w[i] = (x0, x1), w[i+1] = (x2, x3), bf16 pairs low half first
        const float x0 = __uint_as_float(w[i] << 16) * mult, x1 = __uint_as_float(w[i] & 0xFFFF0000u) * mult;
        const float x2 = __uint_as_float(w[i + 1] << 16) * mult;
        const float x3 = __uint_as_float(w[i + 1] & 0xFFFF0000u) * mult;
        const uint32_t h01 = f32x2_to_e4m3x2(x0, x1), h23 = f32x2_to_e4m3x2(x2, x3);
        const float2 v01 = e4m3x2_to_f32x2(h01), v23 = e4m3x2_to_f32x2(h23);
        const uint32_t l01 = f32x2_to_e4m3x2(x0 - v01.x, x1 - v01.y);
        const uint32_t l23 = f32x2_to_e4m3x2(x2 - v23.x, x3 - v23.y);
        hi4[i >> 1] = h01 | (h23 << 16);
        lo4[i >> 1] = l01 | (l23 << 16);
      }
      st_shared_v4(qhi + e_off, hi4[0], hi4[1], hi4[2], hi4[3]);
      st_shared_v4(qlo + e_off, lo4[0], lo4[1], lo4[2], lo4[3]);
      fence_proxy_async_smem();
    }
    named_bar_sync(1, kSoftmaxThreads);  // the rows' scales are written
    if (!failed) {
      const int quad_q = warp & 3, kh_q = warp >> 2;
      const bool lo_part = ((lane >> 3) & 1) != 0;
      const int r = quad_q * 16 + 8 * (lane >> 4) + (lane & 7);
      const float mult = ctrl->q_mult[r];
      const uint32_t qb = qb0 + r * 128;
      const uint32_t lane_q = static_cast<uint32_t>(quad_q * 32) << 16;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        const int c = 4 * kh_q + cb;
        uint32_t codes[16];  // 64 codes of block c, four per word, column order
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {  // bf16 chunk ch = columns 8ch .. 8ch+7
          uint32_t w[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(qb + c * kF16Block + ((ch ^ (r & 7)) << 4)));
#pragma unroll
          for (int i = 0; i < 4; i += 2) {
            const float x0 = __uint_as_float(w[i] << 16) * mult, x1 = __uint_as_float(w[i] & 0xFFFF0000u) * mult;
            const float x2 = __uint_as_float(w[i + 1] << 16) * mult;
            const float x3 = __uint_as_float(w[i + 1] & 0xFFFF0000u) * mult;
            uint32_t c01 = f32x2_to_e4m3x2(x0, x1), c23 = f32x2_to_e4m3x2(x2, x3);
            if (lo_part) {
              const float2 v01 = e4m3x2_to_f32x2(c01), v23 = e4m3x2_to_f32x2(c23);
              c01 = f32x2_to_e4m3x2(x0 - v01.x, x1 - v01.y);
              c23 = f32x2_to_e4m3x2(x2 - v23.x, x3 - v23.y);
            }
            codes[2 * ch + (i >> 1)] = c01 | (c23 << 16);
          }
        }
        tmem_st16(tmem + lane_q + kTmemQ + c * 16, codes);
      }
      tmem_st_wait();
    }
    // every softmax thread has read its part of the bf16 tile (ring stages 1-2) and written
    // its part of the split
    tc_fence_before();
    named_bar_sync(1, kSoftmaxThreads);
    __syncwarp();
    if (!failed && lane == 0) mbar_arrive(&ctrl->q_ready);

    // BMM1 (M = 128) puts row r's hi / lo partial scores in TMEM lanes 16 (r / 8) + r % 8 and
    // 8 further.  Warp w takes lane quadrant quad = w % 4, i.e. rows 16 quad .. +15, and the
    // tiles of parity par = w / 4 (ping-pong: the two warps of a quadrant alternate tiles).
    // Two 16x256b loads (lanes 32 quad .. +15 and 32 quad + 16 .. +31) give thread 4g + c
    // rows 16 quad + g and 16 quad + 8 + g, each row's hi and lo partial in the same thread,
    // keys 8i + 2c and 8i + 2c + 1 (i < 8) of its tiles; a row's four threads combine their
    // maxima by two shuffles.  A tile's running max depends on the previous tile's, which the
    // other parity's warp of the quadrant computed: it is handed over through shared memory
    // and a named barrier (bar.arrive by the sender, bar.sync by the receiver) as soon as it
    // is known, before either warp forms its P.  Each warp keeps its own row sums, relative
    // to the reference max of its last tile; the two are combined after the loop.
    const int quad = warp & 3, par = warp >> 2;
    const int kh = par;  // (the epilogue's rows 32 kh .. +31)
    const int cq = lane & 3;
    const int rr0 = quad * 16 + (lane >> 2);  // rows rr0 and rr0 + 8
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const float v_scale = p.v_scale;
    int lim_abs[2];
    bool row_active[2];
    float scale_log2[2];
    // S holds (q 2^s) . k_code: the row's 2^-s and kv_scale (in p.scale_log2) return here;
    // P carries 2^kPShift, which cancels in O / l and returns in the LSE.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rr0 + 8 * h;
      row_active[h] = r < nrows;
      lim_abs[h] = L - p.T + (row0 + r) / p.H;  // last visible key of the row
      scale_log2[h] = failed ? 0.f : p.scale_log2 * ctrl->q_unscale[r];
    }
    float m_w[2] = {-INFINITY, -INFINITY};  // reference max of this warp's last tile
    float l_sum[2] = {0.f, 0.f}, l_use[2] = {0.f, 0.f};
    // key pair i of this thread in a P buffer: row r (64 bytes), 16-byte chunk i / 2 under
    // the 64-byte swizzle, bytes 8 (i % 2) + 2c, +1
    const uint32_t p_base = smem_u32(smem + kOffP) + 2 * cq;
    const int bar_par = 2 + par;                   // the four warps of this parity (128 threads)
    const int tok_in = 4 + 2 * quad + (par ^ 1);   // handed over by the other parity
    const int tok_out = 4 + 2 * quad + par;        // handed over to it
    // A parity whose closing barrier reports a failure drains: at its next tile it takes the
    // other parity's hand-over and hands one back marked stop, then leaves; a warp that
    // receives a stop mark leaves without handing over.  Every hand-over thus has a receiver.
    bool draining = false;
    // A warp whose 16 rows are all past the group's rows reads no S and writes no P (BMM2
    // reads only the first nq rows of P, and nq <= 16 quad then); it keeps every barrier
    // arrival and the hand-over, and its rows' alpha stays 1.
    const bool idle = kMayIdle && __all_sync(0xffffffffu, !row_active[0] && !row_active[1]);

    for (int j = par; !failed && j < ntiles; j += 2) {
      const int pb = j & 1;  // S buffer, P buffer and flags of this tile (= par)
      const int s = j % kStages;
      const int k0 = kv_start + j * kTileKeys;
      bool fail = draining;
      float x[2][16];
      int lim[2] = {-1, -1};
      float mx[2] = {-INFINITY, -INFINITY};
      if (!fail) fail = __any_sync(0xffffffffu, !mbar_wait(&ctrl->s_full[pb], (j >> 1) & 1, abort_flag));
      if (!fail && idle) {
        tc_fence_after();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->s_free[pb]);
      } else if (!fail) {
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld16x256b_x8(tmem + lane_base + kTmemS + pb * 64, v0);
        tmem_ld16x256b_x8(tmem + lane_base + (16u << 16) + kTmemS + pb * 64, v1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->s_free[pb]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[0][2 * i] = __uint_as_float(v0[4 * i]) + __uint_as_float(v0[4 * i + 2]);
          x[0][2 * i + 1] = __uint_as_float(v0[4 * i + 1]) + __uint_as_float(v0[4 * i + 3]);
          x[1][2 * i] = __uint_as_float(v1[4 * i]) + __uint_as_float(v1[4 * i + 2]);
          x[1][2 * i + 1] = __uint_as_float(v1[4 * i + 1]) + __uint_as_float(v1[4 * i + 3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // the row's last visible key in this tile, counted from this thread's first key 2c
          lim[h] = row_active[h] ? (min(kv_end - 1, lim_abs[h]) - k0 - 2 * cq) : -1;
          if (lim[h] >= 57) {
#pragma unroll
            for (int k = 0; k < 16; ++k) mx[h] = fmaxf(mx[h], x[h][k]);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (8 * i <= lim[h]) mx[h] = fmaxf(mx[h], x[h][2 * i]);
              if (8 * i + 1 <= lim[h]) mx[h] = fmaxf(mx[h], x[h][2 * i + 1]);
            }
          }
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        }
      }
      // the previous tile's reference max, handed over by the other parity
      float mprev[2] = {-INFINITY, -INFINITY};
      if (j >= 1) {
        named_bar_sync(tok_in, 64);
        if (ctrl->tok_stop[par ^ 1][quad] != 0) {  // the other parity has left
          failed = true;
          break;
        }
        mprev[0] = ctrl->tok_m[par ^ 1][rr0];
        mprev[1] = ctrl->tok_m[par ^ 1][rr0 + 8];
      }
      float alpha[2] = {1.f, 1.f}, m_new[2];
      bool need_rescale = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // scale > 0: max commutes with the scaling; -inf stays -inf
        const float mt = mx[h] * scale_log2[h];
        m_new[h] = mprev[h];
        if (fail) {
        } else if (mprev[h] == -INFINITY) {
          m_new[h] = mt;  // first contributing tile: nothing accumulated yet
        } else if (mt > mprev[h] + kRescaleThreshold) {
          alpha[h] = ex2_approx(mprev[h] - mt);
          need_rescale = true;
          m_new[h] = mt;
        }
      }
      if (j + 1 < ntiles) {  // hand this tile's reference max to the other parity
        if (cq == 0) {
          ctrl->tok_m[par][rr0] = m_new[0];
          ctrl->tok_m[par][rr0 + 8] = m_new[1];
        }
        if (lane == 0) ctrl->tok_stop[par][quad] = draining ? 1 : 0;
        asm volatile("bar.arrive %0, %1;" ::"r"(tok_out), "r"(64) : "memory");
      }
      if (draining) {
        failed = true;
        break;
      }
      float off[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // this warp's sums move from its previous reference to this tile's
        if (!fail && m_w[h] != m_new[h] && m_w[h] != -INFINITY) {
          const float f = ex2_approx(m_w[h] - m_new[h]);
          l_sum[h] *= f;
          l_use[h] *= f;
        }
        if (!fail) m_w[h] = m_new[h];
        off[h] = (m_new[h] == -INFINITY) ? 0.f : (kPShift - m_new[h]);
      }
      if (!fail && j >= 2) {  // the P buffer is free once BMM2 of tile j-2 has completed
        fail = !mbar_wait(&ctrl->o_done[pb], ((j - 2) >> 1) & 1, abort_flag);
        fail = __any_sync(0xffffffffu, fail);
      }
      if (!fail) {
#pragma unroll
        for (int h = 0; h < 2 && !idle; ++h) {
          const int r = rr0 + 8 * h;
          uint32_t phi[8], plo[8];
          if (lim[h] >= 57)
            p_split16<true>(x[h], lim[h], scale_log2[h], off[h], l_sum[h], l_use[h], phi, plo);
          else
            p_split16<false>(x[h], lim[h], scale_log2[h], off[h], l_sum[h], l_use[h], phi, plo);
          const uint32_t p_row = p_base + pb * kPBuf + r * 64;
          const uint32_t p_sw = (r >> 1) & 3;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t a = p_row + ((((i >> 1) ^ p_sw) << 4) | ((i & 1) << 3));
            st_shared_u16(a, phi[i]);
            st_shared_u16(a + kPPart, plo[i]);
          }
          if (cq == 0) ctrl->alpha[pb][r] = alpha[h];
        }
        if (idle && cq == 0) ctrl->alpha[pb][rr0] = ctrl->alpha[pb][rr0 + 8] = 1.f;
        const bool any = __any_sync(0xffffffffu, need_rescale);
        if (lane == 0) ctrl->rescale_flag[pb][quad] = any ? 1 : 0;
        // the request's last tile: rows past its end are zeroed in the V blocks (BMM1 of this
        // tile has completed; BMM2 reads them only after p_full)
        const int valid_rows = L - k0;
        if (valid_rows < kTileKeys) {
          const uint32_t stage = smem_u32(smem + kOffRaw + s * kRawTile);
          const int n16 = (kTileKeys - valid_rows) * 4 * (kValueDim / 64);  // 16-byte pieces
          for (int i = quad * 32 + lane; i < n16; i += kSoftmaxThreads / 2) {
            const int row = valid_rows + (i >> 5), blk = (i >> 2) & 7, piece = i & 3;
            st_shared_v4(stage + blk * kRawBlock + row * 64 + piece * 16, 0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();
      if (bar_or(bar_par, kSoftmaxThreads / 2, fail || (*abort_flag != 0))) {
        draining = true;  // leave at this parity's next tile (or now, if it has none)
        continue;
      }
      const int4 f0 = *reinterpret_cast<const int4*>(&ctrl->rescale_flag[pb][0]);
      if (f0.x | f0.y | f0.z | f0.w) {
        // O^T[dim, row] *= alpha[row] for all 512 value columns, once BMM2 of tile j-1 has
        // completed; this thread owns TMEM lane (32 quad + lane) of each 128-column chunk,
        // all 64 rows.  (A wait that gives up raises the abort flag, which the next closing
        // barrier reports.)
        if (j >= 1) mbar_wait(&ctrl->o_done[pb ^ 1], ((j - 1) >> 1) & 1, abort_flag);
        tc_fence_after();
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float al[32];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 f = *reinterpret_cast<const float4*>(&ctrl->alpha[pb][hh * 32 + i]);
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
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->p_full[pb]);
    }
    if (draining) failed = true;

    if (!failed) failed = !mbar_wait(&ctrl->o_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort_flag);
    // this warp's partial row sums (its four threads per row), relative to m_w, to shared
    // memory; the two parities' parts are combined below
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_sum[h] += __shfl_xor_sync(0xffffffffu, l_sum[h], 1);
      l_sum[h] += __shfl_xor_sync(0xffffffffu, l_sum[h], 2);
      l_use[h] += __shfl_xor_sync(0xffffffffu, l_use[h], 1);
      l_use[h] += __shfl_xor_sync(0xffffffffu, l_use[h], 2);
      if (cq == 0) {
        ctrl->fin[par][0][rr0 + 8 * h] = m_w[h];
        ctrl->fin[par][1][rr0 + 8 * h] = l_sum[h];
        ctrl->fin[par][2][rr0 + 8 * h] = l_use[h];
      }
    }
    if (bar_or(1, kSoftmaxThreads, failed || (*abort_flag != 0))) {
      failed = true;
    } else {
      tc_fence_after();
      const bool final_out = (nsplit_b == 1);
      if (par == 0 && cq == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = rr0 + 8 * h;
          // O is relative to the last tile's max, the larger of the two parities' last
          const float ma = ctrl->fin[0][0][r], mb = ctrl->fin[1][0][r];
          const float m = fmaxf(ma, mb);
          const float fa = (ma == -INFINITY) ? 0.f : ex2_approx(ma - m);
          const float fb = (mb == -INFINITY) ? 0.f : ex2_approx(mb - m);
          const float ls = ctrl->fin[0][1][r] * fa + ctrl->fin[1][1][r] * fb;
          const float lu = ctrl->fin[0][2][r] * fa + ctrl->fin[1][2][r] * fb;
          const float lse2 = (ls > 0.f) ? (m + __log2f(ls) - kPShift) : -INFINITY;
          const float lse_nat = lse2 * 0.69314718055994530942f;
          ctrl->row_scale[r] = (lu > 0.f) ? (v_scale / lu) : 0.f;
          if (row_active[h]) {
            const int64_t grow = static_cast<int64_t>(b) * p.R + row0 + r;
            if (final_out)
              p.lse[grow] = lse_nat;
            else
              p.ws_lse[(static_cast<int64_t>(b) * p.max_splits + split) * p.R + row0 + r] = lse_nat;
          }
        }
      }
      named_bar_sync(1, kSoftmaxThreads);
      // Normalised O (bf16) is transposed through ring stages 0-1 (free once the last BMM2
      // has completed) so that global stores are whole 16-byte row chunks.  This thread:
      // value column 32 quad + lane of each 128-column chunk, rows 32kh .. 32kh+31, whose
      // scales stay in registers.
      const uint32_t stage_s = smem_u32(smem + kOffOStage);  // [64][512] bf16
      float rs[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 f = *reinterpret_cast<const float4*>(&ctrl->row_scale[kh * 32 + i]);
        rs[i] = f.x;
        rs[i + 1] = f.y;
        rs[i + 2] = f.z;
        rs[i + 3] = f.w;
      }
#pragma unroll 1
      for (int qc = 0; qc < 4; ++qc) {
        const int dim = qc * 128 + quad * 32 + lane;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + qc * 64 + kh * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(v[i]) * rs[i]);
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(stage_s + ((kh * 32 + i) * kValueDim + dim) * 2),
                       "h"(*reinterpret_cast<const uint16_t*>(&o)));
        }
      }
      const __nv_bfloat16* stage_h = reinterpret_cast<const __nv_bfloat16*>(smem + kOffOStage);
      named_bar_sync(1, kSoftmaxThreads);
      constexpr int kChunksPerRow = kValueDim * 2 / 16;
      __nv_bfloat16* dst = final_out
                               ? p.out + (static_cast<int64_t>(b) * p.R + row0) * kValueDim
                               : p.ws_o + ((static_cast<int64_t>(b) * p.max_splits + split) * p.R + row0) * kValueDim;
      for (int c = threadIdx.x; c < nrows * kChunksPerRow; c += kSoftmaxThreads) {
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
  if (warp == kBmm1Warp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_decode_partial_e4m3(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                       int head_groups, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(decode_partial_e4m3_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_partial_e4m3_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.split_major ? dim3(head_groups, p.B, p.max_splits) : dim3(head_groups, p.max_splits, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // a group of 48 rows or fewer exists when R is not a multiple of 64
  return (p.R % kGroupRows != 0) ? cudaLaunchKernelEx(&cfg, decode_partial_e4m3_kernel<true>, tm_q, tm_kv, p)
                                 : cudaLaunchKernelEx(&cfg, decode_partial_e4m3_kernel<false>, tm_q, tm_kv, p);
}

}  // namespace mla
