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
// Design on sm_103a (one CTA per (64-row group, split, request); one CTA per SM; 480
// threads: softmax warps 0-3, producer warp 4, BMM1 warp 5, decode warps 6-13, BMM2 warp 14):
//  * The raw e4m3 tile (64 keys x 576 codes, 36 KB) arrives by TMA (64-byte swizzle) in a
//    2-stage ring, its rows prefetched into L2 a few tiles earlier, and is the B operand of
//    BMM1 as it is: BMM1 runs on 8-bit operands
//    (kind::f8f6f4).  Q keeps its bf16 value: each query row, scaled by a power of two 2^s
//    that brings its largest element into [128, 256), is split into q_hi = e4m3(q 2^s) and
//    q_lo = e4m3(q 2^s - q_hi), an 8-bit significand in two 4-bit halves.  This is exact
//    for every element within 2^9 of the row's largest |q|; smaller elements fall under
//    e4m3's subnormal floor (2^-9 at that scale) and carry an absolute error of at most
//    2^-17 of the row's largest |q|.  S = (q_hi + q_lo) . k_code takes two passes of MMAs
//    into one fp32 accumulator, and 2^-s returns in the softmax.
//  * Only V (the first 512 columns) is decoded to f16 (exactly: codes times 2^-8), from the
//    raw stage in shared memory into one f16 V stage, by the decode warps, while the
//    tensor core runs BMM1 of the next tile on its raw stage.  The decode warps take a
//    tile's raw V bytes into registers as soon as it lands and release the raw stage at
//    once, so its refill does not wait for the V stage.  BMM2 (O^T += V^T . P^T, M = 128
//    value columns, N = rows, K = 64 keys) reads that stage with f16 P.
//  * BMM1 and BMM2 are issued by two warps, each waiting on its own inputs: issuing blocks
//    while the tensor pipe is busy, and one warp issuing both held each BMM2 behind the
//    next BMM1's issue loop.
//  * Shared memory: q_hi | q_lo (2 x 36 KB) | raw ring (2 x 36 KB) | f16 V stage (64 KB) |
//    P (8 KB).  The bf16 Q tile lands by TMA on the V stage and P (72 KB) and is split
//    from there before the first V decode.
//  * Softmax and epilogue as in the bf16/int8 kernel: M = 64 rows in TMEM lanes
//    32*(r/16) + r%16, each row split over two lanes, lazy rescale, f16 P, bf16 output or
//    split partial for the combine kernel (a programmatic dependent launch).
// Every wait is bounded; on expiry the CTA records a timeout in the status word, drains
// its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda_fp16.h>

#include "kv8_decode.cuh"
#include "mla_internal.h"
#include "sm103a_ptx.cuh"

namespace mla {
namespace {

constexpr int kBlocks = kLatentDim / 64;           // 9 column blocks of 64
constexpr int kRawBlock = 64 * 64;                 // 64 keys x 64 one-byte codes (64-byte swizzle)
constexpr int kRawTile = kBlocks * kRawBlock;      // 36864
constexpr int kQPart = kBlocks * kRawBlock;        // 64 rows x 576 e4m3 codes
constexpr int kF16Block = 64 * 128;                // 64 rows x 64 16-bit columns (128-byte swizzle)
constexpr int kVBytes = (kValueDim / 64) * kF16Block;  // 65536
constexpr int kQBf16Bytes = kBlocks * kF16Block;   // 73728
constexpr int kOffQ8 = 0;                          // q_hi, then q_lo
constexpr int kOffRaw = 2 * kQPart;                // raw ring
constexpr int kOffV = kOffRaw + 2 * kRawTile;      // f16 V stage
constexpr int kOffP = kOffV + kVBytes;             // P [64 rows][64 keys] f16
constexpr int kOffQBf16 = kOffV;                   // the bf16 Q tile lands on V and P
constexpr int kOffCtrl = kOffP + kF16Block;
static_assert(kOffQBf16 + kQBf16Bytes == kOffCtrl, "bf16 Q staging spans V and P exactly");

constexpr int kDecodeWarps = 8;
constexpr int kDecodeWarp0 = 6;
constexpr int kDecodeThreads = 32 * kDecodeWarps;
constexpr int kBmm2Warp = kDecodeWarp0 + kDecodeWarps;  // issues BMM2 (warp 5 issues BMM1)
constexpr int kThreads = 32 * (kBmm2Warp + 1);
constexpr int kSoftmaxThreads = 128;
constexpr int kQThreadsPerRow = kDecodeThreads / kGroupRows;  // 1, 2 or 4 adjacent lanes per Q row
static_assert(kQThreadsPerRow == 1 || kQThreadsPerRow == 2 || kQThreadsPerRow == 4, "Q split threads per row");

struct Ctrl {
  uint64_t q_full;             // bf16 Q tile landed (TMA)
  uint64_t q_ready;            // q_hi / q_lo written (decode threads)
  uint64_t raw_full[2];        // raw tile landed (TMA)
  uint64_t raw_empty[2];       // BMM1 of the tile done (commit) and its V decoded (decode threads)
  uint64_t v_full;             // f16 V stage written (decode threads)
  uint64_t v_empty;            // BMM2 of the V stage's tile done (commit)
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t mma_drain;
  uint64_t mma_drain2;         // the BMM2 warp's MMAs
  uint32_t tmem_base;
  int abort_flag;
  int rescale_flag[4];
  alignas(16) float alpha[kGroupRows];
  alignas(16) float row_scale[kGroupRows];
  alignas(16) float q_unscale[kGroupRows];  // 2^-s of each row's Q split
};
constexpr int kSmemBytes = kOffCtrl + 1024 + 1024;  // + control block + alignment slack
static_assert(sizeof(Ctrl) <= 1024, "control block");

constexpr int kPrefetchAhead = 3;  // raw tiles are prefetched into L2 this many tiles before their TMA load
constexpr int kAbortTimeout = 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;  // S buffers at columns 256 and 320; O^T chunks at 0,64,128,192
constexpr float kRescaleThreshold = 8.0f;

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

__global__ void __launch_bounds__(kThreads, 1)
decode_partial_e4m3_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                           const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kOffCtrl);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = blockIdx.x;
  const int split = blockIdx.y;
  const int b = blockIdx.z;

  // Set-up that reads no input of this call (overlaps the previous kernel's tail: this is a
  // programmatic dependent launch; griddepcontrol.wait below orders every input read).
  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    mbar_init(&ctrl->q_ready, kDecodeThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->raw_full[s], 1);
      mbar_init(&ctrl->raw_empty[s], 1 + kDecodeThreads);
      mbar_init(&ctrl->s_full[s], 1);
      mbar_init(&ctrl->s_free[s], kSoftmaxThreads);
    }
    mbar_init(&ctrl->v_full, kDecodeThreads);
    mbar_init(&ctrl->v_empty, 1);
    mbar_init(&ctrl->p_full, kSoftmaxThreads);
    mbar_init(&ctrl->o_done, 1);
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
  if (warp == 4 && lane == 0) {
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
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int kv_end = min(L, kv_start + p.chunk);
  const int ntiles = (kv_end - kv_start + kTileKeys - 1) / kTileKeys;
  const int nsplit_b = (L + p.chunk - 1) / p.chunk;
  const int row0 = group * kGroupRows;
  const int nrows = min(kGroupRows, p.R - row0);
  const int nq = (nrows + 15) & ~15;  // BMM2 N (multiple of 16)
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == 4) {
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
    int last_issued[2] = {-1, -1};
    bool ok = true;
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctrl->q_full, kQBf16Bytes);
      tma_load_3d(smem + kOffQBf16, &tm_q, &ctrl->q_full, 0, b * p.R + row0, 0, policy_evict_last());
    }
    // L2 prefetch of tile jt's rows (lane l < pages per tile: the rows of its page in the
    // tile), so that each TMA load, issued only once its ring stage frees up, finds them in L2.
    auto prefetch_tile = [&](int jt) {
      const int k = kv_start + jt * kTileKeys + lane * box_rows;
      if (jt >= ntiles || lane >= sub || k >= kv_end) return;
      const unsigned pid = static_cast<unsigned>(__ldg(pt + k / P));
      if (pid >= n_pages) return;  // (reported when its TMA load is issued)
      const int rows = min(box_rows, kv_end - k);
      prefetch_l2_bulk(p.kv_pool + (static_cast<int64_t>(pid) * P + k % P) * kLatentDim,
                       static_cast<uint32_t>(rows * kLatentDim));
    };
    for (int jt = 2; jt < 2 + kPrefetchAhead; ++jt) prefetch_tile(jt);
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
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
      if (j >= 2) {
        bool w = true;
        if (lane == 0) w = mbar_wait(&ctrl->raw_empty[s], ((j >> 1) - 1) & 1, abort_flag);
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
      prefetch_tile(j + 2 + kPrefetchAhead);
      __syncwarp();
    }
    if (bad_pid && lane == 0) atomicOr(p.status, kStatusDeviceArg);
    if (!ok && lane == 0) {
      drain_wait(&ctrl->q_full, 0);
      for (int s = 0; s < 2; ++s)
        if (last_issued[s] >= 0) drain_wait(&ctrl->raw_full[s], (last_issued[s] >> 1) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ BMM1 issuer (whole warp,
    // uniform control flow; one elected thread issues the MMAs and their commits)
    const uint32_t idesc1 = make_idesc_e4m3(64, 64);
    const uint64_t qhi_desc = make_smem_desc_sw64(smem_u32(smem + kOffQ8));
    const uint64_t qlo_desc = make_smem_desc_sw64(smem_u32(smem + kOffQ8 + kQPart));
    bool ok = mbar_wait(&ctrl->q_ready, 0, abort_flag);
    // BMM1(j) as soon as raw tile j has landed and its S buffer is free.  Issuing blocks
    // while the tensor pipe is busy, so BMM2 has a warp of its own and is never held behind
    // this warp's issue loop.
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1, sb = j & 1;
      if (ok) ok = mbar_wait(&ctrl->raw_full[s], (j >> 1) & 1, abort_flag);
      if (ok && j >= 2) ok = mbar_wait(&ctrl->s_free[sb], ((j - 2) >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint64_t k_desc = make_smem_desc_sw64(smem_u32(smem + kOffRaw + s * kRawTile));
      const uint32_t d = tmem + kTmemS + sb * 64;
      // the q descriptors pass through an empty asm on every issue, so that the compiler
      // adds the 36 offsets here instead of keeping 36 precomputed descriptors live
      uint64_t qh = qhi_desc, ql = qlo_desc;
      asm volatile("" : "+l"(qh), "+l"(ql));
      if (elect_one()) {
        // S = q_hi . k + q_lo . k: 2 x 9 blocks x 2 K-steps of 32 codes
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int c = 0; c < kBlocks; ++c) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint64_t off = static_cast<uint64_t>((c * kRawBlock + k * 32) >> 4);
              umma_e4m3(d, (part == 0 ? qh : ql) + off, k_desc + off, idesc1, (part | c | k) != 0 ? 1u : 0u);
            }
          }
        }
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
    const uint32_t idesc2 = make_idesc_f16(128, nq, true, false);
    const uint64_t p_desc = make_smem_desc(smem_u32(smem + kOffP), 16, 1024);
    const uint64_t v_desc = make_smem_desc(smem_u32(smem + kOffV), kF16Block, 1024);
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      if (ok) ok = mbar_wait(&ctrl->p_full, j & 1, abort_flag);
      if (ok) ok = mbar_wait(&ctrl->v_full, j & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t voff = static_cast<uint64_t>((2 * qc * kF16Block + kk * 2048) >> 4);
            const uint64_t poff = static_cast<uint64_t>((kk * 32) >> 4);
            umma_bf16(tmem + qc * 64, v_desc + voff, p_desc + poff, idesc2, (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&ctrl->o_done);
        umma_commit(&ctrl->v_empty);
      }
      __syncwarp();
    }
    if (elect_one()) {
      umma_commit(&ctrl->mma_drain2);
      drain_wait(&ctrl->mma_drain2, 0);
    }
    __syncwarp();
  } else if (warp >= kDecodeWarp0 && warp < kBmm2Warp) {
    // ------------------------------------------------------------------ decode warps
    const int dt = threadIdx.x - kDecodeWarp0 * 32;
    bool ok = mbar_wait(&ctrl->q_full, 0, abort_flag);
    if (ok) {
      // Q split: row r is taken by kQThreadsPerRow adjacent threads; thread h of them takes
      // bf16 chunks [8h/n, 8(h+1)/n) of every 64-column block (e4m3 chunks [4h/n, 4(h+1)/n)).
      constexpr int kE8 = 4 / kQThreadsPerRow;  // e4m3 chunks (16 codes) per block for this thread
      const int r = dt / kQThreadsPerRow, h = dt % kQThreadsPerRow;
      const uint32_t qb = smem_u32(smem + kOffQBf16) + r * 128;
      float mx = 0.f;
      for (int c = 0; c < kBlocks; ++c) {
#pragma unroll
        for (int jj = 0; jj < 2 * kE8; ++jj) {
          uint32_t w[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(qb + c * kF16Block + (((2 * kE8 * h + jj) ^ (r & 7)) << 4)));
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        }
      }
#pragma unroll
      for (int o = 1; o < kQThreadsPerRow; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      int sh = 0;  // the row's power-of-two scale: its largest |q| lands in [128, 256)
      if (mx > 0.f) sh = min(126, max(-120, 7 - (static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127)));
      const float mult = __uint_as_float(static_cast<uint32_t>(sh + 127) << 23);
      if (h == 0) ctrl->q_unscale[r] = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
      const uint32_t qhi = smem_u32(smem + kOffQ8) + r * 64;
      const int sw8 = (r >> 1) & 3;  // the 64-byte swizzle of row r
      for (int c = 0; c < kBlocks; ++c) {
#pragma unroll
        for (int e2 = 0; e2 < kE8; ++e2) {
          const int e = kE8 * h + e2;  // e4m3 chunk (16 codes) = bf16 chunks 2e and 2e+1
          uint32_t w[8];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(qb + c * kF16Block + (((2 * e) ^ (r & 7)) << 4)));
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                       : "r"(qb + c * kF16Block + (((2 * e + 1) ^ (r & 7)) << 4)));
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
          const uint32_t off = c * kRawBlock + ((e ^ sw8) << 4);
          st_shared_v4(qhi + off, hi4[0], hi4[1], hi4[2], hi4[3]);
          st_shared_v4(qhi + kQPart + off, lo4[0], lo4[1], lo4[2], lo4[3]);
        }
      }
      fence_proxy_async_smem();
    }
    // every decode thread has read the bf16 Q tile before any writes the V stage over it
    named_bar_sync(2, kDecodeThreads);
    if (ok) mbar_arrive(&ctrl->q_ready);
    // V decode: raw chunk q = dt + kDecodeThreads i of the tile's eight value blocks (2048
    // chunks): block q / 256, row (q % 256) / 4, 16-code chunk q % 4 -> two 16-byte f16
    // chunks of the row.
    // The raw V bytes of tile j go to registers as soon as the tile lands, and the raw stage
    // is released at once (BMM1 releases it too): its refill need not wait for the V stage,
    // which frees only when BMM2(j - 1) completes.  Then the f16 values are written.
    constexpr int kPerThread = 2048 / kDecodeThreads;
    for (int j = 0; ok && j < ntiles; ++j) {
      const int s = j & 1;
      ok = mbar_wait(&ctrl->raw_full[s], (j >> 1) & 1, abort_flag);
      if (!ok) break;
      const int valid_rows = L - (kv_start + j * kTileKeys);  // rows past the request end become zeros
      const uint32_t raw = smem_u32(smem + kOffRaw + s * kRawTile);
      uint4 w[kPerThread];
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) {
        const int q = dt + kDecodeThreads * i;
        const int blk = q >> 8, row = (q >> 2) & 63, jc = q & 3;
        w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (row < valid_rows) {
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[i].x), "=r"(w[i].y), "=r"(w[i].z), "=r"(w[i].w)
                       : "r"(raw + blk * kRawBlock + row * 64 + ((jc ^ ((row >> 1) & 3)) << 4)));
        }
      }
      mbar_arrive(&ctrl->raw_empty[s]);
      if (j >= 1) ok = mbar_wait(&ctrl->v_empty, (j - 1) & 1, abort_flag);
      if (!ok) break;
      const uint32_t vst = smem_u32(smem + kOffV);
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) {
        const int q = dt + kDecodeThreads * i;
        const int blk = q >> 8, row = (q >> 2) & 63, jc = q & 3;
        store_f16_chunk(vst + blk * kF16Block + row * 128 + jc * 32, (row & 7) << 4, w[i]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&ctrl->v_full);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    // BMM1 runs with M = 64: folded row r lives in TMEM lane 32*(r/16) + r%16, so warp w
    // owns rows 16w .. 16w+15.  Each row is split between lanes i and i+16 of its warp:
    // lane i takes keys 0-31 of every tile, lane i+16 keys 32-63.
    const int half = lane >> 4;
    const bool row_lane = half == 0;
    const int r = warp * 16 + (lane & 15);
    const bool row_active = r < nrows;
    const int t = (row0 + r) / p.H;
    const int lim_abs = L - p.T + t;  // last visible key of this row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_used = -INFINITY;
    float l_sum = 0.f;
    // the rows' 2^-s are written once q_ready completes (CTA-uniform over the four warps,
    // since every later barrier among them counts all 128 threads)
    bool failed = bar_or(1, kSoftmaxThreads, !mbar_wait(&ctrl->q_ready, 0, abort_flag));
    // S holds (q 2^s) . k_code: the row's 2^-s and kv_scale (in p.scale_log2) return here.
    // V is decoded as codes times 2^-8 (exact); that factor returns in the output scale.
    const float scale_log2 = failed ? 0.f : p.scale_log2 * ctrl->q_unscale[r];
    const float v_scale = p.v_scale * 256.f;

    for (int j = 0; !failed && j < ntiles; ++j) {
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
        const int lim = row_active ? (min(kv_end - 1, lim_abs) - k0 - 32 * half) : -1;
        online_softmax_step<32, true, true>(sr, lim, scale_log2, kRescaleThreshold, m_used, l_sum, packed, alpha,
                                            need_rescale);
      }
      if (!fail && j >= 1) {
        fail = !mbar_wait(&ctrl->o_done, (j - 1) & 1, abort_flag);
        fail = __any_sync(0xffffffffu, fail);
      }
      if (!fail) {
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
      if (bar_or(1, kSoftmaxThreads, fail || (*abort_flag != 0))) {
        failed = true;
        break;
      }
      if (ctrl->rescale_flag[0] | ctrl->rescale_flag[1] | ctrl->rescale_flag[2] | ctrl->rescale_flag[3]) {
        // O^T[dim, row] *= alpha[row] for all 512 value columns; this thread owns TMEM lane
        // (warp*32 + lane) of each 128-column chunk.  Rows 32hh .. 32hh+31 at a time, so
        // that only their 32 factors are held in registers.
        tc_fence_after();
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
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&ctrl->p_full);
    }

    if (!failed) failed = !mbar_wait(&ctrl->o_done, (ntiles - 1) & 1, abort_flag);
    if (bar_or(1, kSoftmaxThreads, failed || (*abort_flag != 0))) {
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
      named_bar_sync(1, kSoftmaxThreads);
      // Normalised O (bf16) is transposed through the V stage (free once the last BMM2 has
      // completed) so that global stores are whole 16-byte row chunks.
      const uint32_t stage_s = smem_u32(smem + kOffV);  // [64][512] bf16
      // rows 32hh .. 32hh+31 at a time: their 32 scales stay in registers (shared-memory
      // loads interleaved with the staging stores would each wait for the stores before them)
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
      const __nv_bfloat16* stage_h = reinterpret_cast<const __nv_bfloat16*>(smem + kOffV);
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
  if (warp == 5) {
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
    e = cudaFuncSetAttribute(decode_partial_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(head_groups, p.max_splits, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_partial_e4m3_kernel, tm_q, tm_kv, p);
}

}  // namespace mla
