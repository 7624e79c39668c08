// mla_internal.h -- launch parameter blocks and launcher declarations shared by the host
// API (mla_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int kLatentDim = 576;  // 512 latent + 64 rope columns
constexpr int kValueDim = 512;   // value = first 512 latent columns
constexpr int kTileKeys = 64;    // keys per decode tile
constexpr int kGroupRows = 64;   // folded query rows per decode CTA

// Pool formats of the decode kernel (the values of mla_kv_dtype_t).
constexpr int kKvBf16 = 0;
constexpr int kKvE4m3 = 1;
constexpr int kKvInt8 = 2;
constexpr int kKvInt8Page = 3;  // int8 codes times a scale per page

// Device status word bits (OR-ed by kernels, read and cleared by mla_get_status).
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusDeviceArg = 2u;

struct DecodeParams {
  int B, T, H, R;               // R = T*H folded rows per request
  int page_size, max_pages;     // page geometry and page_table row stride
  int chunk, max_splits, max_seq;
  int split_major;              // grid (groups, B, splits) when set, else (groups, splits, B)
  int kv_dtype;                 // kKvBf16, kKvE4m3, kKvInt8 or kKvInt8Page
  int64_t num_pages;            // pages in the pool: a page id outside [0, num_pages) is reported
  float scale_log2;             // softmax scale * log2(e) (* kv_scale for an 8-bit pool)
  float v_scale;                // 1, or kv_scale for an 8-bit pool (applied in the epilogue)
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* kv_pool;       // pool base (the 8-bit path reads raw rows from here)
  const float* page_scales;     // kKvInt8Page: [num_pages] scale of each page's codes
  float inv_ref_scale;          // kKvInt8Page: 1 / kv_scale (page scales are applied relative to it)
  __nv_bfloat16* out;           // [B, T, H, 512]
  float* lse;                   // [B, T, H]
  __nv_bfloat16* ws_o;          // [B, max_splits, R, 512] partial outputs (normalised, bf16)
  float* ws_lse;                // [B, max_splits, R] partial log-sum-exp (natural log)
  unsigned* status;             // device status word
};

struct PrefillParams {
  int B, H, max_q_blocks;
  int max_seqlen_q;             // host bound on new tokens per request (sizes the grid)
  float scale_log2;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  const int32_t* prefix_lens;
  __nv_bfloat16* out;           // [total_q, H, 128]
  float* lse;                   // [total_q, H]
  int total_q, total_kv;        // rows of q/out/lse and of k/v
  unsigned* status;
  // paged K/V (page_table non-null): row j of request b is row j % page_size of page
  // page_table[b * max_pages + j / page_size]; kv_lens[b] = prefix + new tokens
  const int32_t* page_table;
  const int32_t* kv_lens;
  int page_size, max_pages;
  int64_t num_pages;
};

// Decode: split-KV partial kernel (tensor maps over q and the latent pool).
cudaError_t launch_decode_partial(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                  int head_groups, cudaStream_t stream);
// Decode over an e4m3 pool: the split-KV partial kernel that runs BMM1 on the raw codes.
cudaError_t launch_decode_partial_e4m3(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                       int head_groups, cudaStream_t stream);
// Decode over a bf16 pool for requests of at most 32 folded rows (R <= 32): Q held in
// tensor memory, a three-tile ring (mla_decode_narrow_sm103a.cu).
cudaError_t launch_decode_partial_narrow(const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                         cudaStream_t stream);
// Decode: LSE-merge of the split partials for requests with more than one split.
cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream);
// Watchdog self-test kernel (a wait nothing satisfies; must time out and report).
cudaError_t launch_selftest_timeout(unsigned* status, cudaStream_t stream);
// Prefill: ragged causal prefill with prefix offset (contiguous or paged K/V, by p.page_table).
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, cudaStream_t stream);

}  // namespace mla
