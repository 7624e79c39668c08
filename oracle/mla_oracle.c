/*
 * mla_oracle.c -- plain, slow, obviously-correct CPU oracle for MLA attention over a
 * paged latent KV cache.  TEST INFRASTRUCTURE ONLY: the library's product path never
 * links, loads or calls this file.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.
 *
 * Everything is computed in IEEE double precision with straight loops in the order the
 * definition is written: no blocking, no splitting, no online softmax, no fusion.
 *
 * Sources (the pages never print MLA as an equation; what they fix is stated here):
 *  - "构建面向 Agentic 推理的下一代 LLM 推理引擎" (AICon 2026 talk transcript), section
 *    "Kernel：让 MLA 真正跑满 GPU": MLA compresses K and V into one latent state shared
 *    by all heads; in decode the first matmul is query x latent key; the speculative
 *    decode path feeds several query tokens per request; the prefill path is a ragged,
 *    no-padding batch whose Q and KV lengths differ because a long prefix is cached.
 *  - "TokenSpeed 深度解析" (gitread.org), section "核心技术揭秘", paragraph on paged KV:
 *    KV lives in fixed-size blocks located through a table.
 *  - The attention itself is the textbook definition softmax(scale * q . k_j) weighted
 *    sum of v_j, with the latent row (576 = 512 latent + 64 rope columns) serving as the
 *    key and its first 512 columns as the value (absorbed MLA).
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *  - seq_lens[b] counts every cached token INCLUDING the q_len draft tokens, which are
 *    the last q_len positions; draft t (0-based) sees keys 0 .. L_b - T + t.  A flag
 *    selects the other reading (drafts appended after L_b) for completeness.
 *  - lse is the natural log of sum_j exp(s_j) with s_j the scaled score.
 *  - FP8 KV is OCP e4m3fn (bias 7, no infinities, S.1111.111 is NaN) times one
 *    per-tensor scale; the decode table below is built from that format definition.
 *  - INT8 KV (the talk's section "Kernel：让 MLA 真正跑满 GPU" names INT8 among the KV
 *    quantisations that stay bandwidth-bound) is read as two's-complement int8 codes
 *    times one per-tensor scale, the plainest form the talk leaves open; or, with a
 *    scale per page, each code times the scale of the page that holds its row.
 *  - Prefill: request b has prefix_lens[b] cached tokens followed by its new tokens;
 *    new token i (0-based) sees keys 0 .. prefix_lens[b] + i.
 *
 * Parity pins: every function here is pinned by tests under tests/ (library SDPA on
 * tiny shapes, closed forms, invariants, the full e4m3 code table); none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* Element decoding (exact).                                                             */
/* ------------------------------------------------------------------------------------ */

/* bfloat16 is the upper 16 bits of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * exponent field 0  -> subnormal: (-1)^s * 2^(1-7) * (m/8)
 * exponent 1..15    -> normal:    (-1)^s * 2^(e-7) * (1 + m/8)
 * the single pattern e=15, m=7 (either sign) is NaN; there are no infinities.         */
double oracle_e4m3_to_double(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, 1 - 7);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* kv_dtype: 0 = bf16 (uint16 bit patterns), 1 = e4m3 bytes times kv_scale,
 * 2 = int8 (two's complement) codes times kv_scale (the caller passes the scale of the
 * element's page when the pool has one per page). */
static double kv_elem(const void* pool, int kv_dtype, int64_t idx, double kv_scale) {
  if (kv_dtype == 0) return bf16_bits_to_double(((const uint16_t*)pool)[idx]);
  if (kv_dtype == 2) return (double)((const int8_t*)pool)[idx] * kv_scale;
  return oracle_e4m3_to_double(((const uint8_t*)pool)[idx]) * kv_scale;
}

/* ------------------------------------------------------------------------------------ */
/* One attention row: scores over the visible keys, max-shifted exponentials, weighted  */
/* sum of values, log-sum-exp.  key(j, c) supplies latent column c of visible key j.    */
/* ------------------------------------------------------------------------------------ */

/* Decode: absorbed MLA over the paged latent cache.
 *
 *   q          [B, T, H, D] bf16 bits                 (D = 576 latent + rope columns)
 *   kv_pool    [n_pages, page_size, D] bf16 bits, e4m3 bytes or int8 codes
 *   page_scales optional [n_pages] double (int8 pools only): the scale of each page's
 *              codes, used instead of kv_scale; NULL = one kv_scale for the pool
 *   page_table [B, max_pages] int32: latent row j of request b lives at
 *              kv_pool[page_table[b, j / page_size], j % page_size, :]
 *   seq_lens   [B] int32 cached tokens per request
 *   out        [B, T, H, Dv] double   (V = first Dv columns of the latent row)
 *   lse        [B, T, H] double, natural log
 *   rows       optional list of n_rows flat row ids r = (b*T + t)*H + h; NULL = all rows.
 *              With a list, out/lse are [n_rows, Dv] / [n_rows] in list order.
 * Returns 0, or -1 on an argument error (a row with no visible key, a page id out of
 * range, a length beyond the table).                                                   */
int oracle_mla_decode(int B, int T, int H, int D, int Dv, int page_size, const uint16_t* q,
                      const void* kv_pool, int kv_dtype, double kv_scale, const double* page_scales,
                      int64_t n_pages, const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                      double scale, int lens_include_drafts, const int64_t* rows,
                      int64_t n_rows, double* out, double* lse) {
  int64_t total = rows ? n_rows : (int64_t)B * T * H;
  int err = 0;
  if (page_scales && kv_dtype != 2) return -1;
  /* argument checks first, serially */
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b] + (lens_include_drafts ? 0 : T);
    if (seq_lens[b] < 0 || L < T || (L + page_size - 1) / page_size > max_pages) return -1;
    for (int64_t p = 0; p < (L + page_size - 1) / page_size; ++p) {
      int32_t pid = page_table[(int64_t)b * max_pages + p];
      if (pid < 0 || pid >= n_pages) return -1;
    }
  }
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t i = 0; i < total; ++i) {
    int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= (int64_t)B * T * H) { err |= 1; continue; }
    int h = (int)(r % H);
    int t = (int)((r / H) % T);
    int b = (int)(r / ((int64_t)H * T));
    int64_t L = seq_lens[b] + (lens_include_drafts ? 0 : T);
    int64_t last = L - T + t; /* inclusive index of the last visible key */
    int64_t nvis = last + 1;
    const uint16_t* qrow = q + r * D;
    double* s = (double*)malloc(sizeof(double) * (size_t)nvis);
    double* o = out + i * Dv;
    if (!s) { err |= 1; continue; }
    /* scores */
    for (int64_t j = 0; j < nvis; ++j) {
      int32_t pid = page_table[(int64_t)b * max_pages + j / page_size];
      int64_t base = ((int64_t)pid * page_size + j % page_size) * D;
      double sc = page_scales ? page_scales[pid] : kv_scale;
      double acc = 0.0;
      for (int c = 0; c < D; ++c) acc += bf16_bits_to_double(qrow[c]) * kv_elem(kv_pool, kv_dtype, base + c, sc);
      s[j] = scale * acc;
    }
    /* softmax normaliser */
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) m = s[j] > m ? s[j] : m;
    double Z = 0.0;
    for (int64_t j = 0; j < nvis; ++j) { s[j] = exp(s[j] - m); Z += s[j]; }
    /* weighted sum of values */
    for (int c = 0; c < Dv; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
      int32_t pid = page_table[(int64_t)b * max_pages + j / page_size];
      int64_t base = ((int64_t)pid * page_size + j % page_size) * D;
      double sc = page_scales ? page_scales[pid] : kv_scale;
      double w = s[j];
      for (int c = 0; c < Dv; ++c) o[c] += w * kv_elem(kv_pool, kv_dtype, base + c, sc);
    }
    for (int c = 0; c < Dv; ++c) o[c] /= Z;
    lse[i] = m + log(Z);
    free(s);
  }
  return err ? -1 : 0;
}

/* Prefill: ragged batch, no padding, causal with a cached-prefix offset.
 *
 *   q   [sum n_b, H, Dqk] bf16 bits, request b's new tokens at rows cu_q[b] .. cu_q[b+1]-1
 *   k   [sum (p_b + n_b), H, Dqk] bf16 bits, request b at rows cu_kv[b] .. cu_kv[b+1]-1
 *   v   [sum (p_b + n_b), H, Dv]  bf16 bits
 *   prefix_lens[b] = p_b; kv length of request b must equal p_b + n_b.
 *   out [sum n_b, H, Dv] double; lse [sum n_b, H] double (natural log).
 *   rows optional flat ids r = token * H + h (token indexes q's first axis).
 * New token i of request b sees keys 0 .. p_b + i of its own request.                   */
int oracle_mla_prefill(int B, int H, int Dqk, int Dv, const int32_t* cu_q, const int32_t* cu_kv,
                       const int32_t* prefix_lens, const uint16_t* q, const uint16_t* k,
                       const uint16_t* v, double scale, const int64_t* rows, int64_t n_rows,
                       double* out, double* lse) {
  for (int b = 0; b < B; ++b) {
    int64_t n = cu_q[b + 1] - cu_q[b];
    int64_t kvl = cu_kv[b + 1] - cu_kv[b];
    if (n < 0 || prefix_lens[b] < 0 || kvl != prefix_lens[b] + n) return -1;
  }
  int64_t ntok = cu_q[B];
  int64_t total = rows ? n_rows : ntok * H;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t i = 0; i < total; ++i) {
    int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= ntok * H) { err |= 1; continue; }
    int h = (int)(r % H);
    int64_t tok = r / H;
    int b = 0;
    while (b + 1 <= B && cu_q[b + 1] <= tok) ++b; /* request owning this token */
    int64_t il = tok - cu_q[b];
    int64_t nvis = (int64_t)prefix_lens[b] + il + 1;
    const uint16_t* qrow = q + (tok * H + h) * Dqk;
    double* s = (double*)malloc(sizeof(double) * (size_t)nvis);
    double* o = out + i * Dv;
    if (!s) { err |= 1; continue; }
    for (int64_t j = 0; j < nvis; ++j) {
      const uint16_t* krow = k + ((cu_kv[b] + j) * H + h) * Dqk;
      double acc = 0.0;
      for (int c = 0; c < Dqk; ++c) acc += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
      s[j] = scale * acc;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) m = s[j] > m ? s[j] : m;
    double Z = 0.0;
    for (int64_t j = 0; j < nvis; ++j) { s[j] = exp(s[j] - m); Z += s[j]; }
    for (int c = 0; c < Dv; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
      const uint16_t* vrow = v + ((cu_kv[b] + j) * H + h) * Dv;
      double w = s[j];
      for (int c = 0; c < Dv; ++c) o[c] += w * bf16_bits_to_double(vrow[c]);
    }
    for (int c = 0; c < Dv; ++c) o[c] /= Z;
    lse[i] = m + log(Z);
    free(s);
  }
  return err ? -1 : 0;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
