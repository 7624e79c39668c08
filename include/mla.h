/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention (MLA) over a paged latent KV
 * cache on GB300 (sm_103a).
 *
 * Sources.  The operations follow the TokenSpeed pages:
 *  [TALK]  "构建面向 Agentic 推理的下一代 LLM 推理引擎" (AICon 2026 Shenzhen talk
 *          transcript), section "Kernel：让 MLA 真正跑满 GPU": MLA keeps one latent
 *          state shared by all heads; decode's first matmul is query x latent key with a
 *          query length of one, so query tokens are folded into the head axis; the KV
 *          loop is split into a partial stage and a reduction stage whose split count
 *          and workspace size are computed automatically at run time and cached; the
 *          prefill path is a ragged no-padding batch whose Q and KV lengths differ
 *          because a long prefix (>90% hit rate) is cached and only a few hundred tokens
 *          are appended.  Even with 8-bit KV, loading KV is the bottleneck.
 *  [BLOG]  "英偉達力薦，小團隊兩個月開源一款「光速級」智能體推理引擎" (Synced repost of the
 *          TokenSpeed launch blog), sections "TokenSpeed 技術簡介" and "TokenSpeed 性能
 *          預覽": the decode kernel folds the query-sequence axis into the head axis to
 *          fill the M tile of the first batched matmul; decode is benchmarked with
 *          speculative decoding at batch 4/8/16 over long prefixes; prefill is "prefill
 *          with a long prefix KV cache".
 *  [READ]  "TokenSpeed 深度解析" (gitread.org), section "核心技术揭秘": KV is managed in
 *          fixed-size blocks reached through a table (paged KV).
 *
 * Shapes used throughout: B requests, T = q_len draft tokens per request (1..8192; beyond
 * a few drafts this is the prefill of T new tokens over a paged prefix, absorbed form), H heads,
 * D = 576 latent columns (512 latent + 64 rope), Dv = 512 (the value is the first 512
 * latent columns).  Prefill: 16-bit q/k with Dqk = 192 and v with Dv' = 128.
 *
 * Conventions shared by every call:
 *  - Every pointer argument that is not documented as host memory is DEVICE memory owned
 *    by the caller.  The library never allocates or frees device memory and never
 *    synchronises the stream in mla_decode / mla_prefill_varlen / mla_prefill_paged.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Tensors are dense and row-major (last index fastest), with the layouts given below.
 *  - Every call returns an mla_status_t code; no C++ exception crosses this ABI.
 *    Host-side argument checks run before anything is enqueued; on a non-zero return
 *    nothing was launched unless the code is MLA_ERR_CUDA.
 *  - Device-side failures (a bounded wait that ran out, a length beyond the plan) are
 *    recorded in a per-device status word that mla_get_status() reads and clears.
 */
#ifndef MLA_GB300_MLA_H_
#define MLA_GB300_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status_t {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,         /* null pointer, negative size, inconsistent shapes   */
  MLA_ERR_UNSUPPORTED = 2,         /* shape the kernels do not implement (see each call) */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < plan->workspace_bytes            */
  MLA_ERR_CUDA = 4,                /* a CUDA runtime/driver call or launch failed        */
  MLA_ERR_TIMEOUT = 5,             /* a device-side bounded wait expired (status word)   */
  MLA_ERR_DEVICE_ARG = 6           /* device-side argument check failed (status word)    */
} mla_status_t;

typedef enum mla_kv_dtype_t {
  MLA_KV_BF16 = 0, /* latent pool stored as bfloat16                                     */
  MLA_KV_E4M3 = 1, /* latent pool stored as OCP FP8 e4m3fn codes times one kv_scale      */
  MLA_KV_INT8 = 2, /* latent pool stored as two's-complement int8 codes times one kv_scale.
                    * (The TokenSpeed talk, section "Kernel：让 MLA 真正跑满 GPU", names INT8
                    * among the KV quantisations that keep decode bandwidth-bound; a
                    * per-tensor scale is the plainest form it leaves open.)               */
  MLA_KV_INT8_PAGE = 3 /* int8 codes, each page with its own scale: a latent element is its
                        * code times the scale of the page that holds its row (the other
                        * INT8 form the talk leaves open); decoded by mla_decode_int8_paged  */
} mla_kv_dtype_t;

/* Decode plan: a plain value struct filled by mla_decode_plan(); callers treat the
 * fields as read-only.  It fixes the launch shape of mla_decode for one batch layout. */
typedef struct mla_decode_plan_t {
  int32_t batch;             /* B                                                        */
  int32_t q_len;             /* T, draft tokens per request                              */
  int32_t num_heads;         /* H                                                        */
  int32_t page_size;         /* tokens per page                                          */
  int32_t max_pages_per_seq; /* row stride of page_table                                 */
  int32_t kv_dtype;          /* mla_kv_dtype_t                                           */
  int64_t num_pages;         /* pages in the pool (first dimension of kv_pages)          */
  int32_t num_sms;           /* SMs the split count was sized for                        */
  int32_t rows;              /* T*H folded query rows per request                        */
  int32_t head_groups;       /* CTAs along the folded row axis (64 rows each)            */
  int32_t chunk_tokens;      /* keys per split (multiple of 64)                          */
  int32_t max_splits;        /* splits of the longest request                            */
  int32_t max_seq_len;       /* longest planned request; device seq_lens must not exceed */
  int32_t split_major;       /* launch order of the partial kernel's CTAs: 1 = split by
                                split (plans of more than one wave), 0 = request by request */
  size_t workspace_bytes;    /* bytes mla_decode needs in `workspace` (0 = none)         */
} mla_decode_plan_t;

/* Plan one decode launch: pick the keys-per-split chunk (whole 64-key tiles) and size the
 * workspace for the split partials.  The partial kernel runs one CTA per (request, split,
 * 64-row group); the plan estimates the call's duration by dispatching those CTAs in
 * launch order onto the SM that frees first (each costing its tiles plus a fixed
 * start-up and epilogue cost that depends on the pool format, plus the combine when a
 * request is split), over these chunks: the longest request in 1-4 splits (1-32 with more
 * than one row group when the others leave the SMs idle over a tenth of the call), the
 * smallest
 * chunk that keeps the call in one wave of CTAs when the unsplit call fits one, and, with
 * one row group, the chunks that share all tiles evenly over one or two waves (and up to
 * 8 tiles more than the one-wave one).  The chunk
 * with the shortest estimate wins (fewer splits on a tie), so a split is never taken when
 * it lengthens the call by that estimate.  A plan of one row group and more than one wave
 * launches its CTAs split by split (every request's first split, then every request's
 * second, ...: split_major = 1), so that short remainders go last; every other plan
 * launches them request by request.
 * Plans are memoised on all arguments
 * (the split count and workspace are "computed automatically at run time and cached",
 * [TALK] Kernel section).
 *   seq_lens_host : HOST int32[batch], tokens cached per request INCLUDING the q_len
 *                   draft tokens (the drafts are the last q_len positions).
 *   num_sms       : SMs to plan for; 0 = query the current device.
 * Errors: MLA_ERR_INVALID_ARG (null pointers, batch < 1, a length < q_len or beyond
 * max_pages_per_seq*page_size), MLA_ERR_UNSUPPORTED (q_len > 8192, page_size not one
 * of 8,16,32,64,128,256, or more than 131072 folded rows), MLA_ERR_CUDA (device query). */
int mla_decode_plan(int batch, const int32_t* seq_lens_host, int q_len, int num_heads,
                    int page_size, int max_pages_per_seq, int64_t num_pages, int kv_dtype,
                    int num_sms, mla_decode_plan_t* plan_out);

/* Absorbed MLA decode with speculative draft tokens over the paged latent cache.
 *   q          : [B, T, H, 576] bf16.  Folded row m = t*H + h of request b.
 *   kv_pages   : [num_pages, page_size, 576] bf16, e4m3 or int8 bytes (plan->kv_dtype);
 *                the allocation must hold all num_pages pages in the plan's format (the
 *                library cannot check it: a pool of another format is read out of bounds).
 *   page_table : [B, max_pages_per_seq] int32; latent row j of request b is
 *                kv_pages[page_table[b, j / page_size], j % page_size, :].
 *   seq_lens   : [B] int32 device copy of the planned lengths (each <= max_seq_len).
 *   scale      : softmax scale applied to q . k.
 *   kv_scale   : per-tensor dequantisation scale of an 8-bit pool (ignored for bf16).
 *   out        : [B, T, H, 512] bf16, out[b,t,h] = sum_j softmax_j(scale q.k_j) v_j with
 *                draft t seeing keys 0 .. L_b - T + t and v_j = k_j[:512].
 *   lse        : [B, T, H] fp32, natural-log log-sum-exp of the scaled scores.
 *   workspace  : device scratch of workspace_bytes >= plan->workspace_bytes, 256-byte
 *                aligned; may be NULL when plan->workspace_bytes == 0.  Its contents are
 *                overwritten; calls that share one workspace must be stream-ordered.
 * Enqueues the split-KV partial kernel and, when any request has more than one split,
 * the LSE-merge combine kernel on `stream`.  No allocation, no host synchronisation.
 * Both are programmatic dependent launches: the partial kernel may set itself up while the
 * stream's previous kernel finishes, but reads no input before that kernel has completed;
 * the combine waits in the same way for the partial kernel.  A kernel enqueued after this
 * call as a programmatic dependent must itself wait (griddepcontrol.wait or
 * cudaGridDependencySynchronize) before it reads out or lse.
 * Errors: MLA_ERR_INVALID_ARG (null pointers, q_len/num_heads differ from the plan,
 * misaligned pointers: q, kv_pages 16-byte, out 16-byte), MLA_ERR_WORKSPACE_TOO_SMALL,
 * MLA_ERR_CUDA (tensor-map encoding or launch failure).  Device-side, recorded in the
 * status word as MLA_ERR_DEVICE_ARG (read by mla_get_status): a length below q_len or
 * beyond the plan (that request is skipped, its out/lse rows left unwritten), and a page
 * id outside [0, num_pages) (the rows it names are read as zeros, never from outside the
 * pool). */
int mla_decode(const mla_decode_plan_t* plan, const void* q, const void* kv_pages,
               const int32_t* page_table, const int32_t* seq_lens, int q_len, int num_heads,
               float scale, float kv_scale, void* out, float* lse, void* workspace,
               size_t workspace_bytes, void* stream);

/* mla_decode over an int8 pool with one scale per page (plan->kv_dtype ==
 * MLA_KV_INT8_PAGE; mla_decode and mla_decode_partial reject such plans).  Arguments,
 * layouts and errors as mla_decode, with:
 *   kv_pages    : [num_pages, page_size, 576] int8 codes.
 *   page_scales : [num_pages] fp32 on the device, 4-byte aligned: the scale of each page's
 *                 codes (element = code * page_scales[page]).
 *   kv_scale    : a reference scale > 0 (the largest page scale is the natural choice).
 *                 Each page scale must lie in [0, 255 * kv_scale]; a page scale outside it
 *                 (or not finite) on a page a request reads is reported as
 *                 MLA_ERR_DEVICE_ARG and that request's split is skipped.
 * The codes are multiplied exactly as int8 values; each key's page scale relative to
 * kv_scale multiplies its score (in fp32) and the softmax weight its value row receives,
 * and kv_scale itself is folded into the softmax scale and the output.  The combine
 * stage is the one of mla_decode: mla_decode_combine accepts these plans. */
int mla_decode_int8_paged(const mla_decode_plan_t* plan, const void* q, const void* kv_pages,
                          const float* page_scales, const int32_t* page_table, const int32_t* seq_lens,
                          int q_len, int num_heads, float scale, float kv_scale, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The two stages of mla_decode, for callers that schedule them apart (e.g. to put other
 * work between them, or to time the split-KV partial kernel on its own).  The TokenSpeed
 * talk ("构建面向 Agentic 推理的下一代 LLM 推理引擎", section "Kernel：让 MLA 真正跑满 GPU")
 * describes the kernel as a split-KV partial stage followed by a reduction stage; these
 * calls expose that split.  mla_decode(...) is exactly mla_decode_partial(...) followed by
 * mla_decode_combine(...) on the same stream with the same plan, workspace, out and lse.
 *
 * mla_decode_partial: arguments, layouts and errors as mla_decode.  Enqueues the split-KV
 * partial kernel only.  Requests whose plan gives them one split get their final out/lse
 * rows; the others leave per-split bf16 partial outputs and fp32 log-sum-exps in the
 * workspace, which stay valid until the workspace is next written.
 *
 * mla_decode_combine: merges those partials into out/lse (log-sum-exp weighted mean over
 * the splits of each request).  plan, seq_lens, q_len, num_heads, out, lse and workspace
 * must be the ones given to the mla_decode_partial call it completes, stream-ordered
 * after it.  Enqueues nothing when no request has more than one split.  Errors:
 * MLA_ERR_INVALID_ARG (null plan/seq_lens/out/lse, q_len/num_heads differ from the plan,
 * out not 16-byte or lse not 4-byte aligned, workspace missing or not 256-byte aligned),
 * MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_CUDA (launch failure). */
int mla_decode_partial(const mla_decode_plan_t* plan, const void* q, const void* kv_pages,
                       const int32_t* page_table, const int32_t* seq_lens, int q_len, int num_heads,
                       float scale, float kv_scale, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream);
int mla_decode_combine(const mla_decode_plan_t* plan, const int32_t* seq_lens, int q_len,
                       int num_heads, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream);

/* mla_decode for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is a library convenience.)  Some callers cannot call cudaMalloc, e.g.
 * a serving engine whose memory manager gives every free byte of the device to its
 * KV-cache pool at start-up and refuses later allocations, or a plugin loaded into a host
 * program that offers it no allocator.  This entry point takes the same arguments as
 * mla_decode minus the workspace, and uses as scratch a fixed 32 MiB buffer that lives in
 * the library's own device data: every GPU that loads libmla holds those 32 MiB until the
 * process exits.  It allocates and frees nothing.
 *  - Limit: plan->workspace_bytes must be <= 32 MiB (33554432); larger plans are rejected
 *    with MLA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - The first call on each device looks up the buffer's device address (with that device
 *    current); make that first call before any stream capture.
 *  - All calls on a device share the one buffer, which keeps the previous call's
 *    contents.  Nothing in it has to start at zero: each call writes every partial it
 *    later reads.  Calls whose kernels overlap on the GPU (other streams, other threads)
 *    race on the buffer and corrupt each other's results: order them on one stream.
 * Errors: as mla_decode, plus MLA_ERR_WORKSPACE_TOO_SMALL for plans beyond the limit. */
int mla_decode_noalloc(const mla_decode_plan_t* plan, const void* q, const void* kv_pages,
                       const int32_t* page_table, const int32_t* seq_lens, int q_len, int num_heads,
                       float scale, float kv_scale, void* out, float* lse, void* stream);

/* Ragged (no padding) causal MLA prefill on top of a cached prefix.
 *   q             : [total_q, H, 192] bf16; request b's n_b new tokens are rows
 *                   cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1.
 *   k             : [total_kv, H, 192] bf16; request b's p_b + n_b keys (prefix first) are
 *                   rows cu_seqlens_kv[b] .. cu_seqlens_kv[b+1]-1.
 *   v             : [total_kv, H, 128] bf16, same rows as k.
 *   cu_seqlens_q, cu_seqlens_kv : [batch+1] int32 prefix sums (device).
 *   prefix_lens   : [batch] int32 p_b (device); kv length must equal p_b + n_b.
 *   max_seqlen_q  : host bound on n_b (sizes the grid).
 *   total_q, total_kv : host row counts of q and k/v (bounds of the tensor maps).
 *   out           : [total_q, H, 128] bf16; new token i of request b attends to keys
 *                   0 .. p_b + i of its own request.
 *   lse           : [total_q, H] fp32 natural-log log-sum-exp.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (num_heads < 1 or > 256),
 * MLA_ERR_CUDA.  Device-side, recorded in the status word as MLA_ERR_DEVICE_ARG (read by
 * mla_get_status) before any load or store of the request: its kv length differs from
 * p_b + n_b, n_b > max_seqlen_q, or its rows reach beyond total_q / total_kv.  That
 * request is skipped and its out/lse rows are left unwritten.
 * Scratch: a q block with 8 or more tiles of 128 keys runs as two CTAs over the halves of
 * its keys, which merge through this library's own device scratch (32 MiB per GPU, 1024
 * slots; q blocks past them are not split).  Prefill calls whose kernels overlap on the
 * GPU (other streams, other threads) race on it: order them on one stream.  The first
 * call on each device and host thread looks the scratch up; make it before any stream
 * capture. */
int mla_prefill_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_kv, const int32_t* prefix_lens, int batch,
                       int num_heads, int max_seqlen_q, int total_q, int total_kv, float scale,
                       void* out, float* lse, void* stream);

/* The same prefill with K/V read from a paged cache of per-head k/v rows instead of
 * contiguous per-request rows.  The TokenSpeed pages describe the prefill as "prefill with a
 * long prefix KV cache" ([BLOG] "TokenSpeed 性能預覽"; [TALK] "Kernel：让 MLA 真正跑满 GPU",
 * last paragraph) and keep KV in fixed-size blocks behind a table ([READ] "核心技术揭秘");
 * this call reads both the cached prefix and the new tokens' k/v from such blocks.
 *   q             : [total_q, H, 192] bf16; request b's n_b new tokens are rows
 *                   cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1.
 *   k_pages       : [num_pages, page_size, H, 192] bf16.
 *   v_pages       : [num_pages, page_size, H, 128] bf16.
 *   page_table    : [batch, max_pages_per_seq] int32; key j of request b (prefix first,
 *                   then its new tokens) is row j % page_size of page
 *                   page_table[b, j / page_size] of k_pages / v_pages.
 *   kv_lens       : [batch] int32 (device), p_b + n_b: the request's cached prefix plus
 *                   its new tokens, whose k/v are the last n_b positions.
 *   page_size     : 16, 32, 64, 128 or 256 tokens.
 *   num_pages     : pages in each pool (num_pages * page_size < 2^31).
 *   out, lse      : as mla_prefill_varlen: new token i of request b attends to keys
 *                   0 .. p_b + i.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (num_heads outside 1..256, another page
 * size, too many pool rows), MLA_ERR_CUDA.  Device-side, recorded in the status word as
 * MLA_ERR_DEVICE_ARG: n_b > max_seqlen_q, kv_lens[b] < n_b or beyond the table row, q rows
 * beyond total_q (the request is skipped, before any access), and a page id outside
 * [0, num_pages) (its rows are read as zeros, never from outside the pools).
 * Scratch: as mla_prefill_varlen (the same library-owned scratch: order every prefill
 * call, contiguous or paged, on one stream). */
int mla_prefill_paged(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                      const int32_t* cu_seqlens_q, const int32_t* kv_lens, int batch, int num_heads,
                      int page_size, int max_pages_per_seq, int64_t num_pages, int max_seqlen_q,
                      int total_q, float scale, void* out, float* lse, void* stream);

/* Read and clear the current device's status word after synchronising `stream`.
 * Returns MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_ARG (first recorded), or
 * MLA_ERR_CUDA if the read itself fails.  This call synchronises: keep it off the hot
 * path. */
int mla_get_status(void* stream);

/* Measurement hook: when start/stop are non-NULL cudaEvent_t handles, subsequent
 * mla_decode calls made from the calling host thread record `start` immediately before
 * and `stop` immediately after the split-KV partial kernel (on the call's stream), and
 * mla_prefill_varlen records them around its kernel.  NULL, NULL turns recording off.
 * The library does not own the events.  Returns MLA_OK. */
int mla_set_profile_events(void* start_event, void* stop_event);

/* Elapsed milliseconds between two events recorded through the hook above (including
 * event nodes replayed from a captured CUDA graph).  Returns MLA_ERR_CUDA if either event
 * has not completed. */
int mla_profile_elapsed_ms(void* start_event, void* stop_event, float* ms_out);

/* Watchdog self-test: enqueue a one-warp kernel that waits, through the same bounded
 * mbarrier wait every MLA kernel uses, on a barrier nothing ever arrives on.  The wait
 * gives up after its limit (1 s) and records MLA_ERR_TIMEOUT in the status word, which
 * the next mla_get_status() returns; the CUDA context stays usable.  Returns MLA_OK once
 * enqueued.  (No counterpart on the pages: it exercises the failure-detection path of
 * this library without faulting or hanging the GPU.) */
int mla_selftest_wait_timeout(void* stream);

/* Static, human-readable name of a status code. */
const char* mla_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_MLA_H_ */
