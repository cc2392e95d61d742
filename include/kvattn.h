/*
 * kvattn.h -- C ABI of the GB300 (sm_103a) decode-phase GQA attention library.
 *
 * One call performs one decode step of grouped-query attention for a batch of
 * sequences, each contributing one new token, over a paged KV cache:
 *
 *   1. half-split RoPE on the new query and key ("C17 CPU-first LLM inference
 *      engine", section 4.4 "Attention: GQA + RoPE"; "LLM inference from
 *      smollm3.go", section "Positional encoding: why the model knows order");
 *   2. append of the new key/value into slot seq_lens[b] of the sequence's
 *      pages ("Qwen3-8B inference engine from scratch in C++/CUDA", section
 *      4.3.1 "Paged KV cache"; smollm3.go page, section "KV cache");
 *   3. scores scale * dot(q_h, k_t) for every cached position t = 0..seq_lens[b]
 *      (the new token included) and their softmax (smollm3.go page, section
 *      "Self-attention: how the current token looks back"; Qwen3-8B page,
 *      section 4.4.2 "GQA grouped decode");
 *   4. the softmax-weighted sum of the cached values.
 * Query head h reads KV head h / (n_qh / n_kvh) (smollm3.go page, section
 * "Multi-head attention").  The optional int8 cache stores per-(token, KV
 * head) fp32 scales max|x| / 127 ("lightLLM, a pure-Python inference
 * framework", section 1 "Overview", Int8KV; smollm3.go page, section "int8
 * weight-only quantization").
 *
 * Conventions shared by every entry point
 *  - Pointers marked "device" are CUDA device (or managed) memory owned by the
 *    caller; the library allocates no memory and keeps no pointer after a call
 *    returns, except that work already queued on `stream` uses them until it
 *    completes.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - Arrays are dense, row-major, with the shapes given; bf16 is IEEE
 *    bfloat16 stored in 2 bytes.
 *  - Host-detectable errors return a non-zero status before anything is
 *    launched.  Calls are asynchronous: no call except
 *    kvattn_read_device_status synchronises.
 *  - Errors found on the device (a sequence length or a block-table entry out
 *    of range) never cause an out-of-bounds access: the offending sequence or
 *    page is skipped and a bit is OR-ed into the device status word kept in the
 *    workspace (KVATTN_DEV_* below).
 */
#ifndef KVATTN_H
#define KVATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define KVATTN_OK 0
#define KVATTN_EINVAL 1       /* a NULL/misaligned pointer, a negative or
                                 inconsistent size, n_qh % n_kvh != 0 */
#define KVATTN_EUNSUPPORTED 2 /* head_dim, page_size, kv_dtype or a size
                                 outside what the library is built for (among
                                 them: n_seq * n_kvh * (G / gs) *
                                 max_pages_per_seq * page_size / 16 above
                                 2^28 - 1, the most 16-token work units a step
                                 can hold; G = n_qh / n_kvh, gs = the largest of
                                 4, 2, 1 dividing G) */
#define KVATTN_ECUDA 3        /* a CUDA runtime call or launch failed */
#define KVATTN_EWORKSPACE 4   /* workspace NULL, misaligned or too small */

/* ---- KV cache element types -------------------------------------------- */
#define KVATTN_KV_BF16 0 /* K/V pages hold bf16 */
#define KVATTN_KV_INT8 1 /* K/V pages hold int8 codes; scales hold fp32 */

/* ---- device status bits (sticky, OR-ed into the workspace) ------------- */
#define KVATTN_DEV_BAD_LEN 1u  /* seq_lens[b] < 0 or seq_lens[b] + 1 >
                                  max_pages_per_seq * page_size: sequence
                                  skipped, its output rows not written */
#define KVATTN_DEV_BAD_PAGE 2u /* a block-table entry needed by the step is
                                  outside [0, num_pages): that page's tokens
                                  are left out (and no append lands there) */
#define KVATTN_DEV_TIMEOUT 4u  /* a bounded wait for an on-chip copy gave up;
                                  results of the call are not valid */

/* ---- limits ------------------------------------------------------------ */
#define KVATTN_MAX_SPLITS 4096 /* largest num_splits of kvattn_decode_splits */
#define KVATTN_MAX_SEQS 8192   /* largest n_seq of one call (per layer) */
#define KVATTN_MAX_LAYERS 1024 /* largest n_layers of kvattn_decode_layers */

/*
 * Bytes of device workspace one decode call needs for this shape.  The
 * workspace holds the device status word and the partial softmax states of
 * the (sequence, KV head, query-head group) streams whose work is split
 * across warps.  0 when the shape is invalid.
 */
size_t kvattn_workspace_size(int n_seq, int n_qh, int n_kvh, int head_dim);

/* Workspace bytes of kvattn_decode_layers over n_layers layer caches (0 when
 * the shape is invalid); n_layers = 1 gives kvattn_workspace_size. */
size_t kvattn_workspace_size_layers(int n_layers, int n_seq, int n_qh, int n_kvh, int head_dim);

/*
 * Zero the workspace (all workspace_bytes, asynchronously on `stream`).  Must
 * be called once before the first kvattn_decode on a workspace, and again
 * after a call that reported KVATTN_DEV_TIMEOUT.  A workspace can be reused
 * for any shape it is large enough for.
 * workspace: device, 256-byte aligned, at least 256 bytes.
 */
int kvattn_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step (see the top of this file), queued on `stream`.
 *
 * q            device bf16 [n_seq, n_qh, head_dim], 16-byte aligned; query
 *              before RoPE.
 * k_new, v_new device bf16 [n_seq, n_kvh, head_dim]; new key (before RoPE)
 *              and value.
 * k_pages,     device [num_pages, n_kvh, page_size, head_dim], bf16 or int8
 * v_pages      per kv_dtype, 16-byte aligned; read, and written only in slot
 *              seq_lens[b] % page_size of page block_table[b][seq_lens[b] /
 *              page_size] for every valid sequence b.  Cached keys are stored
 *              after RoPE.
 * block_table  device int32 [n_seq, max_pages_per_seq]; physical page of each
 *              logical page of a sequence.  The page of slot seq_lens[b] must
 *              already be assigned (page allocation is the caller's policy).
 * seq_lens     device int32 [n_seq]; tokens cached before this step, i.e. the
 *              slot the new token goes to.  Attention covers seq_lens[b] + 1
 *              tokens.
 * positions    device int32 [n_seq]; RoPE position of the new token.
 * out          device bf16 [n_seq, n_qh, head_dim]; attention output, fp32
 *              accumulation rounded to nearest even.
 * n_seq >= 0; with n_seq == 0 the call returns KVATTN_OK once the sizes pass
 *              their checks, without looking at any pointer or launching.
 * n_qh, n_kvh >= 1, n_qh % n_kvh == 0.
 * head_dim     64 or 128.
 * page_size    16, 32, 64, 128 or 256 tokens.
 * rope_theta   RoPE base; <= 0 disables RoPE (a NoPE layer).  Frequency of
 *              pair i is rope_theta^(-2i/head_dim); pairs are (i, i + head_dim/2).
 * scale        score scale (usually 1/sqrt(head_dim)); finite.
 * kv_dtype     KVATTN_KV_BF16 or KVATTN_KV_INT8.
 * stream       cudaStream_t.
 * max_pages_per_seq >= 1: row length of block_table.
 * num_pages >= 1: pages in each of k_pages / v_pages (for bounds checks).
 * k_scales,    device fp32 [num_pages, n_kvh, page_size], 16-byte aligned;
 * v_scales     required for int8 (the scale of each cached row), NULL for bf16.
 * workspace    device, 256-byte aligned, >= kvattn_workspace_size(...) bytes,
 *              initialised once with kvattn_workspace_init.  Calls that share
 *              a workspace must be ordered on one stream (or otherwise not
 *              overlap on the GPU).
 *
 * The appended key is rotated with fp32 cos/sin (computed in double, then
 * rounded), fp32 products and sums each rounded separately, then stored as
 * bf16 (nearest even) or as int8 codes clamp(rint(x / s), -127, 127) with
 * s = max|x| / 127 (s = 0 for an all-zero row); the value is stored as given
 * (bf16) or quantised the same way.  The new token is attended through its
 * stored value.
 */
int kvattn_decode(const void *q, const void *k_new, const void *v_new, void *k_pages,
                  void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                  const int32_t *positions, void *out, int n_seq, int n_qh, int n_kvh,
                  int head_dim, int page_size, float rope_theta, float scale, int kv_dtype,
                  void *stream, int max_pages_per_seq, int num_pages, float *k_scales,
                  float *v_scales, void *workspace, size_t workspace_bytes);

/*
 * kvattn_decode with an explicit work split: the flattened list of 16-token
 * units over all (sequence, KV head) pairs is cut into at most `num_splits`
 * equal shares, one per warp; a sequence cut across shares is finished by a
 * log-sum-exp merge of the shares' partial softmax states.  num_splits = 0
 * picks the default (a multiple of the GPU's SM count); otherwise
 * 1 <= num_splits <= KVATTN_MAX_SPLITS.  Results for different splits agree
 * to fp32 rounding.
 */
int kvattn_decode_splits(const void *q, const void *k_new, const void *v_new,
                         void *k_pages, void *v_pages, const int32_t *block_table,
                         const int32_t *seq_lens, const int32_t *positions, void *out,
                         int n_seq, int n_qh, int n_kvh, int head_dim, int page_size,
                         float rope_theta, float scale, int kv_dtype, void *stream,
                         int max_pages_per_seq, int num_pages, float *k_scales,
                         float *v_scales, void *workspace, size_t workspace_bytes,
                         int num_splits);

/*
 * One decode step over n_layers layer caches in one launch.  The decode phase
 * pays for many small kernel launches ("Qwen3-8B inference engine from
 * scratch in C++/CUDA", section 2.2): when the queries of several layers are
 * ready together (for example a benchmark that runs every layer cache of a
 * step), one call streams all of them in one balanced work split, so the
 * start-up, tail and merge of a call are paid once instead of once per layer.
 * The layers share the block table, lengths and positions (a paged cache keeps
 * one page table for all layers; each layer has its own pool); each layer
 * computes exactly what kvattn_decode computes for it.
 *
 * n_layers     1 <= n_layers <= KVATTN_MAX_LAYERS.
 * q, out       device bf16 [n_layers, n_seq, n_qh, head_dim] (layer-major).
 * k_new, v_new device bf16 [n_layers, n_seq, n_kvh, head_dim].
 * k_pages,     device [n_layers, num_pages, n_kvh, page_size, head_dim]: layer
 * v_pages      l's pool of num_pages pages, then layer l + 1's.
 * k_scales,    device fp32 [n_layers, num_pages, n_kvh, page_size] (int8), or
 * v_scales     NULL (bf16).
 * block_table, seq_lens, positions: as for kvattn_decode, shared by all layers.
 * workspace    >= kvattn_workspace_size_layers(n_layers, ...) bytes, set up as
 *              for kvattn_decode.
 * layer_rope   host uint8 [n_layers] or NULL: a layer whose entry is 0 has no
 *              RoPE (its query and new key are not rotated), as in a model whose
 *              RoPE and NoPE layers alternate ("LLM inference from smollm3.go",
 *              section "Positional encoding: why the model knows order");
 *              NULL: every layer is rotated (unless rope_theta <= 0, which turns
 *              RoPE off for all).  Read during the call only.
 * Other arguments, checks and errors as for kvattn_decode; additionally
 * n_layers * num_pages * n_kvh * page_size must stay below 2^31 (pool rows are
 * addressed with 32-bit coordinates), else KVATTN_EUNSUPPORTED.  With
 * n_layers = 1 the call is kvattn_decode.
 */
int kvattn_decode_layers(int n_layers, const void *q, const void *k_new, const void *v_new,
                         void *k_pages, void *v_pages, const int32_t *block_table,
                         const int32_t *seq_lens, const int32_t *positions, void *out, int n_seq,
                         int n_qh, int n_kvh, int head_dim, int page_size, float rope_theta,
                         float scale, int kv_dtype, void *stream, int max_pages_per_seq,
                         int num_pages, float *k_scales, float *v_scales, void *workspace,
                         size_t workspace_bytes, const uint8_t *layer_rope);

/*
 * Paged chunked prefill: each sequence b brings n_b >= 0 new tokens after the
 * ctx_lens[b] tokens its pages already hold (a prompt, the next chunk of a
 * long one, or the draft tokens of a speculative step to verify).  The new
 * keys and values are appended to slots ctx_lens[b] .. ctx_lens[b] + n_b - 1
 * (keys rotated at those positions with the storage recipe of kvattn_decode),
 * then new token i attends over keys 0 .. ctx_lens[b] + i: causal attention
 * over the cache and the earlier new tokens ("LLM inference from
 * smollm3.go", section "Prefill: the whole prompt at once"; "Qwen3-8B
 * inference engine from scratch in C++/CUDA", section 4.4.1).  A sequence
 * with n_b = 1 gets exactly the decode step (with seq_lens = positions =
 * ctx_lens), for the bf16 and the int8 cache alike (the int8 rows are
 * dequantised to f16 for the tensor cores: code * scale, rounded once).
 *
 * q, out       device bf16 [n_tok, n_qh, head_dim]: the new tokens of all
 *              sequences back to back, 16-byte aligned (out 4-byte).
 * k_new, v_new device bf16 [n_tok, n_kvh, head_dim], 16-byte aligned.
 * k_pages,     device [num_pages, n_kvh, page_size, head_dim], bf16 or int8
 * v_pages      per kv_dtype, as for kvattn_decode; the pages of every appended
 *              slot must be assigned in block_table.
 * k_scales,    as for kvattn_decode (int8 only).
 * v_scales
 * block_table  device int32 [n_seq, max_pages_per_seq].
 * seq_starts   device int32 [n_seq + 1]: sequence b's new tokens are rows
 *              seq_starts[b] .. seq_starts[b + 1] - 1 of q, k_new, v_new, out.
 * ctx_lens     device int32 [n_seq]: tokens cached before the call; new token
 *              i has slot and RoPE position ctx_lens[b] + i.
 * n_qh / n_kvh must be a multiple of 4 (a CTA serves 4 query heads of a group),
 *              else KVATTN_EUNSUPPORTED.
 * max_new_tokens  an upper bound on every n_b; it sizes the launch: up to 4
 *              (speculative drafts), 4 new tokens a sequence are covered, by a
 *              kernel whose MMA rows are 4 tokens x 4 heads; above, the bound
 *              rounded up to a multiple of 16, by 16-token query tiles.  A
 *              sequence with more new tokens than the launch covers has the
 *              rest neither appended nor attended, and KVATTN_DEV_BAD_LEN is
 *              reported.
 * dev_status   device uint32, 4-byte aligned, or NULL: KVATTN_DEV_BAD_LEN is
 *              OR-ed in for a sequence whose rows or slots do not fit (it is
 *              skipped), KVATTN_DEV_BAD_PAGE for a page outside [0, num_pages)
 *              (its tokens are left out, no append lands there).
 * workspace    device, 16-byte aligned, or NULL; workspace_bytes its size.  With
 *              max_new_tokens <= 64 (short chunks over long contexts: a
 *              speculative check) the key tiles of a query tile are shared
 *              among up to 16 CTAs whose partial softmax states are merged by
 *              a third kernel; they need kvattn_prefill_workspace_size(...)
 *              bytes (fewer splits when the workspace is smaller, none
 *              without one).  Its contents need no initialisation and are
 *              not kept between calls; calls sharing a workspace must not
 *              overlap on the GPU.
 * Other arguments, checks and errors as for kvattn_decode.
 */
int kvattn_prefill(const void *q, const void *k_new, const void *v_new, void *k_pages,
                   void *v_pages, const int32_t *block_table, const int32_t *seq_starts,
                   const int32_t *ctx_lens, void *out, int n_seq, int n_tok, int n_qh, int n_kvh,
                   int head_dim, int page_size, float rope_theta, float scale, int kv_dtype,
                   void *stream, int max_pages_per_seq, int num_pages, float *k_scales,
                   float *v_scales, int max_new_tokens, uint32_t *dev_status, void *workspace,
                   size_t workspace_bytes);

/* Workspace bytes kvattn_prefill can use for n_tok new tokens (0 when the
 * shape is invalid). */
size_t kvattn_prefill_workspace_size(int n_tok, int n_qh, int head_dim);

/*
 * kvattn_decode for callers that can neither pass a workspace nor let the
 * library allocate one.  The source pages have no counterpart of this entry
 * point.
 *
 * Such callers exist: an engine that reserved nearly all of HBM for its
 * KV-page pool at start-up and keeps no allocator for anything else, or a
 * plugin inside a host framework that owns every device allocation and does
 * not allow plugins to call cudaMalloc.  The scratch that kvattn_decode keeps
 * in the caller's workspace lives here in one fixed array inside the library,
 * KVATTN_NOALLOC_SCRATCH_BYTES long; every GPU that loads the library holds it
 * until the process exits.  No cudaMalloc/cudaFree or other allocation is
 * made.
 *
 * Arguments: those of kvattn_decode without workspace/workspace_bytes, plus
 * dev_status  device uint32, 4-byte aligned, that receives this call's
 *             KVATTN_DEV_* bits; may be NULL.
 * Returns KVATTN_EUNSUPPORTED, before anything is queued, when the shape needs
 * more scratch than the array holds, i.e. when
 * kvattn_workspace_size(n_seq, n_qh, n_kvh, head_dim) >
 * KVATTN_NOALLOC_SCRATCH_BYTES.
 * The first call on a device (with that device current) looks up the array's
 * device address; make that first call before any stream capture.  That
 * address is kept until the process exits: do not use this entry point
 * across cudaDeviceReset (or any other destruction of the device's primary
 * context), after which the array may lie elsewhere.
 * Every host check of kvattn_decode is made before anything is queued: a
 * call that returns an error has queued no work.
 * Every call uses the same array and finds the previous call's contents in it:
 * calls that overlap on the GPU (other streams, other host threads) race and
 * corrupt each other's results, so order them on one stream.
 */
#define KVATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
int kvattn_decode_noalloc(const void *q, const void *k_new, const void *v_new,
                          void *k_pages, void *v_pages, const int32_t *block_table,
                          const int32_t *seq_lens, const int32_t *positions, void *out,
                          int n_seq, int n_qh, int n_kvh, int head_dim, int page_size,
                          float rope_theta, float scale, int kv_dtype, void *stream,
                          int max_pages_per_seq, int num_pages, float *k_scales,
                          float *v_scales, uint32_t *dev_status);

/*
 * Wait for `stream`, copy the device status word (KVATTN_DEV_* bits OR-ed by
 * every call since the last read or init) into *bits, and clear it.
 * Synchronises `stream`.
 */
int kvattn_read_device_status(void *workspace, void *stream, uint32_t *bits);

/* Static English description of a return code (never NULL). */
const char *kvattn_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int kvattn_version(void);

/*
 * The cudaError_t value behind this thread's most recent KVATTN_ECUDA return
 * (0 when no call on this thread has returned KVATTN_ECUDA).  A pool whose
 * tensor map could not be encoded reports cudaErrorInvalidValue (1).  Not a
 * step of the method: a diagnostic for callers that receive KVATTN_ECUDA.
 */
int kvattn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVATTN_H */
