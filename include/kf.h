/*
 * kf.h -- C ABI of the GB300 (sm_103a) split-KV paged decode attention library.
 *
 * The operation: one decode step of attention for a batch of requests, each
 * with one new query token, over a paged KV cache read through a block
 * table, in split-KV form: a request's tokens are cut into ranges, each range
 * yields a partial (o, lse), and the partials are combined by an exact
 * log-sum-exp merge.
 *
 * Sources (pages this library restates):
 *  - KernelFlume (academ.us/article/2606.29207), section 3.1 "Kernel-level
 *    Disaggregation" and 3.2 "Workflow of Elastic Decoding": attention nodes
 *    own token-range partitions of the KV cache; the tail node appends the
 *    step's K_new/V_new, then every node computes local attention and returns
 *    partials (o_i, m_i, l_i), which are merged by the online-softmax (LSE)
 *    reduction; section 5.1: the merge equals attention over the full range.
 *  - "Disaggregated Inference Architecture: Paged KV-Cache Tiering, Chunked
 *    Prefill, and Asynchronous Overlap" (ultrainstinct.tech), "Physical Memory
 *    Block Layout" (blocks of block_size tokens x H_KV x D, a block table from
 *    logical to physical blocks) and "Mathematical Formulation of Chunked
 *    Attention" (the m/l/O merge update).
 *  - "The signature-dish specialist: vLLM's attention backend" (blog.lo0.es),
 *    "How the backend reads the paged KV": the decode kernel gathers the
 *    physical blocks named by the block table; decode is bound by HBM
 *    bandwidth ("Why prefill and decode are opposite problems").
 *
 * Conventions for every call:
 *  - Memory: every pointer is DEVICE memory owned by the caller, 16-byte
 *    aligned, densely packed in the layout stated. The library never
 *    allocates per call and keeps no per-call state. One exception: the
 *    kf_decode_step calls (all four) also take pinned host memory that the GPU
 *    addresses directly (CUDA unified addressing, e.g. cudaHostAlloc) for
 *    their per-step inputs and outputs -- q, k_new, v_new, block_tables,
 *    context_lens_before, out and lse_out -- and read or write it in place over
 *    the host link; on GB300 (NVLink-C2C) that is faster for a step's small
 *    inputs and outputs than copying them. The caches, scales, workspace and
 *    extra partials stay device memory.
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and the call returns without synchronising.
 *  - Host errors: arguments that can be checked on the host are checked
 *    before anything is launched; a failing check returns KF_ERR_INVALID or
 *    KF_ERR_UNSUPPORTED and launches nothing. A failed launch returns
 *    KF_ERR_CUDA.
 *  - Device errors: values only the GPU sees (block-table entries, context
 *    lengths) are checked by the kernels. A bad value never causes an
 *    out-of-bounds access: the access is redirected or skipped, the output
 *    for that request is unspecified, and a bit is OR-ed into the current
 *    device's error word, read and cleared by kf_get_device_error().
 *  - Threads: calls may come from any host thread; the device error word is
 *    the only state shared between calls.
 *  - Layouts (bf16 = 16-bit brain float, f32 = IEEE single):
 *      q            bf16 [batch, num_q_heads, head_dim]
 *      k_cache      bf16 [num_blocks, block_size, num_kv_heads, head_dim]
 *      v_cache      bf16 [num_blocks, block_size, num_kv_heads, head_dim]
 *      block_tables int32 [batch, bt_stride]; entry (b, i) = physical block
 *                   holding tokens [i*block_size, (i+1)*block_size) of request b
 *      out_partial  f32 [num_splits, batch, num_q_heads, head_dim]
 *      lse_partial  f32 [num_splits, batch, num_q_heads]
 *    Query head h attends with KV head h / (num_q_heads / num_kv_heads).
 *  - Supported shapes: head_dim 64 or 128; block_size 16 or 32;
 *    num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 */
#ifndef KF_H
#define KF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *kf_stream_t;

typedef enum {
    KF_OK = 0,
    KF_ERR_INVALID = 1,     /* an argument failed a host-side check; nothing launched */
    KF_ERR_UNSUPPORTED = 2, /* valid but unsupported shape; nothing launched */
    KF_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    KF_ERR_DEVICE = 4       /* kf_get_device_error: a kernel recorded an error */
} kf_status;

typedef enum { KF_BF16 = 0, KF_F32 = 1 } kf_dtype;

/* Bits of the device error word. */
#define KF_DEVERR_BLOCK_ID    0x01u /* a block-table entry outside [0, num_blocks) */
#define KF_DEVERR_CONTEXT_LEN 0x02u /* a context length < 0 or above bt_stride*block_size */
#define KF_DEVERR_MAX_CONTEXT 0x04u /* a context length above max_context_len */
#define KF_DEVERR_APPEND_POS  0x08u /* an append position outside the block table */
#define KF_DEVERR_TIMEOUT     0x10u /* a pipeline wait in a kernel gave up */

/*
 * kf_append_kv -- write the step's new K/V row of every request into the cache.
 *
 * KernelFlume section 3.2: the tail attention node appends (K_new, V_new)
 * and then attends over the updated range. For each request b the new token
 * goes to position p = context_lens_before[b]: physical block
 * block_tables[b][p / block_size], slot p % block_size, all KV heads. The
 * copy is bit-exact; no other byte of the caches is written.
 *
 *   k_new, v_new         bf16 [batch, num_kv_heads, head_dim]
 *   k_cache, v_cache     bf16 [num_blocks, block_size, num_kv_heads, head_dim] (written)
 *   block_tables         int32 [batch, bt_stride]
 *   context_lens_before  int32 [batch], tokens cached before this step (not modified)
 *
 * Device errors: p outside [0, bt_stride*block_size) -> KF_DEVERR_APPEND_POS;
 * a block id outside [0, num_blocks) -> KF_DEVERR_BLOCK_ID; that request's row
 * is not written. batch == 0 is a no-op.
 */
kf_status kf_append_kv(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       const int32_t *block_tables, int bt_stride,
                       const int32_t *context_lens_before, int batch, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, kf_stream_t stream);

/*
 * kf_paged_decode_attention -- split-KV decode attention producing partials.
 *
 * KernelFlume sections 3.1-3.2 and 5.1 (local attention over a token range,
 * returning (o, m, l)); ultrainstinct.tech "Mathematical Formulation of
 * Chunked Attention". For request b with L_b = context_lens[b] tokens,
 * query head h (KV head h / G), and split s:
 *   n_max = ceil(max_context_len / block_size), c = max(1, ceil(n_max / num_splits)),
 *   the split covers tokens [s*c*block_size, min((s+1)*c*block_size, L_b)),
 *   s_t = scale * <q[b,h,:], K_t>,  m = max s_t,  l = sum_t e^{s_t - m},
 *   out_partial[s,b,h,:] = sum_t e^{s_t - m} V_t / l,  lse_partial[s,b,h] = m + ln l.
 * A split with no tokens writes out_partial = 0 and lse_partial = -inf.
 * Accumulation is fp32; K/V/q are read as bf16.
 *
 *   context_lens     int32 [batch], tokens to attend over (after any append);
 *                    0 is allowed (every split empty)
 *   max_context_len  host-side upper bound of context_lens (sets the chunk c)
 *   scale            softmax scale, e.g. 1/sqrt(head_dim)
 *   num_splits       >= 1; see kf_choose_num_splits. 0 is not "let the library
 *                    choose" here: the caller sizes out_partial and lse_partial,
 *                    so it fixes num_splits (kf_choose_num_splits gives the
 *                    library's plan; the step calls, whose partials are
 *                    internal, take 0 as their own schedule)
 *
 * A shard (a token-range partition held under its own block table, as on
 * KernelFlume's attention nodes) is one call with that shard's table and
 * shard-local lengths, writing its partials at out_partial + j*batch*num_q_heads*head_dim
 * and lse_partial + j*batch*num_q_heads; one kf_merge_partials over all slots
 * then gives the full result.
 *
 * Host errors: null pointers, batch < 0, num_splits < 1, bt_stride < 1,
 * num_blocks < 1, max_context_len < 0, a non-finite scale -> KF_ERR_INVALID;
 * unsupported head_dim, block_size or group -> KF_ERR_UNSUPPORTED.
 * Device errors: KF_DEVERR_BLOCK_ID, KF_DEVERR_CONTEXT_LEN, KF_DEVERR_MAX_CONTEXT
 * (tokens beyond the last split are then not attended).
 */
kf_status kf_paged_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int bt_stride,
                                    const int32_t *context_lens, int max_context_len, int batch,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int64_t num_blocks, float scale,
                                    int num_splits, float *out_partial, float *lse_partial,
                                    kf_stream_t stream);

/*
 * kf_paged_multiquery_attention -- paged attention of many query tokens per
 * request: chunked prefill and speculative verify (causal = 1) and the
 * shared-prefix pass of cascade attention (causal = 0).
 *
 * "Disaggregated Inference Architecture: Paged KV-Cache Tiering, Chunked
 * Prefill, and Asynchronous Overlap" (ultrainstinct.tech), "Mathematical
 * Formulation of Chunked Attention": a chunk's queries attend to earlier
 * chunks' keys in the paged cache without a mask and to their own chunk
 * causally. Request b owns query rows q_start[b] .. q_start[b+1]-1 (C_b of
 * them) of q, and its cache holds L_b = context_lens[b] tokens with the chunk
 * as the last C_b. Causal: query j (0-based in the chunk) attends tokens
 * [0, L_b - C_b + j]; non-causal: all L_b tokens. Cascade attention ("What
 * FlashInfer brings: JIT and cascade attention", blog.lo0.es) is one
 * non-causal call with batch = 1, the prefix's table and q_start = {0, B}
 * (every request's query), whose partials are merged by kf_merge_partials
 * with those of kf_paged_decode_attention over each request's own suffix.
 *
 *   q             bf16 [num_q_tokens, num_q_heads, head_dim]
 *   q_start       int32 [batch + 1] (device), ascending, q_start[batch] <= num_q_tokens
 *   context_lens  int32 [batch]; causal calls need C_b <= L_b
 *   max_context_len, max_query_len  host-side bounds of L_b and C_b
 *   out_partial   f32 [num_splits, num_q_tokens, num_q_heads, head_dim]
 *   lse_partial   f32 [num_splits, num_q_tokens, num_q_heads]
 * Splits follow kf_paged_decode_attention's rule, each clipped to its query's
 * limit; a (split, query) pair with no token gives (0, -inf). Rows of q not
 * covered by q_start are not written. Merge with kf_merge_partials(batch =
 * num_q_tokens). Accumulation fp32, inputs bf16.
 * Host errors: null pointers, negative sizes, causal not 0/1 -> KF_ERR_INVALID;
 * unsupported head_dim/block_size/group or batch * query tiles > 65535 ->
 * KF_ERR_UNSUPPORTED. Device errors: KF_DEVERR_BLOCK_ID, KF_DEVERR_CONTEXT_LEN
 * (length out of range, or C_b > L_b when causal), KF_DEVERR_MAX_CONTEXT
 * (L_b above max_context_len or C_b above max_query_len).
 */
kf_status kf_paged_multiquery_attention(const void *q, const int32_t *q_start, const void *k_cache,
                                        const void *v_cache, const int32_t *block_tables,
                                        int bt_stride, const int32_t *context_lens, int causal,
                                        int max_context_len, int max_query_len, int batch,
                                        int num_q_tokens, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int64_t num_blocks,
                                        float scale, int num_splits, float *out_partial,
                                        float *lse_partial, kf_stream_t stream);

/*
 * kf_choose_num_splits -- the split count the library would pick for a batch.
 *
 * A host-side plan (no device work): it models the decode kernel's schedule
 * on `device` (SM count, resident work units) and returns the num_splits in
 * [1, 1024] with the lowest modelled time of attention plus merge. If
 * context_lens_host (int32 [batch], host memory, nullable) is given it plans
 * for those lengths; otherwise it assumes every request has max_context_len
 * tokens. Returns a value < 1 on invalid arguments or a CUDA error.
 * The plan needs the head counts and head_dim (they fix the kernel's work
 * units and bytes per token) and, when given, every request's length (a
 * ragged batch plans differently from one of max_context_len throughout).
 */
int kf_choose_num_splits(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_context_len, const int32_t *context_lens_host,
                         int device);

/*
 * kf_choose_num_splits_fp8 -- the plan for the FP8-cache calls
 * (kf_paged_decode_attention_fp8, kf_decode_step_fp8) on a GPU with `num_sms`
 * SMs: same model with one-byte elements and the FP8 kernel's shape.
 */
int kf_choose_num_splits_fp8(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_context_len,
                             const int32_t *context_lens_host, int num_sms);

/*
 * kf_choose_num_splits_for -- the same plan for a GPU with `num_sms` SMs,
 * without touching any device (for planning on the host ahead of time).
 * The paged-decode pages give no split rule; this is the library's own
 * schedule model. Returns a value < 1 on invalid arguments.
 */
int kf_choose_num_splits_for(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_context_len,
                             const int32_t *context_lens_host, int num_sms);

/*
 * kf_merge_partials -- exact LSE merge of partial slots.
 *
 * ultrainstinct.tech "Mathematical Formulation of Chunked Attention"
 * (m_new = max(m_prev, m_cur); l and O rescaled by e^{m - m_new} and
 * summed), restated for normalised partials: for each (b, h),
 *   M = max_s lse_s,  w_s = e^{lse_s - M},
 *   out = sum_s w_s o_s / sum_s w_s,  lse_out = M + ln sum_s w_s.
 * A partial with lse = -inf has weight 0; if every partial of a row is
 * -inf, out = 0 and lse_out = -inf. KernelFlume section 5.1: the merge of
 * partials over a partition of the tokens equals attention over all of them.
 *
 *   out_partial  f32 [num_partials, batch, num_q_heads, head_dim]
 *   lse_partial  f32 [num_partials, batch, num_q_heads]
 *   out          [batch, num_q_heads, head_dim] of out_dtype (bf16 is
 *                rounded to nearest even)
 *   lse_out      f32 [batch, num_q_heads], or NULL
 *
 * Host errors: null pointers, num_partials < 1, batch < 0, num_q_heads < 1,
 * bad out_dtype -> KF_ERR_INVALID; head_dim not 64 or 128 -> KF_ERR_UNSUPPORTED.
 */
kf_status kf_merge_partials(const float *out_partial, const float *lse_partial,
                            int num_partials, int batch, int num_q_heads, int head_dim,
                            void *out, kf_dtype out_dtype, float *lse_out, kf_stream_t stream);

/*
 * kf_decode_step -- the whole decode step in one kernel launch: append,
 * split-KV attention and LSE merge.
 *
 * Same arithmetic as kf_append_kv, then kf_paged_decode_attention over
 * context_lens_before[b] + 1 tokens, then kf_merge_partials (KernelFlume
 * sections 3.2 and 5.1; ultrainstinct.tech "Mathematical Formulation of
 * Chunked Attention"), with the split rule of kf_paged_decode_attention and
 * c computed from max_context_len. Differences in what is written: the new
 * K/V row goes to the cache as in kf_append_kv; splits with no tokens write
 * nothing; partials of requests with more than one non-empty split live in
 * `workspace` and are merged there by the last work unit to finish; only
 * `out` and `lse_out` are results.
 *
 *   context_lens_before  int32 [batch], tokens cached before this step (>= 0)
 *   max_context_len      host-side upper bound of context_lens_before + 1
 *   num_splits           >= 1 (the split rule, c from max_context_len), or
 *                        KF_SPLITS_BALANCED (below)
 *   workspace            device scratch of kf_decode_step_workspace_size() bytes,
 *                        16-byte aligned, ZERO-FILLED before its first use; every
 *                        completed call leaves its counters at zero again. Calls
 *                        that share a workspace must not overlap on the GPU.
 *                        May be NULL when num_splits == 1.
 *   out                  [batch, num_q_heads, head_dim] of out_dtype
 *   lse_out              f32 [batch, num_q_heads], or NULL
 *
 * num_splits = KF_SPLITS_BALANCED (0) replaces the split rule by a balanced
 * partition of the same tokens (same result up to fp32 rounding order; the
 * exact merge of KernelFlume section 5.1 holds for any partition): the
 * 16-token stages of all requests, laid end to end in request order, are cut
 * into P equal runs, one per CTA, where P x ceil(num_kv_heads / H) is the
 * number of CTAs the GPU holds at once (H = KV heads per CTA, chosen by the
 * library); a run may span several requests. Every CTA then does the same
 * work, so the step takes one even wave whatever the batch's length mix. It
 * always needs the workspace, of kf_decode_step_workspace_size(..., 0) bytes
 * on the current device.
 *
 * Host errors as kf_paged_decode_attention, plus: num_splits < 0; a missing or
 * short workspace with num_splits > 1 or num_splits == 0 -> KF_ERR_INVALID;
 * num_splits too large for the merge to fit in the kernel's shared memory ->
 * KF_ERR_UNSUPPORTED.
 * Device errors: KF_DEVERR_BLOCK_ID, KF_DEVERR_CONTEXT_LEN (negative length),
 * KF_DEVERR_APPEND_POS (no room in the table), KF_DEVERR_MAX_CONTEXT.
 */
#define KF_SPLITS_BALANCED 0

/*
 * kf_decode_step_workspace_size -- workspace bytes of the kf_decode_step
 * calls (bf16 and FP8 caches alike). num_splits >= 1: partials
 * [num_splits, batch, num_q_heads] of head_dim + 1 floats and [batch,
 * num_kv_heads] counters. num_splits == KF_SPLITS_BALANCED: partial slots of
 * [num_q_heads, head_dim + 1] floats, two per CTA of the largest one-wave grid
 * on the CURRENT device plus one per request, and the counters; 0 if that
 * device cannot be queried or the arguments are invalid.
 */
size_t kf_decode_step_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                     int num_splits);

kf_status kf_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int32_t *block_tables, int bt_stride,
                         const int32_t *context_lens_before, int max_context_len, int batch,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, float scale, int num_splits, void *workspace,
                         size_t workspace_bytes, void *out, kf_dtype out_dtype, float *lse_out,
                         kf_stream_t stream);

/*
 * kf_decode_step_merge_partials -- kf_decode_step whose final LSE merge also
 * takes num_extra partials computed elsewhere: the one-launch form of the
 * suffix step of cascade attention ("What FlashInfer brings: JIT and cascade
 * attention", blog.lo0.es), where the extra partials are those of the shared
 * prefix (kf_paged_multiquery_attention, causal = 0, batch = 1) and the
 * block tables are each request's own blocks after the prefix. The merge is
 * the exact one of kf_merge_partials ("Mathematical Formulation of Chunked
 * Attention", ultrainstinct.tech; KernelFlume section 5.1) over this step's
 * non-empty splits and the extra slots together, so the result equals
 * attention over the tokens of both.
 *
 *   extra_out_partial  f32 [num_extra, batch, num_q_heads, head_dim], 16-byte aligned
 *   extra_lse_partial  f32 [num_extra, batch, num_q_heads]; -inf marks an empty
 *                      slot (its o may hold any bits: it is ignored)
 *   num_extra          >= 0; 0 is kf_decode_step
 *   workspace          as kf_decode_step, and required whenever num_extra > 0
 *                      (the merge counts its work units there even at num_splits = 1)
 * Everything else, and the error behaviour, as kf_decode_step, plus:
 * num_extra < 0, or num_extra > 0 with a null or misaligned extra pointer ->
 * KF_ERR_INVALID; num_splits + num_extra too large for the merge to fit in
 * the kernel's shared memory -> KF_ERR_UNSUPPORTED (the balanced schedule,
 * num_splits = KF_SPLITS_BALANCED, merges in registers and has no such
 * limit). The extra partials must be complete when the call runs (e.g.
 * written earlier on the same stream).
 */
kf_status kf_decode_step_merge_partials(const void *q, const void *k_new, const void *v_new,
                                        void *k_cache, void *v_cache, const int32_t *block_tables,
                                        int bt_stride, const int32_t *context_lens_before,
                                        int max_context_len, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int64_t num_blocks, float scale, int num_splits,
                                        const float *extra_out_partial,
                                        const float *extra_lse_partial, int num_extra,
                                        void *workspace, size_t workspace_bytes, void *out,
                                        kf_dtype out_dtype, float *lse_out, kf_stream_t stream);

/*
 * FP8 (E4M3) KV cache: kf_append_kv_fp8, kf_paged_decode_attention_fp8,
 * kf_decode_step_fp8.
 *
 * The decode posts of blog.lo0.es ("Quantised KV cache -- --kv-cache-dtype
 * fp8") keep K/V in 8-bit floats with scales, halving the bytes a decode step
 * reads. Here k_cache/v_cache hold OCP FP8 E4M3 codes (1 byte per element,
 * same [num_blocks, block_size, num_kv_heads, head_dim] layout) and
 * k_scale/v_scale are fp32 [num_kv_heads] device arrays: element value =
 * e4m3(code) * scale of its KV head. The calls take the same arguments as
 * their bf16 counterparts plus the two scale arrays and compute the same
 * thing on the dequantised values; q, k_new and v_new stay bf16. The append
 * (and the fused step's append) stores code = E4M3 round-to-nearest-even,
 * saturating to +-448, of the fp32 quotient float(x) / scale. The decode
 * kernel widens the codes to bf16 exactly and accumulates in fp32.
 * Host errors as the bf16 calls, plus null scales -> KF_ERR_INVALID.
 */
kf_status kf_append_kv_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           const float *k_scale, const float *v_scale, const int32_t *block_tables,
                           int bt_stride, const int32_t *context_lens_before, int batch,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           kf_stream_t stream);

kf_status kf_paged_decode_attention_fp8(const void *q, const void *k_cache, const void *v_cache,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *block_tables, int bt_stride,
                                        const int32_t *context_lens, int max_context_len,
                                        int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int64_t num_blocks,
                                        float scale, int num_splits, float *out_partial,
                                        float *lse_partial, kf_stream_t stream);

kf_status kf_decode_step_fp8(const void *q, const void *k_new, const void *v_new, void *k_cache,
                             void *v_cache, const float *k_scale, const float *v_scale,
                             const int32_t *block_tables, int bt_stride,
                             const int32_t *context_lens_before, int max_context_len, int batch,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, float scale, int num_splits, void *workspace,
                             size_t workspace_bytes, void *out, kf_dtype out_dtype,
                             float *lse_out, kf_stream_t stream);

/*
 * kf_decode_step_static -- kf_decode_step without a caller-provided workspace,
 * for callers that may not allocate device memory.
 *
 * The paged-decode pages have no counterpart to this call; it exists for
 * users of this library whose device memory is reserved up front by their
 * own pool allocator, plugin hosts that pass a library only the buffers of
 * each call, and decode loops that cannot afford cudaMalloc's implicit device
 * synchronisation. It computes exactly what kf_decode_step computes (same
 * arguments, minus the workspace), and allocates nothing: its scratch is a
 * KF_STATIC_SCRATCH_BYTES array in the library's own device memory, which
 * every GPU that loads the library keeps until the process exits.
 *
 * Limits and behaviour:
 *  - Calls whose kf_decode_step_workspace_size(...) exceeds
 *    KF_STATIC_SCRATCH_BYTES return KF_ERR_UNSUPPORTED (use kf_decode_step with
 *    your own workspace, or fewer splits).
 *  - Shapes the step does not support, bad arguments and a device that cannot
 *    be queried give the same status as kf_decode_step with a workspace.
 *  - The first call on a device looks up the array's device address (a
 *    one-time set-up on that device, repeated in a new context of the device,
 *    e.g. after cudaDeviceReset, because the array may then sit elsewhere);
 *    make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents; each call clears the part that must start at zero (the
 *    merge counters) on its own stream, after every argument check, so a
 *    refused call queues no work. Calls that overlap on the GPU (on different
 *    streams, or from different threads) race on the array and give wrong
 *    results: serialise them.
 */
#define KF_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

kf_status kf_decode_step_static(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                void *v_cache, const int32_t *block_tables, int bt_stride,
                                const int32_t *context_lens_before, int max_context_len, int batch,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, float scale, int num_splits, void *out,
                                kf_dtype out_dtype, float *lse_out, kf_stream_t stream);

/*
 * kf_get_device_error -- read and clear the current device's error word.
 *
 * Synchronises `stream`, copies the word (KF_DEVERR_* bits) to *flags and
 * resets it to 0. Returns KF_OK if no bit was set, KF_ERR_DEVICE if some
 * bit was, KF_ERR_CUDA if a CUDA call failed, KF_ERR_INVALID if flags is NULL.
 * One status covers every kind of device error (a bad block id, a length out
 * of range, a wait that gave up); the bits in *flags say which occurred.
 */
kf_status kf_get_device_error(unsigned int *flags, kf_stream_t stream);

/*
 * kf_check_bounded_wait -- exercise the timeout path of the kernels' waits.
 *
 * The TMA-fed kernels wait on shared-memory mbarriers, each wait bounded: a
 * wait that gives up sets KF_DEVERR_TIMEOUT in the error word and the kernel
 * returns instead of hanging. This call launches one block that waits, with
 * the same bounded wait at a short limit (2^16 polls, milliseconds), on a
 * barrier that nothing completes, so it always sets KF_DEVERR_TIMEOUT; a
 * following kf_get_device_error reports it, and the context stays usable.
 * Returns KF_ERR_CUDA if the launch fails.
 */
kf_status kf_check_bounded_wait(kf_stream_t stream);

/* Static description of a status code. */
const char *kf_status_string(kf_status s);

/* Library version, major*10000 + minor*100 + patch. */
int kf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KF_H */
