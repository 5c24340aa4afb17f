// kf_internal.cuh -- declarations shared by the library's translation units.
//
// Internal only: the public surface is include/kf.h. Everything here is
// device-side helpers and the launch functions the C-ABI layer calls after
// it has validated the arguments on the host.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kf.h"

namespace kf {

// Parameters of one decode-attention launch (already validated).
struct DecodeParams {
    const uint16_t *q;        // bf16 [B, Hq, D]
    const uint16_t *k_cache;  // bf16 [NB, bs, Hkv, D]
    const uint16_t *v_cache;
    const int32_t *block_tables;
    const int32_t *ctx_lens;
    float *out_partial;       // f32 [S, B, Hq, D]
    float *lse_partial;       // f32 [S, B, Hq]
    unsigned int *err;        // device error word
    int64_t num_blocks;
    int bt_stride;
    int max_context_len;
    int batch, num_q_heads, num_kv_heads, head_dim, block_size;
    int num_splits;
    int chunk_blocks;         // blocks per split: max(1, ceil(ceil(max_ctx/bs)/S))
    float scale_log2;         // scale * log2(e)
    const float *k_scale;     // FP8 caches: per-KV-head dequantisation scales, else null
    const float *v_scale;
};

// Extra arguments of the single-launch decode step (append + attention + merge).
struct StepArgs {
    const uint16_t *k_new;   // bf16 [B, Hkv, D]
    const uint16_t *v_new;
    void *k_cache;           // written at each request's new position (bf16 or E4M3)
    void *v_cache;
    float *ws_o;             // workspace partials [S, B, Hq, D]
    float *ws_lse;           // workspace lse [S, B, Hq]
    unsigned int *counters;  // workspace [B, Hkv], zero between steps
    void *out;               // [B, Hq, D] of out_dtype
    float *lse_out;          // [B, Hq] or null
    int out_dtype;
    const float *ex_o;       // extra partials merged in: [n_ex, B, Hq, D] (or null)
    const float *ex_lse;     //                           [n_ex, B, Hq]
    int n_ex;
};

// Parameters of one multi-query (chunked prefill / shared prefix) launch.
struct MqParams {
    const uint16_t *q;          // bf16 [num_q_tokens, Hq, D]
    const int32_t *q_start;     // [batch + 1]
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    const int32_t *block_tables;
    const int32_t *ctx_lens;    // [batch], tokens in the cache including the chunk
    float *out_partial;         // f32 [S, num_q_tokens, Hq, D]
    float *lse_partial;         // f32 [S, num_q_tokens, Hq]
    unsigned int *err;
    int64_t num_blocks;
    int bt_stride;
    int max_context_len, max_query_len;
    int batch, num_q_tokens, num_q_heads, num_kv_heads, head_dim, block_size;
    int num_splits, chunk_blocks, causal, q_tiles;
    float scale_log2;
};

cudaError_t launch_multiquery(MqParams p, cudaStream_t stream, void *encode_fn);
// tcgen05 version (128-row query tiles, TMEM accumulators); same contract.
cudaError_t launch_multiquery_tc05(MqParams p, cudaStream_t stream, void *encode_fn);
// tcgen05, 128-token KV tiles and two query tiles per CTA (> 128 rows per KV head).
cudaError_t launch_multiquery_tc05w(MqParams p, cudaStream_t stream, void *encode_fn);
// tcgen05 on CTA pairs (cta_group::2, M = 256 across two SMs), head_dim 128.
cudaError_t launch_multiquery_tc05p(MqParams p, cudaStream_t stream, void *encode_fn);

// Decode kernels, one per implementation. Each returns the launch status.
cudaError_t launch_decode_simt(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream, void *encode_fn);
cudaError_t launch_decode_step_tc(const DecodeParams &p, const StepArgs &a, cudaStream_t stream,
                                  void *encode_fn);
cudaError_t launch_decode_tc_fp8(const DecodeParams &p, cudaStream_t stream, void *encode_fn);
cudaError_t launch_decode_step_tc_fp8(const DecodeParams &p, const StepArgs &a, cudaStream_t stream,
                                      void *encode_fn);
// The decode step on the balanced schedule: `ctas` CTAs per KV-head group,
// one wave (see kf_decode_bal.cuh); StepArgs' workspace pointers hold its
// layout. *_resident: CTAs of that kernel one SM holds for this shape.
cudaError_t decode_bal_resident(int head_dim, int num_q_heads, int num_kv_heads, int *resident);
cudaError_t decode_bal_resident_fp8(int head_dim, int num_q_heads, int num_kv_heads, int *resident);
cudaError_t launch_decode_step_bal(const DecodeParams &p, const StepArgs &a, int ctas, cudaStream_t stream,
                                   void *encode_fn);
cudaError_t launch_decode_step_bal_fp8(const DecodeParams &p, const StepArgs &a, int ctas,
                                       cudaStream_t stream, void *encode_fn);
// One bounded wait that nothing completes (sets KF_DEVERR_TIMEOUT).
cudaError_t launch_wait_check(unsigned int *err, cudaStream_t stream);

// Process-unique id of the CUDA context current on the calling thread (0 if
// none): device addresses looked up in one context are stale in the next.
unsigned long long current_context_id();

// kf_decode_step that clears its workspace's merge counters on `stream` after
// every argument check, right before the launch.
kf_status decode_step_clearing_counters(const void *q, const void *k_new, const void *v_new,
                                        void *k_cache, void *v_cache, const int32_t *block_tables,
                                        int bt_stride, const int32_t *context_lens_before,
                                        int max_context_len, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int64_t num_blocks, float scale, int num_splits,
                                        void *workspace, size_t workspace_bytes, void *out,
                                        kf_dtype out_dtype, float *lse_out, kf_stream_t stream);
// Bytes of the tensor-core kernel's shared-memory ring (the fused merge reuses it).
int decode_tc_ring_bytes(int num_kv_heads, int head_dim, bool kv8);
// Largest number of resident CTAs per SM and KV heads per CTA the tensor-core
// kernel uses for this shape (for the split planner).
void decode_tc_shape(int num_kv_heads, int head_dim, int block_size, bool kv8, int *heads_per_cta,
                     int *ctas_per_sm);

cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                          uint16_t *v_cache, const int32_t *block_tables, int bt_stride,
                          const int32_t *ctx_before, int batch, int num_kv_heads, int head_dim,
                          int block_size, int64_t num_blocks, unsigned int *err,
                          cudaStream_t stream);

cudaError_t launch_append_fp8(const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_cache,
                              uint8_t *v_cache, const float *k_scale, const float *v_scale,
                              const int32_t *block_tables, int bt_stride, const int32_t *ctx_before,
                              int batch, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, unsigned int *err, cudaStream_t stream);

cudaError_t launch_merge(const float *out_partial, const float *lse_partial, int num_partials,
                         int batch, int num_q_heads, int head_dim, void *out, int out_dtype,
                         float *lse_out, cudaStream_t stream);

// Which decode kernel a call uses: 0 = tensor-core (default), 1 = CUDA-core.
int decode_impl();

// --------------------------------------------------------------------------
// Device helpers
// --------------------------------------------------------------------------

__device__ __forceinline__ void raise_error(unsigned int *err, unsigned int bit) {
    atomicOr(err, bit);
}

// The two bf16 halves of a 32-bit word as fp32 (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Validated context length and the token range of split `s`.
struct SplitRange {
    int64_t t_begin, t_end;
};

__device__ __forceinline__ SplitRange split_range(const DecodeParams &p, int b, int s,
                                                  bool report) {
    int64_t L = p.ctx_lens[b];
    const int64_t cap = (int64_t)p.bt_stride * p.block_size;
    if (L < 0 || L > cap) {
        if (report) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        L = L < 0 ? 0 : cap;
    }
    if (L > p.max_context_len && report) raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
    const int64_t span = (int64_t)p.chunk_blocks * p.block_size;
    int64_t lo = (int64_t)s * span;
    int64_t hi = lo + span;
    if (lo > L) lo = L;
    if (hi > L) hi = L;
    return {lo, hi};
}

// Physical block of logical block `lb` of request b, redirected to block 0
// (and reported) if the table entry is out of range.
// log2 of a power-of-two block size (every supported size is one): hot loops
// shift and mask instead of dividing a 64-bit token index.
__device__ __forceinline__ int block_shift(int block_size) { return 31 - __clz(block_size); }

__device__ __forceinline__ int64_t physical_block(const DecodeParams &p, int b, int64_t lb) {
    int64_t phys = p.block_tables[(int64_t)b * p.bt_stride + lb];
    if (phys < 0 || phys >= p.num_blocks) {
        raise_error(p.err, KF_DEVERR_BLOCK_ID);
        phys = 0;
    }
    return phys;
}

}  // namespace kf
