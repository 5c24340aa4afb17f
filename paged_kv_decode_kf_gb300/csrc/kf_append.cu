// kf_append.cu -- the step's K/V append into the paged cache.
//
// KernelFlume (academ.us/article/2606.29207), section 3.2: the tail node
// appends (K_new, V_new) to its partition before attending. Request b's new
// row goes to position p = ctx_before[b]: block block_tables[b][p / bs],
// slot p % bs. The row of one token is num_kv_heads*head_dim contiguous bf16
// values in the [num_blocks, bs, Hkv, D] layout, so the copy is a run of
// 16-byte vectors, one CTA per request.
#include "kf_internal.cuh"

namespace kf {
namespace {

__global__ void __launch_bounds__(128)
append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
              uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
              const int32_t *__restrict__ block_tables, int bt_stride,
              const int32_t *__restrict__ ctx_before, int row_vecs, int block_size,
              int64_t num_blocks, unsigned int *err) {
    const int b = blockIdx.x;
    const int64_t pos = ctx_before[b];
    if (pos < 0 || pos >= (int64_t)bt_stride * block_size) {
        if (threadIdx.x == 0) raise_error(err, KF_DEVERR_APPEND_POS);
        return;
    }
    const int64_t phys = block_tables[(int64_t)b * bt_stride + pos / block_size];
    if (phys < 0 || phys >= num_blocks) {
        if (threadIdx.x == 0) raise_error(err, KF_DEVERR_BLOCK_ID);
        return;
    }
    const int64_t dst = (phys * block_size + pos % block_size) * row_vecs;
    const int64_t src = (int64_t)b * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        k_cache[dst + i] = k_new[src + i];
        v_cache[dst + i] = v_new[src + i];
    }
}

// FP8 cache: each thread quantises 16 elements (two 16-byte bf16 vectors) of
// its KV head to E4M3 codes of x / scale (fp32 division, round to nearest
// even, saturating to +-448), one 16-byte store.
__global__ void __launch_bounds__(128)
append_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                  uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                  const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                  const int32_t *__restrict__ block_tables, int bt_stride,
                  const int32_t *__restrict__ ctx_before, int row_chunks, int head_chunks,
                  int block_size, int64_t num_blocks, unsigned int *err) {
    const int b = blockIdx.x;
    const int64_t pos = ctx_before[b];
    if (pos < 0 || pos >= (int64_t)bt_stride * block_size) {
        if (threadIdx.x == 0) raise_error(err, KF_DEVERR_APPEND_POS);
        return;
    }
    const int64_t phys = block_tables[(int64_t)b * bt_stride + pos / block_size];
    if (phys < 0 || phys >= num_blocks) {
        if (threadIdx.x == 0) raise_error(err, KF_DEVERR_BLOCK_ID);
        return;
    }
    const int64_t dst = (phys * block_size + pos % block_size) * row_chunks;
    const int64_t src = (int64_t)b * row_chunks * 2;
    for (int i = threadIdx.x; i < 2 * row_chunks; i += blockDim.x) {
        const bool is_v = i >= row_chunks;
        const int c = is_v ? i - row_chunks : i;
        const float s = (is_v ? v_scale : k_scale)[c / head_chunks];
        const uint4 *in = (is_v ? v_new : k_new) + src + 2 * c;
        const uint4 x0 = in[0], x1 = in[1];
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            unsigned short lo, hi;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo)
                : "f"(bf16_hi(w[2 * e]) / s), "f"(bf16_lo(w[2 * e]) / s));
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi)
                : "f"(bf16_hi(w[2 * e + 1]) / s), "f"(bf16_lo(w[2 * e + 1]) / s));
            o[e] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        (is_v ? v_cache : k_cache)[dst + c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_append_fp8(const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_cache,
                              uint8_t *v_cache, const float *k_scale, const float *v_scale,
                              const int32_t *block_tables, int bt_stride, const int32_t *ctx_before,
                              int batch, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, unsigned int *err, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    const int row_chunks = num_kv_heads * head_dim / 16;  // 16-code vectors per token row
    const int threads = 2 * row_chunks < 128 ? ((2 * row_chunks + 31) / 32) * 32 : 128;
    append_fp8_kernel<<<batch, threads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
        reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), k_scale, v_scale,
        block_tables, bt_stride, ctx_before, row_chunks, head_dim / 16, block_size, num_blocks, err);
    return cudaGetLastError();
}

cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                          uint16_t *v_cache, const int32_t *block_tables, int bt_stride,
                          const int32_t *ctx_before, int batch, int num_kv_heads, int head_dim,
                          int block_size, int64_t num_blocks, unsigned int *err,
                          cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    const int row_vecs = num_kv_heads * head_dim / 8;  // 16-byte vectors per token row
    const int threads = row_vecs < 128 ? ((row_vecs + 31) / 32) * 32 : 128;
    append_kernel<<<batch, threads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
        reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), block_tables,
        bt_stride, ctx_before, row_vecs, block_size, num_blocks, err);
    return cudaGetLastError();
}

}  // namespace kf
