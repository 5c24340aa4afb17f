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

}  // namespace

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
