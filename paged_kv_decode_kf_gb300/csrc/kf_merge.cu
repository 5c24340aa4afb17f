// kf_merge.cu -- exact LSE merge of split/shard partials.
//
// "Disaggregated Inference Architecture: Paged KV-Cache Tiering, Chunked
// Prefill, and Asynchronous Overlap" (ultrainstinct.tech), "Mathematical
// Formulation of Chunked Attention": m_new = max(m_prev, m_cur) and l, O
// rescaled by e^{m - m_new} and summed. With normalised partials
// (o_s, lse_s = m_s + ln l_s) this is, per (b, h):
//   M = max_s lse_s, w_s = e^{lse_s - M}, out = sum w_s o_s / sum w_s,
//   lse = M + ln(sum w_s).
// KernelFlume (academ.us/article/2606.29207) section 5.1: merging the
// partials of a partition of the tokens equals attention over all of them.
//
// Mapping: one CTA per (b, h) row; P groups of D/4 threads each take every
// P-th partial (so S partials are read P at a time, coalesced 16-byte vectors,
// 4 loads in flight per thread), then the groups' sums are combined in shared
// memory. The row max M is found first by all threads striding over the S
// lse values.
#include <math.h>

#include "kf_internal.cuh"

namespace kf {
namespace {

constexpr int kGroups = 8;  // partial groups per row

template <int D>
__global__ void __launch_bounds__(kGroups *(D / 4))
merge_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part, int S,
             int64_t rows, void *__restrict__ out, int out_dtype, float *__restrict__ lse_out) {
    constexpr int TPR = D / 4;  // threads per group: 4 outputs each
    const int64_t row = blockIdx.x;
    const int c = threadIdx.x % TPR, grp = threadIdx.x / TPR;

    __shared__ float sm_red[kGroups * TPR / 32 + 1];
    __shared__ __align__(16) float4 sm_acc[kGroups][TPR];
    __shared__ float sm_w[kGroups];

    // 1. M = max_s lse_s
    float M = -INFINITY;
    for (int s = threadIdx.x; s < S; s += blockDim.x) M = fmaxf(M, lse_part[(int64_t)s * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if ((threadIdx.x & 31) == 0) sm_red[threadIdx.x >> 5] = M;
    __syncthreads();
    M = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) M = fmaxf(M, sm_red[i]);

    // 2. this group's share of sum_s w_s o_s and sum_s w_s
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll 4
        for (int s = grp; s < S; s += kGroups) {
            const float l = lse_part[(int64_t)s * rows + row];
            if (l == -INFINITY) continue;  // empty partial: weight 0, o not read
            const float w = expf(l - M);
            const float4 o = reinterpret_cast<const float4 *>(o_part + ((int64_t)s * rows + row) * D)[c];
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
            wsum += w;
        }
    }
    sm_acc[grp][c] = acc;
    if (c == 0) sm_w[grp] = wsum;
    __syncthreads();
    if (grp != 0) return;

    // 3. combine the groups and write
    wsum = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        const float4 a = sm_acc[g][c];
        acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
        wsum += sm_w[g];
    }
    if (M != -INFINITY) {
        const float inv = 1.f / wsum;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    }
    if (out_dtype == KF_F32) {
        reinterpret_cast<float4 *>(static_cast<float *>(out) + row * D)[c] = acc;
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t *>(&lo);
        v.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + row * D)[c] = v;
    }
    if (lse_out != nullptr && c == 0) lse_out[row] = (M == -INFINITY) ? -INFINITY : M + logf(wsum);
}

}  // namespace

cudaError_t launch_merge(const float *out_partial, const float *lse_partial, int num_partials,
                         int batch, int num_q_heads, int head_dim, void *out, int out_dtype,
                         float *lse_out, cudaStream_t stream) {
    const int64_t rows = (int64_t)batch * num_q_heads;
    if (rows == 0) return cudaSuccess;
    if (rows > 0x7fffffff) return cudaErrorInvalidValue;
    if (head_dim == 128)
        merge_kernel<128><<<(unsigned)rows, kGroups * 32, 0, stream>>>(
            out_partial, lse_partial, num_partials, rows, out, out_dtype, lse_out);
    else
        merge_kernel<64><<<(unsigned)rows, kGroups * 16, 0, stream>>>(
            out_partial, lse_partial, num_partials, rows, out, out_dtype, lse_out);
    return cudaGetLastError();
}

}  // namespace kf
