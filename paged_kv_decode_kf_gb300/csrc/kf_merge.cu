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
// Mapping: D/4 threads per (b, h) row, each owning 4 consecutive outputs, so
// every partial row is read as coalesced 16-byte vectors; the lse column is
// read once per thread (the reads of one row hit the same line).
#include <math.h>

#include "kf_internal.cuh"

namespace kf {
namespace {

template <int D>
__global__ void __launch_bounds__(128)
merge_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part, int S,
             int64_t rows, void *__restrict__ out, int out_dtype, float *__restrict__ lse_out) {
    constexpr int TPR = D / 4;  // threads per row
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / TPR) + threadIdx.x / TPR;
    const int c = threadIdx.x % TPR;
    if (row >= rows) return;

    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, lse_part[(int64_t)s * rows + row]);

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < S; ++s) {
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
    const int threads = 128;
    if (head_dim == 128) {
        const int64_t rpb = threads / 32;
        merge_kernel<128><<<(unsigned)((rows + rpb - 1) / rpb), threads, 0, stream>>>(
            out_partial, lse_partial, num_partials, rows, out, out_dtype, lse_out);
    } else {
        const int64_t rpb = threads / 16;
        merge_kernel<64><<<(unsigned)((rows + rpb - 1) / rpb), threads, 0, stream>>>(
            out_partial, lse_partial, num_partials, rows, out, out_dtype, lse_out);
    }
    return cudaGetLastError();
}

}  // namespace kf
