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
// Mapping: one warp per (b, h) row, 8 rows per CTA, no block-level
// synchronisation. Lane k loads lse of partials k, k + 32, ... once (kept in
// registers for up to 64 partials); a shuffle reduction gives M; each lane
// turns its lse into a weight, and the weights of 32 partials at a time are
// broadcast by shuffles while the lanes load the non-empty partials' o rows
// (16-byte vectors at D = 128, 8 at D = 64), sixteen partials in flight: a
// merge of up to 16 partials is two dependent memory round trips. An empty
// partial (lse = -inf) has weight 0 and its o is not read.
#include <math.h>

#include "kf_internal.cuh"

namespace kf {
namespace {

constexpr int kRowsPerCta = 8;
constexpr int kInFlight = 16;  // partials loaded together

template <int D>
struct MergeVec;
template <>
struct MergeVec<128> {
    using T = float4;
    static __device__ __forceinline__ void fma(float w, const T &o, T &a) {
        a.x = fmaf(w, o.x, a.x); a.y = fmaf(w, o.y, a.y); a.z = fmaf(w, o.z, a.z); a.w = fmaf(w, o.w, a.w);
    }
    static __device__ __forceinline__ T zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct MergeVec<64> {
    using T = float2;
    static __device__ __forceinline__ void fma(float w, const T &o, T &a) {
        a.x = fmaf(w, o.x, a.x); a.y = fmaf(w, o.y, a.y);
    }
    static __device__ __forceinline__ T zero() { return make_float2(0.f, 0.f); }
};

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerCta)
merge_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part, int S,
             int64_t rows, void *__restrict__ out, int out_dtype, float *__restrict__ lse_out) {
    using MV = MergeVec<D>;
    using T = typename MV::T;
    constexpr int V = D / 32;  // floats per lane
    const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;

    if (S == 1) {
        // one partial: the merge is the identity (w = 1); lse and o load together
        const float l = __ldg(lse_part + row);
        T o = __ldg(reinterpret_cast<const T *>(o_part + row * D) + lane);
        if (l == -INFINITY) o = MV::zero();
        const float *a = reinterpret_cast<const float *>(&o);
        if (out_dtype == KF_F32) {
            reinterpret_cast<T *>(static_cast<float *>(out) + row * D)[lane] = o;
        } else {
            uint16_t *o16 = static_cast<uint16_t *>(out) + row * D + V * lane;
#pragma unroll
            for (int i = 0; i < V; i += 2)
                *reinterpret_cast<__nv_bfloat162 *>(o16 + i) = __floats2bfloat162_rn(a[i], a[i + 1]);
        }
        if (lse_out != nullptr && lane == 0) lse_out[row] = l;
        return;
    }

    // 1. M = max_s lse_s (the first 64 partials' lse stay in registers)
    const float l0 = lane < S ? __ldg(lse_part + (int64_t)lane * rows + row) : -INFINITY;
    const float l1 = lane + 32 < S ? __ldg(lse_part + (int64_t)(lane + 32) * rows + row) : -INFINITY;
    float M = fmaxf(l0, l1);
    for (int s = lane + 64; s < S; s += 32) M = fmaxf(M, __ldg(lse_part + (int64_t)s * rows + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    // 2. sum_s w_s o_s and sum_s w_s, w_s = e^{lse_s - M}
    T acc = MV::zero();
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int c0 = 0; c0 < S; c0 += 32) {
            const int sl = c0 + lane;
            const float l = c0 == 0 ? l0 : c0 == 32 ? l1 : (sl < S ? __ldg(lse_part + (int64_t)sl * rows + row) : -INFINITY);
            const float w = l == -INFINITY ? 0.f : expf(l - M);
            wsum += w;
            const int n = S - c0 < 32 ? S - c0 : 32;
            for (int u0 = 0; u0 < n; u0 += kInFlight) {
                T o[kInFlight];
                float wu[kInFlight];
#pragma unroll
                for (int u = 0; u < kInFlight; ++u) {
                    wu[u] = __shfl_sync(0xffffffffu, w, (u0 + u) & 31);
                    if (u0 + u >= n) wu[u] = 0.f;
                    o[u] = wu[u] != 0.f
                               ? __ldg(reinterpret_cast<const T *>(o_part + ((int64_t)(c0 + u0 + u) * rows + row) * D) + lane)
                               : MV::zero();
                }
#pragma unroll
                for (int u = 0; u < kInFlight; ++u) MV::fma(wu[u], o[u], acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
        const float inv = 1.f / wsum;
        float *a = reinterpret_cast<float *>(&acc);
#pragma unroll
        for (int i = 0; i < V; ++i) a[i] *= inv;
    }

    // 3. write
    const float *a = reinterpret_cast<const float *>(&acc);
    if (out_dtype == KF_F32) {
        reinterpret_cast<T *>(static_cast<float *>(out) + row * D)[lane] = acc;
    } else {
        uint16_t *o16 = static_cast<uint16_t *>(out) + row * D + V * lane;
#pragma unroll
        for (int i = 0; i < V; i += 2) {
            __nv_bfloat162 v = __floats2bfloat162_rn(a[i], a[i + 1]);
            *reinterpret_cast<__nv_bfloat162 *>(o16 + i) = v;
        }
    }
    if (lse_out != nullptr && lane == 0) lse_out[row] = (M == -INFINITY) ? -INFINITY : M + logf(wsum);
}

}  // namespace

cudaError_t launch_merge(const float *out_partial, const float *lse_partial, int num_partials,
                         int batch, int num_q_heads, int head_dim, void *out, int out_dtype,
                         float *lse_out, cudaStream_t stream) {
    const int64_t rows = (int64_t)batch * num_q_heads;
    if (rows == 0) return cudaSuccess;
    const int64_t ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
    if (head_dim == 128)
        merge_kernel<128><<<(unsigned)ctas, 32 * kRowsPerCta, 0, stream>>>(out_partial, lse_partial, num_partials,
                                                                         rows, out, out_dtype, lse_out);
    else
        merge_kernel<64><<<(unsigned)ctas, 32 * kRowsPerCta, 0, stream>>>(out_partial, lse_partial, num_partials,
                                                                        rows, out, out_dtype, lse_out);
    return cudaGetLastError();
}

}  // namespace kf
