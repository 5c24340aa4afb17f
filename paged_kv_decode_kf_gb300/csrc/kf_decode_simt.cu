// kf_decode_simt.cu -- split-KV paged decode attention on the CUDA cores.
//
// The plain CUDA-core formulation, kept beside the tensor-core kernel as the
// measured alternative. What it computes (KernelFlume,
// academ.us/article/2606.29207, sections 3.1-3.2: local attention of the
// decode query over a token-range partition returning (o, m, l); the online
// softmax update of "Disaggregated Inference Architecture: Paged KV-Cache
// Tiering, Chunked Prefill, and Asynchronous Overlap", ultrainstinct.tech,
// "Mathematical Formulation of Chunked Attention"): for one split of one
// request and the G query heads of one KV head, o = softmax(q K^T scale) V
// over the split's tokens, written with lse = m + ln l.
//
// Mapping: one CTA per (split, KV head, request), 4 warps. The split's
// tokens are walked in 16-token sub-blocks (a block, or half a 32-token
// block), sub-block j by warp j % 4. In a warp, D/8 lanes hold one token row
// as 16-byte vectors (two or four tokens per pass); every K and V row of the
// sub-block is loaded with 128-bit read-only loads before any arithmetic, so
// a warp keeps 8 KiB in flight. Scores are reduced with xor shuffles, the
// running max/sum are kept in base 2 (scores pre-multiplied by
// scale*log2(e)), and the four warps' states are merged in shared memory.
#include <math.h>

#include "kf_internal.cuh"

namespace kf {
namespace {

constexpr int kWarps = 4;
constexpr int kSub = 16;  // tokens per sub-block

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
decode_simt_kernel(const DecodeParams p) {
    constexpr int LPT = D / 8;        // lanes per token row
    constexpr int TPP = 32 / LPT;     // tokens per pass
    constexpr int PASSES = kSub / TPP;

    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tok = lane / LPT, chunk = lane % LPT;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, bs = p.block_size;
    const int64_t row0 = ((int64_t)s * p.batch + b) * Hq + (int64_t)h * G;  // first output row

    const SplitRange r = split_range(p, b, s, threadIdx.x == 0 && s == 0 && h == 0);
    if (r.t_begin >= r.t_end) {
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) p.out_partial[row0 * D + i] = 0.f;
        if (threadIdx.x < G) p.lse_partial[row0 + threadIdx.x] = -INFINITY;
        return;
    }

    // this lane's 8 query elements of each head, fp32
    float qf[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 v = reinterpret_cast<const uint4 *>(p.q + ((int64_t)b * Hq + h * G + g) * D)[chunk];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qf[g][2 * e] = bf16_lo(w[e]);
            qf[g][2 * e + 1] = bf16_hi(w[e]);
        }
    }

    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    }

    const int64_t row_vecs = (int64_t)Hkv * D / 8;  // 16-byte vectors between slots
    const uint4 *kc = reinterpret_cast<const uint4 *>(p.k_cache);
    const uint4 *vc = reinterpret_cast<const uint4 *>(p.v_cache);
    const int64_t sb_begin = r.t_begin / kSub, sb_end = (r.t_end + kSub - 1) / kSub;

    for (int64_t sb = sb_begin + warp; sb < sb_end; sb += kWarps) {
        const int64_t t_base = sb * kSub;
        const int64_t phys = physical_block(p, b, t_base / bs);
        const int64_t base = ((phys * bs + t_base % bs) * Hkv + h) * (D / 8) + chunk;
        uint4 kr[PASSES], vr[PASSES];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int t = ps * TPP + tok;
            kr[ps] = __ldg(kc + base + t * row_vecs);
            vr[ps] = __ldg(vc + base + t * row_vecs);
        }
        // scores (base 2), -inf past the split end
        float sc[PASSES][G];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const uint32_t w[4] = {kr[ps].x, kr[ps].y, kr[ps].z, kr[ps].w};
            float kf[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kf[2 * e] = bf16_lo(w[e]);
                kf[2 * e + 1] = bf16_hi(w[e]);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) d = fmaf(qf[g][e], kf[e], d);
#pragma unroll
                for (int off = 1; off < LPT; off <<= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                const bool valid = t_base + ps * TPP + tok < r.t_end;
                sc[ps][g] = valid ? d * p.scale_log2 : -INFINITY;
            }
        }
        // block max over the warp's 16 tokens, then the online update
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float bm = sc[0][g];
#pragma unroll
            for (int ps = 1; ps < PASSES; ++ps) bm = fmaxf(bm, sc[ps][g]);
#pragma unroll
            for (int off = LPT; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
            const float m_new = fmaxf(m[g], bm);
            const float alpha = exp2f(m[g] - m_new);
            m[g] = m_new;
            l[g] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
        }
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const bool valid = t_base + ps * TPP + tok < r.t_end;
            if (!valid) continue;  // never multiply a stale slot's value (it may be non-finite)
            const uint32_t w[4] = {vr[ps].x, vr[ps].y, vr[ps].z, vr[ps].w};
            float vf[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                vf[2 * e] = bf16_lo(w[e]);
                vf[2 * e + 1] = bf16_hi(w[e]);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pr = exp2f(sc[ps][g] - m[g]);
                l[g] += pr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pr, vf[e], acc[g][e]);
            }
        }
    }

    // sum the token groups of the warp (m is warp-uniform)
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1) {
            l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], off);
        }
    }

    // merge the warps' states
    __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
    __shared__ __align__(16) float sm_acc[kWarps][G][D];
    if (lane < LPT) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int e = 0; e < 8; ++e) sm_acc[warp][g][chunk * 8 + e] = acc[g][e];
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            sm_m[warp][g] = m[g];
            sm_l[warp][g] = l[g];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][g]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(sm_m[w][g] - M);  // 0 for a warp that saw no token
            num = fmaf(f, sm_acc[w][g][d], num);
            den = fmaf(f, sm_l[w][g], den);
        }
        p.out_partial[(row0 + g) * D + d] = num / den;
        if (d == 0) p.lse_partial[row0 + g] = (M + log2f(den)) * 0.6931471805599453f;
    }
}

template <int D>
cudaError_t launch_d(const DecodeParams &p, cudaStream_t stream) {
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: decode_simt_kernel<D, 1><<<grid, kWarps * 32, 0, stream>>>(p); break;
        case 2: decode_simt_kernel<D, 2><<<grid, kWarps * 32, 0, stream>>>(p); break;
        case 4: decode_simt_kernel<D, 4><<<grid, kWarps * 32, 0, stream>>>(p); break;
        case 8: decode_simt_kernel<D, 8><<<grid, kWarps * 32, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams &p, cudaStream_t stream) {
    if (p.batch == 0) return cudaSuccess;
    return p.head_dim == 128 ? launch_d<128>(p, stream) : launch_d<64>(p, stream);
}

}  // namespace kf
