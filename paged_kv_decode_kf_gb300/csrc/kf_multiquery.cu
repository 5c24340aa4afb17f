// kf_multiquery.cu -- paged attention of many query tokens per request:
// chunked prefill / speculative verify (causal) and the shared-prefix pass of
// cascade attention (non-causal).
//
// What it computes: "Mathematical Formulation of Chunked Attention" on the
// ultrainstinct.tech page ("Disaggregated Inference Architecture: Paged
// KV-Cache Tiering, Chunked Prefill, and Asynchronous Overlap"): the queries
// of a chunk attend to the keys of earlier chunks in the paged cache without
// a mask and to their own chunk causally. With the chunk already in the cache
// (L tokens, the chunk its last C), query j attends to tokens [0, L - C + j].
// Non-causal, every query attends to all L tokens: cascade attention
// ("What FlashInfer brings: JIT and cascade attention", blog.lo0.es) attends
// a prefix shared by many requests once for all their queries and merges the
// result with each request's own suffix by the same LSE merge. Output is the
// split partials (o, lse) of the decode kernel, one row per query token.
//
// Design: one CTA per (split, KV head, request x query tile). Its NW consumer
// warps each own 8 query columns -- a column is a (query token, query head of
// the KV head's group) pair -- and all of them read the same K/V stages, so
// the KV is loaded once per CTA for 8*NW columns. Per 16-token stage a warp
// runs the decode kernel's tile: S^T = K Q^T (ldmatrix + mma.m16n8k16), the
// online softmax per column with that column's causal limit as a mask, and
// O^T += V^T P^T (ldmatrix.trans, movmatrix.trans, P = P_hi + P_lo). A
// column whose whole range is masked ends as (o = 0, lse = -inf). The TMA
// producer, the bounded mbarrier waits and the block-id checks are those of
// the decode kernel.
#include "kf_decode_tc.cuh"

namespace kf {
namespace {

using namespace tc;

template <int D, int G, int NW, int NS>
struct MqShape {
    static constexpr int kHalves = D / 64;
    static constexpr int kBoxBytes = 64 * kTok * 2;  // one head
    static constexpr int kStageBytes = 2 * kHalves * kBoxBytes;
    static constexpr int kSmemBytes = NS * kStageBytes + NS * 16 + 1024;
    static constexpr int kThreads = 32 * (NW + 1);
};

template <int D, int G, int NW, int NS>
__global__ void __launch_bounds__(MqShape<D, G, NW, NS>::kThreads)
mq_kernel(const MqParams p, const __grid_constant__ CUtensorMap tmap_k,
          const __grid_constant__ CUtensorMap tmap_v) {
    using Sh = MqShape<D, G, NW, NS>;
    constexpr int KS = D / 16;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + NS * Sh::kStageBytes;

    const int s = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / p.q_tiles, qt = blockIdx.z % p.q_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.num_q_heads;

    const int q0 = p.q_start[b], q1 = p.q_start[b + 1];
    if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens) {  // rows outside q: touch nothing
        if (threadIdx.x == 0 && s == 0 && h == 0 && qt == 0) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        return;
    }
    const int64_t C = (int64_t)q1 - q0;
    int64_t L = p.ctx_lens[b];
    const int64_t cap = (int64_t)p.bt_stride * p.block_size;
    const bool report = threadIdx.x == 0 && s == 0 && h == 0 && qt == 0;
    if (L < 0 || L > cap || C < 0 || (p.causal && C > L)) {
        if (report) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        L = L < 0 ? 0 : (L > cap ? cap : L);
    }
    if (L > p.max_context_len && report) raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
    const int64_t ncol_all = C * G;
    // more queries than the host bound max_query_len covers: the rest are not computed
    if (threadIdx.x == 0 && s == 0 && h == 0 && qt == p.q_tiles - 1 &&
        ncol_all > (int64_t)p.q_tiles * 8 * NW)
        raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
    const int64_t col0 = (int64_t)qt * 8 * NW;
    if (col0 >= ncol_all) return;  // beyond this request's queries: nothing to write
    const int64_t ncols = ncol_all - col0 < 8 * NW ? ncol_all - col0 : 8 * NW;

    // token range: the split, clipped to the context and to the last column's limit
    const int64_t span = (int64_t)p.chunk_blocks * p.block_size;
    int64_t t_lo = (int64_t)s * span, t_hi = t_lo + span;
    int64_t t_max = L;
    if (p.causal) {
        const int64_t j_last = (col0 + ncols - 1) / G;
        t_max = L - C + j_last + 1;
    }
    if (t_hi > t_max) t_hi = t_max;
    if (t_lo > t_hi) t_lo = t_hi;

    // column c of this CTA -> (query row, query head) and its token limit
    auto col_row = [&](int64_t c) { return (int64_t)q0 + c / G; };
    auto col_head = [&](int64_t c) { return h * G + (int)(c % G); };
    auto col_limit = [&](int64_t c) { return p.causal ? L - C + c / G + 1 : L; };

    if (t_lo >= t_hi || (*(volatile unsigned int *)p.err & KF_DEVERR_TIMEOUT)) {
        for (int64_t i = threadIdx.x; i < ncols * D; i += blockDim.x) {
            const int64_t c = col0 + i / D;
            p.out_partial[(((int64_t)s * p.num_q_tokens + col_row(c)) * Hq + col_head(c)) * D + i % D] = 0.f;
        }
        for (int64_t i = threadIdx.x; i < ncols; i += blockDim.x) {
            const int64_t c = col0 + i;
            p.lse_partial[((int64_t)s * p.num_q_tokens + col_row(c)) * Hq + col_head(c)] = -INFINITY;
        }
        return;
    }
    const int64_t sb0 = t_lo / kTok;
    const int n_sub = (int)((t_hi + kTok - 1) / kTok - sb0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bars + 8 * i, 1);
            mbar_init(bars + 8 * (NS + i), NW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------ producer ------------------------------
        // whole warp: table entries 32 at a time, lane 0 waits and issues
        const int bs_shift = block_shift(p.block_size);
        int64_t tab_base = -1;
        int32_t tab_ent = -1;
        for (int i = 0; i < n_sub; ++i) {
            const int st = i % NS;
            int go = 1;
            if (lane == 0 && !mbar_wait(bars + 8 * (NS + st), ((i / NS) & 1) ^ 1)) {
                raise_error(p.err, KF_DEVERR_TIMEOUT);
                go = 0;
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            const int64_t t_base = (sb0 + i) * kTok;
            const int64_t lb = t_base >> bs_shift;
            if (tab_base < 0 || lb >= tab_base + 32) {
                tab_base = lb;
                const int64_t e = lb + lane;
                tab_ent = e < p.bt_stride ? p.block_tables[(int64_t)b * p.bt_stride + e] : -1;
            }
            int64_t phys = __shfl_sync(0xffffffffu, tab_ent, (int)(lb - tab_base));
            if (lane == 0) {
                if (phys < 0 || phys >= p.num_blocks) {
                    raise_error(p.err, KF_DEVERR_BLOCK_ID);
                    phys = 0;
                }
                const int slot = (int)(t_base & (p.block_size - 1));
                const uint32_t full = bars + 8 * st;
                const uint32_t dst = base + st * Sh::kStageBytes;
                mbar_arrive_expect_tx(full, Sh::kStageBytes);
#pragma unroll
                for (int hf = 0; hf < Sh::kHalves; ++hf) {
                    tma_load_4d(dst + hf * Sh::kBoxBytes, &tmap_k, 64 * hf, slot, h, (int)phys, full);
                    tma_load_4d(dst + (Sh::kHalves + hf) * Sh::kBoxBytes, &tmap_v, 64 * hf, slot, h,
                                (int)phys, full);
                }
            }
        }
        return;
    }

    // ------------------------------- consumers --------------------------------
    const int g = lane >> 2, qd = lane & 3;
    const int64_t wcol = col0 + 8 * warp;  // this warp's first column

    uint32_t qb[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) qb[ks][0] = qb[ks][1] = 0u;
    if (wcol + g < col0 + ncols) {
        const int64_t c = wcol + g;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + (col_row(c) * Hq + col_head(c)) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = qrow[8 * ks + qd];
            qb[ks][1] = qrow[8 * ks + 4 + qd];
        }
    }
    // this thread's two C-fragment columns
    const int64_t c0 = wcol + 2 * qd, c1 = c0 + 1;
    const bool v0 = c0 < col0 + ncols, v1 = c1 < col0 + ncols;
    const int64_t lim0 = v0 ? col_limit(c0) : 0, lim1 = v1 ? col_limit(c1) : 0;

    float oacc[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_acc[2] = {0.f, 0.f};
    const int lj = lane >> 3, lr = lane & 7;
    bool ok = true;

    for (int i = 0; i < n_sub; ++i) {
        const int st = i % NS;
        if (!mbar_wait(bars + 8 * st, (i / NS) & 1)) {
            raise_error(p.err, KF_DEVERR_TIMEOUT);
            ok = false;
            break;
        }
        const uint32_t kbuf = base + st * Sh::kStageBytes;
        const uint32_t vbuf = kbuf + Sh::kHalves * Sh::kBoxBytes;
        const int64_t t_base = (sb0 + i) * kTok;
        const int64_t rem_tok = t_hi - t_base;
        const int nvalid = rem_tok < kTok ? (int)rem_tok : kTok;
        bool wrote_smem = false;

        if (nvalid < kTok) {
            // V rows past the range are zeroed (their weights are 0, but 0 * NaN is NaN).
            // Every consumer warp zeroes them itself before it reads: the other warps'
            // identical writes cannot change what it sees, so no cross-warp barrier.
            for (int idx = lane; idx < (kTok - nvalid) * 8 * Sh::kHalves; idx += 32) {
                const int hf = idx / ((kTok - nvalid) * 8);
                const int rem = idx % ((kTok - nvalid) * 8);
                const int t = nvalid + rem / 8, c = rem % 8;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vbuf + hf * Sh::kBoxBytes + t * 128 + c * 16),
                             "r"(0u)
                             : "memory");
            }
            wrote_smem = true;
            __syncwarp();
        }

        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int t = lr + ((lj & 1) << 3);
            const int chunk = 2 * ks + (lj >> 1);
            uint32_t fr[4];
            ldsm_x4(kbuf + (chunk >> 3) * Sh::kBoxBytes + swz<128>(t, chunk & 7), fr);
            mma_bf16((ks & 1) ? sd : sc, fr, qb[ks][0], qb[ks][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] += sd[e];
        const int64_t ta = t_base + g, tb = t_base + g + 8;
        const float x0 = (g < nvalid && ta < lim0) ? sc[0] * p.scale_log2 : -INFINITY;
        const float x1 = (g < nvalid && ta < lim1) ? sc[1] * p.scale_log2 : -INFINITY;
        const float x2 = (g + 8 < nvalid && tb < lim0) ? sc[2] * p.scale_log2 : -INFINITY;
        const float x3 = (g + 8 < nvalid && tb < lim1) ? sc[3] * p.scale_log2 : -INFINITY;
        float mx[2] = {fmaxf(x0, x2), fmaxf(x1, x3)};
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (mx[j] > m_run[j] + kRescaleSlack) {
                const float alpha = exp2f(m_run[j] - mx[j]);
                m_run[j] = mx[j];
                l_acc[j] *= alpha;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    oacc[mt][j] *= alpha;
                    oacc[mt][j + 2] *= alpha;
                }
            }
        }
        // a column with no token yet keeps m = -inf: its weights are 0
        const float mu0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
        const float mu1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
        const float p0 = exp2f(x0 - mu0), p1 = exp2f(x1 - mu1);
        const float p2 = exp2f(x2 - mu0), p3 = exp2f(x3 - mu1);
        l_acc[0] += p0 + p2;
        l_acc[1] += p1 + p3;
        const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
        const uint32_t r01 = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        const uint32_t r23 = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
        const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
        const uint32_t bl0 = movmatrix_trans(r01), bl1 = movmatrix_trans(r23);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int t = lr + ((lj >> 1) << 3);
            const int chunk = 2 * mt + (lj & 1);
            uint32_t fr[4];
            ldsm_x4_trans(vbuf + (chunk >> 3) * Sh::kBoxBytes + swz<128>(t, chunk & 7), fr);
            mma_bf16(oacc[mt], fr, bh0, bh1);
            mma_bf16(oacc[mt], fr, bl0, bl1);
        }
        if (wrote_smem) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (NS + st));
    }
    if (!ok) return;

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_acc[0] += __shfl_xor_sync(0xffffffffu, l_acc[0], off);
        l_acc[1] += __shfl_xor_sync(0xffffffffu, l_acc[1], off);
    }
    const bool e0 = l_acc[0] == 0.f, e1 = l_acc[1] == 0.f;  // no token in range: (0, -inf)
    const float inv0 = e0 ? 0.f : 1.f / l_acc[0], inv1 = e1 ? 0.f : 1.f / l_acc[1];
    float *o0 = v0 ? p.out_partial + (((int64_t)s * p.num_q_tokens + col_row(c0)) * Hq + col_head(c0)) * D : nullptr;
    float *o1 = v1 ? p.out_partial + (((int64_t)s * p.num_q_tokens + col_row(c1)) * Hq + col_head(c1)) * D : nullptr;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        const int d0 = 16 * mt + g;
        if (o0) {
            o0[d0] = oacc[mt][0] * inv0;
            o0[d0 + 8] = oacc[mt][2] * inv0;
        }
        if (o1) {
            o1[d0] = oacc[mt][1] * inv1;
            o1[d0 + 8] = oacc[mt][3] * inv1;
        }
    }
    if (g == 0) {
        if (v0)
            p.lse_partial[((int64_t)s * p.num_q_tokens + col_row(c0)) * Hq + col_head(c0)] =
                e0 ? -INFINITY : (m_run[0] + log2f(l_acc[0])) * 0.6931471805599453f;
        if (v1)
            p.lse_partial[((int64_t)s * p.num_q_tokens + col_row(c1)) * Hq + col_head(c1)] =
                e1 ? -INFINITY : (m_run[1] + log2f(l_acc[1])) * 0.6931471805599453f;
    }
}

template <int D, int G, int NW>
cudaError_t launch_mq_t(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk,
                        const CUtensorMap &mv) {
    constexpr int NS = 8;  // 8 KiB stages (one head, bf16): 64 KiB ring
    using Sh = MqShape<D, G, NW, NS>;
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        e = cudaFuncSetAttribute(mq_kernel<D, G, NW, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch * p.q_tiles);
    mq_kernel<D, G, NW, NS><<<grid, Sh::kThreads, Sh::kSmemBytes, stream>>>(p, mk, mv);
    return cudaGetLastError();
}

template <int D, int NW>
cudaError_t launch_mq_g(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk,
                        const CUtensorMap &mv) {
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: return launch_mq_t<D, 1, NW>(p, stream, mk, mv);
        case 2: return launch_mq_t<D, 2, NW>(p, stream, mk, mv);
        case 4: return launch_mq_t<D, 4, NW>(p, stream, mk, mv);
        case 8: return launch_mq_t<D, 8, NW>(p, stream, mk, mv);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int mq_columns_per_cta(int max_query_len, int group) {
    return (int64_t)max_query_len * group <= 32 ? 32 : 64;
}

cudaError_t launch_multiquery(MqParams p, cudaStream_t stream, void *encode) {
    if (p.batch == 0 || p.num_q_tokens == 0) return cudaSuccess;
    const int G = p.num_q_heads / p.num_kv_heads;
    const int cols = mq_columns_per_cta(p.max_query_len, G);
    p.q_tiles = (int)(((int64_t)p.max_query_len * G + cols - 1) / cols);
    if ((int64_t)p.batch * p.q_tiles > 65535) return cudaErrorInvalidValue;
    tc::EncodeFn fn = reinterpret_cast<tc::EncodeFn>(encode);
    CUtensorMap mk, mv;
    if (!tc::encode_cache_map(fn, &mk, p.k_cache, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim,
                              1, false) ||
        !tc::encode_cache_map(fn, &mv, p.v_cache, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim,
                              1, false))
        return cudaErrorInvalidValue;
    if (p.head_dim == 128)
        return cols == 32 ? launch_mq_g<128, 4>(p, stream, mk, mv) : launch_mq_g<128, 8>(p, stream, mk, mv);
    return cols == 32 ? launch_mq_g<64, 4>(p, stream, mk, mv) : launch_mq_g<64, 8>(p, stream, mk, mv);
}

}  // namespace kf
