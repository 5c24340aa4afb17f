// kf_decode_bal.cuh -- the single-launch decode step (append + split-KV
// attention + LSE merge) on a balanced schedule (kernel template;
// instantiated by kf_decode_bal.cu for bf16 caches and kf_decode_bal_fp8.cu
// for FP8 E4M3 caches).
//
// What it computes is what the split-rule step computes: KernelFlume
// (academ.us/article/2606.29207) sections 3.1-3.2 for each token range, and
// the exact merge of section 5.1 ("Mathematical Formulation of Chunked
// Attention", ultrainstinct.tech) over the ranges of a request. Only the
// partition of the tokens into ranges differs, which section 5.1 leaves free:
// any partition merges to attention over all the tokens.
//
// Schedule. The split rule cuts every request into the same number of
// chunks, so the work of one CTA follows the longest request and a grid of
// B x groups x S CTAs rarely fills the GPU's CTA slots evenly: with three
// FP8 CTAs per SM, 384 CTAs leave 80 SMs with three and 72 with two, and the
// loaded SMs set the step time. Here the grid is exactly one wave
// (P CTAs per KV-head group, P x groups = resident CTAs per SM x SMs), and
// the 16-token stages of all requests, laid end to end in request order
// (T stages in all), are cut into P' = min(P, T) equal runs: CTA c < P'
// takes stages [floor(cT/P'), floor((c+1)T/P')), never empty. A run may cross
// request boundaries; each piece of it (a segment) is one request's tokens,
// attended with that request's q and appended row, and finished on its own:
//  - a request whose stages all fall in one CTA is complete there: its rows
//    go straight to the output;
//  - otherwise the segment is a partial (o, lse). Only a CTA's first and last
//    segments can be cut, so each CTA owns two workspace slots (2c: first,
//    2c+1: last) of [Hq, D] rows. The request's CTAs are c0..c1, from the
//    stage formula; its slots are 2c0 + (request starts after c0's first
//    stage) and 2c for c > c0. With extra partials to merge, a request inside
//    one CTA goes through a slot of its own, 2P + b.
// Every CTA computes T and the request at its first stage itself, from the
// context lengths (a block-wide scan), so the step needs no planning launch
// and no host synchronisation.
//
// Merge. A consumer warp stores its segments' rows as it goes and waits on
// nothing at a request boundary; after its run it fences once and counts its
// partials, one counter per (request, KV head); the warp that brings a count
// to the request's number of CTAs merges that head's G rows from the slots
// (plus any extra partials) in registers, and clears the counter for the
// next step.
//
// Per-stage work (TMA ring, tensor-core tiles, online softmax, FP8 widening)
// is the split-rule kernel's, shared through kf_decode_tc.cuh.
#pragma once

#include "kf_decode_tc.cuh"

namespace kf {
namespace tc {

// Tokens a request attends in this step (cached + the appended one), from
// its cached length `before`, and the position of the append (-1 if the table
// has no room or the length is negative); the same checks as the split-rule
// step, reported when `report`.
__device__ __forceinline__ int64_t step_len(const DecodeParams &p, int64_t before, bool report, int64_t &p_new) {
    const int64_t cap = (int64_t)p.bt_stride * p.block_size;
    int64_t L = before + 1;
    p_new = before;
    if (before < 0 || L > cap) {
        if (report) raise_error(p.err, before < 0 ? KF_DEVERR_CONTEXT_LEN : KF_DEVERR_APPEND_POS);
        L = before < 0 ? 0 : cap;
        p_new = -1;
    }
    if (L > p.max_context_len && report) raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
    return L;
}

// CTA whose run holds global stage y: the largest c with floor(cT/P) <= y.
__device__ __forceinline__ int cta_of(int64_t y, int64_t T, int P) {
    return (int)(((y + 1) * (int64_t)P - 1) / T);
}

__device__ __forceinline__ int64_t run_start(int c, int64_t T, int P) {
    return (int64_t)c * T / P;
}

// Workspace slot of the segment of request b (stages [Rb, Rb + nb) of the
// whole batch) in CTA c, whose run starts at x0; -1: the segment is the whole
// request and has nothing to merge with, its rows are final. A request cut
// across CTAs c0..c1 has partial 2c0 + (it starts after c0's run does) and 2c
// for c > c0 (only a run's first and last segments can be cut); a whole
// request with extra partials to merge has slot 2 Pmax + b, Pmax = the grid's
// CTAs per group.
__device__ __forceinline__ int bal_slot(int64_t Rb, int nb, int b, int64_t T, int64_t x0, int Pe, int c, int Pmax,
                                        int n_ex) {
    const int c0 = cta_of(Rb, T, Pe), c1 = cta_of(Rb + nb - 1, T, Pe);
    if (c0 == c1) return n_ex == 0 ? -1 : 2 * Pmax + b;
    return 2 * c + (Rb <= x0 ? 0 : 1);
}

// Exact LSE merge of one (request, KV head)'s G rows by one warp: partial 0
// is workspace slot s0, partial 0 < k < n_cta slot 2(c0 + k), partial k >=
// n_cta extra slot k - n_cta. w_k = e^{lse_k - M}, out = sum w_k o_k / sum w_k,
// lse = M + ln sum w_k; a zero weight drops its o whatever its bits.
// (Out of line, arguments by value: it runs once per request and head, and
// inlined it would weigh on the stage loop's register budget.)
struct MergeArgs {
    const float *ws_o, *ws_lse, *ex_o, *ex_lse;
    void *out;
    float *lse_out;
    int n_ex, out_dtype, batch, num_q_heads;
};

__device__ __forceinline__ MergeArgs merge_args(const DecodeParams &p, const StepParams &sp) {
    MergeArgs m;
    m.ws_o = sp.ws_o;
    m.ws_lse = sp.ws_lse;
    m.ex_o = sp.ex_o;
    m.ex_lse = sp.ex_lse;
    m.out = sp.out;
    m.lse_out = sp.lse_out;
    m.n_ex = sp.n_ex;
    m.out_dtype = sp.out_dtype;
    m.batch = p.batch;
    m.num_q_heads = p.num_q_heads;
    return m;
}

template <int D, int G>
__device__ __noinline__ void warp_merge(const MergeArgs m, int b, int hq, int c0, int n_cta, int s0, int lane) {
    constexpr int C4 = D / 4;               // float4 units per row
    constexpr int NU = (G * C4 + 31) / 32;  // units per lane
    constexpr int KPR = 32 / G;             // partials per round of the lse pass (lane = k * G + r)
    constexpr int MAXR = 4;                 // rounds kept in registers
    constexpr int SB = 16 / NU > 0 ? 16 / NU : 1;  // partials per batch of o loads (16 float4 in flight)
    const int Hq = m.num_q_heads;
    const int n = n_cta + m.n_ex;
    auto row_of = [&](int k, int r) -> int64_t {  // row index of partial k, query head hq + r
        return k < n_cta ? (int64_t)(k == 0 ? s0 : 2 * (c0 + k)) * Hq + hq + r
                         : ((int64_t)(k - n_cta) * m.batch + b) * Hq + hq + r;
    };
    auto lse_at = [&](int k, int r) -> float { return __ldcg((k < n_cta ? m.ws_lse : m.ex_lse) + row_of(k, r)); };
    // lse pass, lane-parallel: lane (k % KPR) * G + r holds partial k's lse for
    // row r in round k / KPR; the row max and the weight sum by shuffles over
    // the lanes of one row. Up to MAXR * KPR partials stay in registers;
    // beyond that the weights are recomputed from the lse when needed.
    const int r_l = lane % G, k_l = lane / G;
    float lv[MAXR];
    float Mr = -INFINITY;
#pragma unroll
    for (int q = 0; q < MAXR; ++q) {
        const int k = q * KPR + k_l;
        lv[q] = k < n ? lse_at(k, r_l) : -INFINITY;
        Mr = fmaxf(Mr, lv[q]);
    }
    for (int k = MAXR * KPR + k_l; k < n; k += KPR) Mr = fmaxf(Mr, lse_at(k, r_l));
#pragma unroll
    for (int off = G; off < 32; off <<= 1) Mr = fmaxf(Mr, __shfl_xor_sync(0xffffffffu, Mr, off));
    float Sr = 0.f;
#pragma unroll
    for (int q = 0; q < MAXR; ++q) {
        lv[q] = lv[q] == -INFINITY ? 0.f : expf(lv[q] - Mr);  // now the weight
        Sr += lv[q];
    }
    for (int k = MAXR * KPR + k_l; k < n; k += KPR) {
        const float l = lse_at(k, r_l);
        Sr += l == -INFINITY ? 0.f : expf(l - Mr);
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1) Sr += __shfl_xor_sync(0xffffffffu, Sr, off);

    int rr[NU];
    float4 acc[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int unit = lane + 32 * u;
        rr[u] = unit < G * C4 ? unit / C4 : 0;  // (dead units read row 0 and are not stored)
        acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // weight of partial k for row r: from the lse pass's registers, or recomputed
    auto weight = [&](int k, int r, float Mrow) -> float {
        if (k < MAXR * KPR) {
            float w = 0.f;
#pragma unroll
            for (int q = 0; q < MAXR; ++q) {
                const float v = __shfl_sync(0xffffffffu, lv[q], (k % KPR) * G + r);
                if (q == k / KPR) w = v;
            }
            return w;
        }
        const float l = lse_at(k, r);
        return l == -INFINITY ? 0.f : expf(l - Mrow);
    };
    for (int k0 = 0; k0 < n; k0 += SB) {
        float4 o[SB][NU];
#pragma unroll
        for (int j = 0; j < SB; ++j)
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int k = k0 + j;
                const float *ob = k < n_cta ? m.ws_o : m.ex_o;
                o[j][u] = k < n ? __ldcg(reinterpret_cast<const float4 *>(ob + row_of(k, rr[u]) * D) +
                                         (lane + 32 * u) % C4)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int j = 0; j < SB; ++j) {
            const int k = k0 + j;
            if (k >= n) break;
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const float Mrow = __shfl_sync(0xffffffffu, Mr, rr[u]);  // lane rr[u] holds row rr[u]'s max
                const float w = weight(k, rr[u], Mrow);
                // a zero weight drops o whatever its bits (an empty extra slot)
                if (w != 0.f) {
                    acc[u].x = fmaf(w, o[j][u].x, acc[u].x);
                    acc[u].y = fmaf(w, o[j][u].y, acc[u].y);
                    acc[u].z = fmaf(w, o[j][u].z, acc[u].z);
                    acc[u].w = fmaf(w, o[j][u].w, acc[u].w);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const float Srow = __shfl_sync(0xffffffffu, Sr, rr[u]);
        const float Mrow = __shfl_sync(0xffffffffu, Mr, rr[u]);
        if (lane + 32 * u >= G * C4) continue;
        const int c = (lane + 32 * u) % C4;
        const int64_t row = (int64_t)b * Hq + hq + rr[u];
        const float inv = 1.f / Srow;
        float4 a = acc[u];
        a.x *= inv;
        a.y *= inv;
        a.z *= inv;
        a.w *= inv;
        if (m.out_dtype == KF_F32) {
            reinterpret_cast<float4 *>(static_cast<float *>(m.out) + row * D)[c] = a;
        } else {
            uint2 v;
            v.x = pack_bf16(a.x, a.y);
            v.y = pack_bf16(a.z, a.w);
            reinterpret_cast<uint2 *>(static_cast<uint16_t *>(m.out) + row * D)[c] = v;
        }
        if (c == 0 && m.lse_out) m.lse_out[row] = Mrow + logf(Srow);
    }
}

// Register budget: three FP8 CTAs per SM (the split-rule kernel's), and for
// bf16 caches at most 168 per thread, so that two CTAs of five warps fit: an
// SM sub-partition holds floor(16384 / (32 x regs)) warps, three at 168.
template <int D, int HPC, int G, int NS, bool KV8>
__global__ void __launch_bounds__(TcShape<D, HPC, NS, KV8>::kThreads, (KV8 && HPC <= 4) ? 3 : 1)
__maxnreg__((KV8 && HPC <= 4) ? 128 : 168)
decode_bal_kernel(const DecodeParams p, const StepParams sp, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v) {
    using Sh = TcShape<D, HPC, NS, KV8>;
    constexpr int RB = Sh::kRowBytes;
    constexpr int KS = D / 16;
    constexpr int NW = HPC + 1;  // warps

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + NS * Sh::kStageBytes;  // full[NS] then empty[NS]

    // grid (groups, P): the CTAs of one run, one per KV-head group, launch side
    // by side, and read the two halves of the same cache rows at the same time
    const int hg = blockIdx.x, pc = blockIdx.y, P = (int)gridDim.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = hg * HPC;
    const int Hq = p.num_q_heads;
    const int B = p.batch;

    // ---- this CTA's run of stages: block-wide scan of the requests' stage counts ----
    __shared__ long long sh_warp[NW];
    __shared__ long long sh_first_r;  // global stage index of the first request's stage 0
    __shared__ long long sh_run[4];   // T, x0, x1, P' (read at segment ends, not held in registers)
    __shared__ int sh_first_b;
    const bool report = pc == 0 && hg == 0;
    const int per = (B + (int)blockDim.x - 1) / (int)blockDim.x;
    const int lo = (int)threadIdx.x * per, hi = lo + per < B ? lo + per : B;
    long long mine = 0;
    for (int bb = lo; bb < hi; ++bb) {
        int64_t pn;
        mine += (step_len(p, p.ctx_lens[bb], report, pn) + kTok - 1) / kTok;
    }
    long long incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) sh_warp[warp] = incl;
    if (threadIdx.x == 0) sh_first_b = -1;
    __syncthreads();
    long long before = 0, T = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        before += w < warp ? sh_warp[w] : 0;
        T += sh_warp[w];
    }
    const long long excl = before + incl - mine;  // stages of requests < lo
    // with fewer stages than CTAs only the first T CTAs get a (one-stage) run:
    // every run is non-empty, so a request's CTAs c0..c1 all hold a piece of it
    const int Pe = T < (long long)P ? (int)T : P;
    const int64_t x0 = pc < Pe ? run_start(pc, T, Pe) : 0, x1 = pc < Pe ? run_start(pc + 1, T, Pe) : 0;
    if (threadIdx.x == 0) {
        sh_run[0] = T;
        sh_run[1] = x0;
        sh_run[2] = x1;
        sh_run[3] = Pe;
    }
    if (x0 < x1 && excl <= x0 && x0 < excl + mine) {
        int64_t R = excl;
        for (int bb = lo; bb < hi; ++bb) {
            int64_t pn;
            const int64_t nb = (step_len(p, p.ctx_lens[bb], false, pn) + kTok - 1) / kTok;
            if (x0 < R + nb) {
                sh_first_b = bb;
                sh_first_r = R;
                break;
            }
            R += nb;
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bars + 8 * i, 1);           // full: producer's expect_tx arrival
            mbar_init(bars + 8 * (NS + i), HPC);  // empty: one arrival per consumer warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int b_first = sh_first_b;
    if (b_first < 0) return;  // no stages for this CTA (T < P), or no tokens at all
    const int64_t r_first = sh_first_r;

    if (warp == HPC) {
        // ------------------------------ producer ------------------------------
        // walks the run's segments; per segment, table entries 32 at a time
        const int bs_shift = block_shift(p.block_size);
        unsigned int i = 0;  // ring stage counter over the whole run
        int b = b_first;
        int64_t Rb = r_first, y = x0;
        bool go = true;
        while (go && y < x1) {
            int64_t pn;
            const int64_t nb = (step_len(p, p.ctx_lens[b], false, pn) + kTok - 1) / kTok;
            const int64_t s_hi = (Rb + nb < x1 ? Rb + nb : x1) - Rb;
            int64_t tab_base = -1;
            int32_t tab_ent = -1;
            for (int64_t j = y - Rb; j < s_hi; ++j, ++i) {
                const int st = (int)(i % NS);
                int ok = 1;
                if (lane == 0 && !mbar_wait(bars + 8 * (NS + st), ((i / NS) & 1) ^ 1)) {
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
                    ok = 0;
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    go = false;
                    break;
                }
                const int64_t t_base = j * kTok;
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
                        tma_load_4d(dst + hf * Sh::kBoxBytes, &tmap_k, 64 * hf, slot, h0, (int)phys, full);
                        tma_load_4d(dst + (Sh::kHalves + hf) * Sh::kBoxBytes, &tmap_v, 64 * hf, slot, h0,
                                    (int)phys, full);
                    }
                }
            }
            y = Rb + s_hi;
            Rb += nb;
            ++b;
        }
        return;
    }

    // ------------------------------- consumers --------------------------------
    // The segment's request, its stage offset, stage count, token count and
    // append position live in shared memory (one record per warp) and are
    // read back after the stage loop: across the loop only 32-bit stage
    // counters stay in registers, which leaves the loop's own invariants in
    // registers under the FP8 kernel's three-CTAs-per-SM cap. At a request
    // boundary the next request's length and q words are loaded before this
    // segment's rows are stored, and nothing else waits: partials are counted
    // (and merged) after the run, behind one fence. Without extra partials
    // only a run's first and last segments can be cut, and the warp keeps
    // those two in shared memory; with extra partials every segment merges,
    // and a second walk over the run's segments finds them.
    __shared__ long long sh_seg_r[HPC], sh_seg_p[HPC], sh_seg_l[HPC];
    __shared__ int sh_seg_b[HPC], sh_seg_n[HPC];
    __shared__ long long sh_pend_r[HPC][2];
    __shared__ int sh_pend_b[HPC][2], sh_pend_n[HPC][2];
    volatile long long *seg_r = sh_seg_r + warp, *seg_p = sh_seg_p + warp, *seg_l = sh_seg_l + warp;
    volatile int *seg_b = sh_seg_b + warp, *seg_n = sh_seg_n + warp;
    volatile long long *pend_r = sh_pend_r[warp];
    volatile int *pend_b = sh_pend_b[warp], *pend_n = sh_pend_n[warp];
    const volatile long long *run = sh_run;
    const int hkv = h0 + warp;
    const uint32_t head_off = warp * (kTok * RB);  // this head's 16 rows in a box
    bool ok = true;
    unsigned int i = 0;           // ring stage counter over the whole run (unsigned: i % NS is a mask)
    int j = (int)(x0 - r_first);  // first stage of the current segment, local to its request
    int n_pend = 0;
    uint32_t qb[KS][2];
    {
        int64_t p_new;
        const int64_t L = step_len(p, p.ctx_lens[b_first], false, p_new);
        if (lane == 0) {
            *seg_b = b_first;
            *seg_r = r_first;
            *seg_n = (int)((L + kTok - 1) / kTok);
            *seg_l = L;
            *seg_p = p_new;
        }
        load_q_raw<D, G, KV8>(p.q + ((int64_t)b_first * Hq + hkv * G + (lane >> 2)) * D, lane, qb);
    }
    __syncwarp();
    for (;;) {
        int s_hi, last, last_valid, app_j, app_t;
        bool more;
        {
            const int64_t Rb = *seg_r, L = *seg_l, p_new = *seg_p;
            const int nb = *seg_n;
            const int64_t room = run[2] - Rb;  // stages of the run left from the request's start
            s_hi = nb < room ? nb : (int)room;
            more = nb < room;  // the run goes on into the next request
            // per-stage bookkeeping in stage-local terms: the last stage and its
            // valid tokens, the stage and slot of the append
            last = nb - 1;
            last_valid = (int)(L - (int64_t)last * kTok);
            app_j = p_new >= 0 ? (int)(p_new / kTok) : -1;
            app_t = (int)(p_new % kTok);
        }
        const bool nonempty = j < s_hi;
        const float qe_scale = prep_q<D, KV8>(qb);
        const float sl2 = KV8 ? p.scale_log2 * p.k_scale[hkv] * qe_scale : p.scale_log2;
        float oacc[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_acc[2] = {0.f, 0.f};
        // (after a timeout the warp skips the stages but still walks the
        // segments and counts them, so the counters stay consistent)
        for (; ok && j < s_hi; ++j, ++i) {
            const int st = (int)(i % NS);
            if (!mbar_wait(bars + 8 * st, (i / NS) & 1)) {
                raise_error(p.err, KF_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            const uint32_t kbuf = base + st * Sh::kStageBytes + head_off;
            const uint32_t vbuf = kbuf + Sh::kHalves * Sh::kBoxBytes;
            const int nvalid = j == last ? last_valid : kTok;
            bool wrote_smem = false;
            if (j == app_j) {
                append_row<Sh, D, KV8>(p, sp, *seg_b, hkv, *seg_p, app_t, kbuf, vbuf, lane);
                wrote_smem = true;
                __syncwarp();
            }
            if (nvalid < kTok) {
                zero_v_tail<Sh>(vbuf, nvalid, lane);
                wrote_smem = true;
                __syncwarp();
            }
            stage_math<Sh, D, KV8>(kbuf, vbuf, nvalid, qb, sl2, oacc, m_run, l_acc, lane);
            if (wrote_smem) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (NS + st));
        }
        // the next request's length and q words, loaded before this segment's
        // rows are stored so that the two latencies overlap
        int64_t Ln = 0, pn = -1;
        if (more) {
            const int bn = *seg_b + 1;
            Ln = step_len(p, p.ctx_lens[bn], false, pn);
            load_q_raw<D, G, KV8>(p.q + ((int64_t)bn * Hq + hkv * G + (lane >> 2)) * D, lane, qb);
        }
        if (nonempty) {
            // the segment's rows: final, or a partial (slot of bal_slot)
            const int b = *seg_b;
            const int64_t Rb = *seg_r;
            const int nb = *seg_n;
            const int slot = bal_slot(Rb, nb, b, run[0], run[1], (int)run[3], (int)blockIdx.y, P, sp.n_ex);
            const float vsc = KV8 ? p.v_scale[hkv] : 1.f;
            const int64_t row = (slot < 0 ? (int64_t)b : (int64_t)slot) * Hq + hkv * G;
            write_rows<D, G, KV8>(oacc, l_acc, m_run, vsc, row, slot < 0 ? nullptr : sp.ws_o, sp.out,
                                  sp.out_dtype, slot < 0 ? sp.lse_out : sp.ws_lse, lane);
            if (slot >= 0 && sp.n_ex == 0) {
                if (lane == 0) {
                    pend_b[n_pend] = b;
                    pend_r[n_pend] = Rb;
                    pend_n[n_pend] = nb;
                }
                ++n_pend;
            }
        }
        if (!more) break;
        const int64_t Rn = *seg_r + *seg_n;
        __syncwarp();
        if (lane == 0) {
            *seg_b = *seg_b + 1;
            *seg_r = Rn;
            *seg_n = (int)((Ln + kTok - 1) / kTok);
            *seg_l = Ln;
            *seg_p = pn;
        }
        __syncwarp();
        j = 0;
    }
    // count the run's partials behind one fence; the warp that completes a
    // request's count merges it
    if (sp.n_ex == 0 && n_pend == 0) return;
    __threadfence();
    __syncwarp();
    const int64_t Tv = run[0], x1v = run[2];
    const int Pev = (int)run[3];
    // one loop over the partials: the recorded ones, or a walk over the run
    int bw = b_first, e = 0;
    int64_t Rw = r_first;
    for (;;) {
        int b, nb, slot = 0;
        int64_t Rb;
        if (sp.n_ex == 0) {
            if (e >= n_pend) break;
            b = pend_b[e];
            Rb = pend_r[e];
            nb = pend_n[e];
            ++e;
        } else {
            if (Rw >= x1v) break;
            int64_t pn;
            b = bw;
            Rb = Rw;
            nb = (int)((step_len(p, p.ctx_lens[b], false, pn) + kTok - 1) / kTok);
            Rw += nb;
            ++bw;
            if (nb == 0) continue;
            slot = bal_slot(Rb, nb, b, Tv, run[1], Pev, (int)blockIdx.y, P, sp.n_ex);
        }
        const int c0 = cta_of(Rb, Tv, Pev), n_cta = cta_of(Rb + nb - 1, Tv, Pev) - c0 + 1;
        unsigned int is_last = 0;
        if (lane == 0) {
            unsigned int *ctr = sp.counters + (int64_t)b * p.num_kv_heads + hkv;
            is_last = atomicAdd(ctr, 1u) == (unsigned int)(n_cta - 1);
            if (is_last) *ctr = 0u;  // every other CTA of the request has counted: reset
        }
        if (__shfl_sync(0xffffffffu, is_last, 0) && ok) {
            __threadfence();
            const int s0 = n_cta == 1 ? slot : 2 * c0 + (Rb == run_start(c0, Tv, Pev) ? 0 : 1);
            warp_merge<D, G>(merge_args(p, sp), b, hkv * G, c0, n_cta, s0, lane);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int V>
using IntC = std::integral_constant<int, V>;

// Calls f(IntC<D>, IntC<HPC>, IntC<G>) for the runtime shape.
template <class F>
cudaError_t bal_dispatch(int head_dim, int hpc, int group, F &&f) {
    auto by_g = [&](auto d, auto h) -> cudaError_t {
        switch (group) {
            case 1: return f(d, h, IntC<1>{});
            case 2: return f(d, h, IntC<2>{});
            case 4: return f(d, h, IntC<4>{});
            case 8: return f(d, h, IntC<8>{});
        }
        return cudaErrorInvalidValue;
    };
    auto by_h = [&](auto d) -> cudaError_t {
        switch (hpc) {
            case 8: return by_g(d, IntC<8>{});
            case 4: return by_g(d, IntC<4>{});
            case 2: return by_g(d, IntC<2>{});
            case 1: return by_g(d, IntC<1>{});
        }
        return cudaErrorInvalidValue;
    };
    if (head_dim == 128) return by_h(IntC<128>{});
    if (head_dim == 64) return by_h(IntC<64>{});
    return cudaErrorInvalidValue;
}

// The kernel instantiation's shared-memory opt-in (once per device) and its
// resident CTAs per SM from the occupancy calculator (registers, shared
// memory and threads together), cached per device.
template <int D, int HPC, int G, bool KV8>
cudaError_t bal_prepare(int *resident) {
    constexpr int NS = stages_for<D, HPC, KV8>();
    using Sh = TcShape<D, HPC, NS, KV8>;
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int r = cached[dev].load();
    if (r == 0) {
        e = cudaFuncSetAttribute(decode_bal_kernel<D, HPC, G, NS, KV8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, decode_bal_kernel<D, HPC, G, NS, KV8>,
                                                          Sh::kThreads, Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (r < 1) return cudaErrorInvalidConfiguration;
        cached[dev].store(r);
    }
    *resident = r;
    return cudaSuccess;
}

template <bool KV8>
cudaError_t bal_resident(int head_dim, int num_q_heads, int num_kv_heads, int *resident) {
    return bal_dispatch(head_dim, heads_per_cta(num_kv_heads), num_q_heads / num_kv_heads,
                        [&](auto d, auto h, auto g) -> cudaError_t {
                            return bal_prepare<decltype(d)::value, decltype(h)::value, decltype(g)::value,
                                               KV8>(resident);
                        });
}

// Launch with `ctas` CTAs per KV-head group (the caller sizes it to one wave).
template <bool KV8>
cudaError_t launch_bal(const DecodeParams &p, const StepParams &sp, int ctas, cudaStream_t stream,
                       void *encode) {
    if (p.batch == 0) return cudaSuccess;
    const int hpc = heads_per_cta(p.num_kv_heads);
    EncodeFn fn = reinterpret_cast<EncodeFn>(encode);
    CUtensorMap mk, mv;
    if (!encode_cache_map(fn, &mk, p.k_cache, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim, hpc,
                          KV8) ||
        !encode_cache_map(fn, &mv, p.v_cache, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim, hpc,
                          KV8))
        return cudaErrorInvalidValue;
    return bal_dispatch(p.head_dim, hpc, p.num_q_heads / p.num_kv_heads,
                        [&](auto d, auto h, auto g) -> cudaError_t {
                            constexpr int D = decltype(d)::value, HPC = decltype(h)::value,
                                          G = decltype(g)::value;
                            constexpr int NS = stages_for<D, HPC, KV8>();
                            using Sh = TcShape<D, HPC, NS, KV8>;
                            int resident = 0;
                            cudaError_t e = bal_prepare<D, HPC, G, KV8>(&resident);
                            if (e != cudaSuccess) return e;
                            const dim3 grid(p.num_kv_heads / HPC, ctas, 1);
                            decode_bal_kernel<D, HPC, G, NS, KV8>
                                <<<grid, Sh::kThreads, Sh::kSmemBytes, stream>>>(p, sp, mk, mv);
                            return cudaGetLastError();
                        });
}

}  // namespace tc
}  // namespace kf
