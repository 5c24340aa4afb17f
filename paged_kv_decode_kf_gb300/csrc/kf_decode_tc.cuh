// kf_decode_tc.cuh -- split-KV paged decode attention, TMA-fed, GQA-grouped
// tensor-core tiles (kernel template; instantiated by kf_decode_tc.cu for
// bf16 caches and kf_decode_tc_fp8.cu for FP8 E4M3 caches).
//
// What it computes is the decode attention of KernelFlume
// (academ.us/article/2606.29207), sections 3.1-3.2: for one split (token
// range) of one request, each query head's softmax(q K^T scale) V over the
// range, returned as a partial (o, lse) for the LSE merge; the running
// max/sum update is the online-softmax step of "Disaggregated Inference
// Architecture: Paged KV-Cache Tiering, Chunked Prefill, and Asynchronous
// Overlap" (ultrainstinct.tech), "Mathematical Formulation of Chunked
// Attention". The pages size no kernel for this GPU; the design below is
// this library's own.
//
// Work unit: one CTA per (split, group of HPC KV heads, request).
//
// Data movement: the cache is [num_blocks, bs, Hkv, D] bf16. A 4-D tensor map
// views it as (d, slot, head, block) with strides (2 B, Hkv*D*2, D*2,
// bs*Hkv*D*2) and boxes of 64 d x 16 slots x HPC heads x 1 block, 128-byte
// swizzled. One stage = 16 tokens of HPC heads, K and V (D/64 boxes each);
// a producer warp walks the split's blocks through the block table and
// issues the stage's TMA loads on a full/empty mbarrier ring of NS stages, so
// up to NS stages (NS * 64*HPC*D bytes) are in flight per CTA. With HPC = Hkv
// a stage is one contiguous run of the block per operand.
//
// Arithmetic: consumer warp w owns KV head h0 + w and its G query heads. Per
// 16-token stage it runs the two small contractions on the tensor cores with
// mma.m16n8k16 (bf16 in, fp32 accumulate):
//   S^T[16 tok x 8 heads] = K[16 x D] * Q^T[D x 8]     (ldmatrix K, Q^T in registers)
//   O^T[D x 8 heads]    += V^T[D x 16] * P^T[16 x 8]   (ldmatrix.trans V, P^T from
//                                                      movmatrix.trans of the bf16 P)
// The G <= 8 query heads are the N = 8 columns (padded with zero rows of Q).
// Softmax is online in base 2 (scores times scale*log2 e); the running max is
// raised only when a tile exceeds it by more than 8 (p <= 2^8), which leaves
// o = O/l and lse = (m + log2 l) ln 2 unchanged. l sums p in fp32; P enters the
// PV product as a bf16 pair P_hi + P_lo (two MMAs on the same V fragment), so
// the weights carry about 16 significant bits instead of bf16's 8. The 128-byte
// swizzle puts the 8 token rows that one ldmatrix reads in 8 different bank
// groups.
//
// FP8 E4M3 caches (per-KV-head fp32 scales; the "--kv-cache-dtype fp8" option
// of the decode posts on blog.lo0.es, "Quantised KV cache"): the TMA box is
// one row of D codes per token, and the products run in fp16 (every E4M3
// value is exact in fp16; q is scaled per warp by an exact power of two into
// fp16's range, where its 8 significant bits fit exactly). K goes through
// ldmatrix as is; each thread's 32-bit register then holds 4 consecutive
// codes of one token, widened with cvt.rn.f16x2.e4m3x2 and used as the A
// fragment of S^T = K Q^T under the k <-> d order (2qd+e <-> 4qd+e,
// 2qd+8+e <-> 4qd+2+e), with Q^T's fragments loaded in the same order. V goes
// through a transposed byte ldmatrix (16 x 16 codes per tile): each thread
// gets one d of 4 consecutive tokens, whose widened pairs are the A fragment
// of O^T += V^T P^T directly, under a permuted token order (k 2qd+e <-> token
// 4qd+e, 2qd+8+e <-> 4qd+2+e) that the S^T rows -- K's ldmatrix row addresses
// -- and so P^T follow; P enters that product as one fp16 value
// (11 significant bits against bf16's 8, so no P_lo term). The scales
// multiply the scores and the output. The fused step quantises the appended
// row (x / scale, nearest-even, saturating) with cvt.rn.satfinite.e4m3x2.f32.
//
// Safety: every mbarrier wait is bounded; a wait that gives up sets
// KF_DEVERR_TIMEOUT and the CTA stops. Out-of-range table entries are
// redirected to block 0 and reported. V rows past the context end in a
// partial last tile are zeroed in shared memory before use (their scores are
// masked to -inf, but 0 * NaN would still poison the product).
#pragma once

#include <cuda.h>
#include <math.h>
#include <stdlib.h>

#include <atomic>

#include "kf_internal.cuh"

namespace kf {
namespace tc {

constexpr int kTok = 16;              // tokens per stage
constexpr uint32_t kMaxSpins = 1u << 22;
constexpr float kRescaleSlack = 8.f;  // log2 of the largest unnormalised p

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete: at most `limit` polls
// (each try_wait returns after at most a hardware time slice), then false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit = kMaxSpins) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, int w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Two 16x16 tiles of bytes, transposed: lanes 0-15 / 16-31 give the 16 row
// addresses of tile 0 / 1; lane 4g + q receives, of tile i, rows 4q .. 4q+3 of
// column g in r[2i] and of column g + 8 in r[2i+1] (byte j = row 4q + j).
__device__ __forceinline__ void ldsm_b8_x2_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// FP8 stages take the 16 tokens of a stage in the order that a transposed byte
// ldmatrix of V delivers them: MMA k index (and S^T row) 2q + j is token
// 4q + j, and 2q + 8 + j is token 4q + 2 + j (q < 4, j < 2).
__device__ __forceinline__ int fp8_token(int r) {
    return r < 8 ? 4 * (r >> 1) + (r & 1) : 4 * ((r - 8) >> 1) + 2 + (r & 1);
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats to a bf16 pair (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
// Extra inputs/outputs of the single-launch decode step.
struct StepParams {
    const uint16_t *k_new;   // bf16 [B, Hkv, D]
    const uint16_t *v_new;
    void *k_cache;           // the caches (bf16 or E4M3), written at the appended position
    void *v_cache;
    float *ws_o;             // workspace: partials [S, B, Hq, D]
    float *ws_lse;           //            lse     [S, B, Hq]
    unsigned int *counters;  //            [B, Hkv], zero between steps
    void *out;               // final [B, Hq, D] (f32 or bf16)
    float *lse_out;          // final [B, Hq], or null
    int out_dtype;
    const float *ex_o;       // extra partials, merged with the splits': [n_ex, B, Hq, D]
    const float *ex_lse;     //                                         [n_ex, B, Hq]
    int n_ex;
};

// Shared-memory geometry. bf16 caches: boxes of 64 elements (128-byte rows),
// D/64 boxes per operand. FP8 caches: one box of D one-byte elements per
// operand (128- or 64-byte rows).
template <int D, int HPC, int NS, bool KV8>
struct TcShape {
    static constexpr int kRowBytes = KV8 ? D : 128;          // bytes of one box row
    static constexpr int kHalves = KV8 ? 1 : D / 64;          // boxes per operand
    static constexpr int kBoxBytes = kRowBytes * kTok * HPC;  // one box
    static constexpr int kStageBytes = 2 * kHalves * kBoxBytes;
    static constexpr int kSmemBytes = NS * kStageBytes + NS * 16 + 1024;
    static constexpr int kThreads = 32 * (HPC + 1);
};

// Byte offset of 16-byte chunk `c` of row t inside a swizzled box with
// rows of RB bytes (TMA 128-byte swizzle for RB = 128, 64-byte for RB = 64):
// the chunk index is XOR-ed with address bits 7.. of the row.
template <int RB>
__device__ __forceinline__ uint32_t swz(int t, int c) {
    return RB == 128 ? (uint32_t)(t * 128 + ((c ^ (t & 7)) << 4))
                     : (uint32_t)(t * 64 + ((c ^ ((t >> 1) & 3)) << 4));
}

// Two E4M3 codes (low byte first) to an fp16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    const unsigned short h = (unsigned short)(two & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

// Two floats to an fp16 pair (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float f16_lo(uint32_t w) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(w));
    return f;
}

__device__ __forceinline__ float f16_hi(uint32_t w) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(w));
    return f;
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats to two E4M3 codes (`lo` in the low byte), nearest-even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Number of splits of a request with L tokens that hold at least one token.
__device__ __forceinline__ int nonempty_splits(const DecodeParams &p, int64_t L) {
    const int64_t nb = (L + p.block_size - 1) / p.block_size;
    int64_t n = (nb + p.chunk_blocks - 1) / p.chunk_blocks;
    return (int)(n < p.num_splits ? n : p.num_splits);
}

// Last-arriving CTA of a (request, KV-head group): LSE merge of the n_ne
// partials in the workspace into the final rows (same arithmetic as the merge
// kernel). Uses the shared-memory ring, which is idle by now.
template <int D, int R>
__device__ void merge_group(const DecodeParams &p, const StepParams &sp, int b, int row_first,
                            int n_sp, float *sm) {
    // partial s < n_sp is a split's (workspace), s >= n_sp the extra slot s - n_sp
    const int n_ne = n_sp + sp.n_ex;
    const int64_t rows = (int64_t)p.batch * p.num_q_heads;
    auto lse_of = [&](int s) { return s < n_sp ? sp.ws_lse + (int64_t)s * rows : sp.ex_lse + (int64_t)(s - n_sp) * rows; };
    float *sm_w = sm;                 // [n_ne][R] lse, then weights
    float *sm_m = sm + n_ne * R;      // [R] row max
    float *sm_sum = sm_m + R;         // [R] sum of weights
    const int nt = blockDim.x, tid = threadIdx.x;
    for (int i = tid; i < n_ne * R; i += nt) {
        const int s = i / R, r = i % R;
        sm_w[i] = __ldcg(lse_of(s) + (int64_t)b * p.num_q_heads + row_first + r);
    }
    __syncthreads();
    for (int r = tid; r < R; r += nt) {
        float M = -INFINITY;
        for (int s = 0; s < n_ne; ++s) M = fmaxf(M, sm_w[s * R + r]);
        float sum = 0.f;
        for (int s = 0; s < n_ne; ++s) {
            const float w = sm_w[s * R + r] == -INFINITY ? 0.f : expf(sm_w[s * R + r] - M);
            sm_w[s * R + r] = w;
            sum += w;
        }
        sm_m[r] = M;
        sm_sum[r] = sum;
    }
    __syncthreads();
    // each thread owns up to U (row, 4-column) units and walks the partials in
    // batches of SB, keeping U*SB 16-byte loads in flight before it sums them
    constexpr int C = D / 4;
    constexpr int U = 4, SB = 4;
    for (int u0 = tid; u0 < R * C; u0 += nt * U) {
        float4 acc[U];
        int64_t rowu[U];
        bool live[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int u = u0 + k * nt;
            live[k] = u < R * C;
            rowu[k] = (int64_t)b * p.num_q_heads + row_first + (live[k] ? u / C : 0);
            acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // partials [first, first + n) at `obase` (workspace or extra slots); their
        // weights sit at sm_w[(w0 + s) * R + row]
        auto accumulate = [&](const float *obase, int n, int w0) {
            for (int s0 = 0; s0 < n; s0 += SB) {
                float4 o[SB][U];
#pragma unroll
                for (int j = 0; j < SB; ++j)
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const int u = u0 + k * nt;
                        o[j][k] = (live[k] && s0 + j < n)
                                      ? __ldcg(reinterpret_cast<const float4 *>(
                                                   obase + ((int64_t)(s0 + j) * rows + rowu[k]) * D) + u % C)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                for (int j = 0; j < SB; ++j)
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const int u = u0 + k * nt;
                        const float w = (live[k] && s0 + j < n) ? sm_w[(w0 + s0 + j) * R + u / C] : 0.f;
                        // a zero weight (an empty extra slot) drops o whatever its bits
                        if (w != 0.f) {
                            acc[k].x = fmaf(w, o[j][k].x, acc[k].x);
                            acc[k].y = fmaf(w, o[j][k].y, acc[k].y);
                            acc[k].z = fmaf(w, o[j][k].z, acc[k].z);
                            acc[k].w = fmaf(w, o[j][k].w, acc[k].w);
                        }
                    }
            }
        };
        accumulate(sp.ws_o, n_sp, 0);
        if (sp.n_ex > 0) accumulate(sp.ex_o, sp.n_ex, n_sp);
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (!live[k]) continue;
            const int u = u0 + k * nt;
            const int r = u / C, c = u % C;
            const int64_t row = rowu[k];
            const float inv = 1.f / sm_sum[r];
            float4 a = acc[k];
            a.x *= inv; a.y *= inv; a.z *= inv; a.w *= inv;
            if (sp.out_dtype == KF_F32) {
                reinterpret_cast<float4 *>(static_cast<float *>(sp.out) + row * D)[c] = a;
            } else {
                uint2 v;
                v.x = pack_bf16(a.x, a.y);
                v.y = pack_bf16(a.z, a.w);
                reinterpret_cast<uint2 *>(static_cast<uint16_t *>(sp.out) + row * D)[c] = v;
            }
            if (c == 0 && sp.lse_out) sp.lse_out[row] = sm_m[r] + logf(sm_sum[r]);
        }
    }
}

// ---------------------------------------------------------------------------
// Consumer-warp pieces (one warp = one KV head and its G query heads), shared
// by the split-rule kernel below and the balanced-schedule kernel
// ---------------------------------------------------------------------------

// Q^T of the warp's G query heads as B fragments, in two steps so that the
// loads can be issued early: load_q_raw reads this lane's words of query head
// g = lane/4 of the group (q_row; read only for g < G, rows g >= G are zero)
// into qb as bf16 pairs, b0 = Q[g][16ks + 2qd .. +1], b1 = Q[g][16ks + 8 +
// 2qd .. +1]; FP8 caches take the k index of a step to d = 16ks + 4qd +
// {0,1} / {2,3} (the order in which ldmatrix delivers the cache bytes; see
// stage_math). prep_q then, for FP8 caches, scales q by an exact power of two
// 2^qe that puts the warp's largest |q| in [2^14, 2^15), so its 8 significant
// bits are exact in fp16, and returns 2^-qe (1 for bf16).
template <int D, int G, bool KV8>
__device__ __forceinline__ void load_q_raw(const uint16_t *q_row, int lane, uint32_t (&qb)[D / 16][2]) {
    constexpr int KS = D / 16;
    const int g = lane >> 2, qd = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) qb[ks][0] = qb[ks][1] = 0u;
    if (g < G) {
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(q_row);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (KV8) {
                const uint2 v = reinterpret_cast<const uint2 *>(qrow)[4 * ks + qd];
                qb[ks][0] = v.x;
                qb[ks][1] = v.y;
            } else {
                qb[ks][0] = qrow[8 * ks + qd];
                qb[ks][1] = qrow[8 * ks + 4 + qd];
            }
        }
    }
}

template <int D, bool KV8>
__device__ __forceinline__ float prep_q(uint32_t (&qb)[D / 16][2]) {
    constexpr int KS = D / 16;
    float qe_scale = 1.f;
    if (KV8) {
        float mx = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_lo(qb[ks][0])), fabsf(bf16_hi(qb[ks][0]))),
                                 fmaxf(fabsf(bf16_lo(qb[ks][1])), fabsf(bf16_hi(qb[ks][1])))));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const int qe = (mx > 0.f && isfinite(mx)) ? 14 - ilogbf(mx) : 0;
        const float up = ldexpf(1.f, qe);
        qe_scale = ldexpf(1.f, -qe);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = pack_f16(bf16_lo(qb[ks][0]) * up, bf16_hi(qb[ks][0]) * up);
            qb[ks][1] = pack_f16(bf16_lo(qb[ks][1]) * up, bf16_hi(qb[ks][1]) * up);
        }
    }
    return qe_scale;
}

// The step's append inside a stage: KV head hkv's new K/V row of request b
// goes to slot t of the stage and to the cache at position p_new (FP8 caches:
// 16 bf16 values per lane quantised to E4M3 codes of x / scale).
template <class Sh, int D, bool KV8>
__device__ __forceinline__ void append_row(const DecodeParams &p, const StepParams &sp, int b, int hkv,
                                           int64_t p_new, int t, uint32_t kbuf, uint32_t vbuf, int lane) {
    constexpr int RB = Sh::kRowBytes;
    constexpr int CH = KV8 ? D / 16 : D / 8;  // 16-byte chunks per row
    constexpr int CPB = RB / 16;               // chunks per box row
    if (lane >= 2 * CH) return;
    const bool is_v = lane >= CH;
    const int c = is_v ? lane - CH : lane;
    const uint16_t *src = (is_v ? sp.v_new : sp.k_new) + ((int64_t)b * p.num_kv_heads + hkv) * D;
    uint4 val;
    if (KV8) {
        const float s_q = is_v ? p.v_scale[hkv] : p.k_scale[hkv];
        const uint4 x0 = reinterpret_cast<const uint4 *>(src)[2 * c];
        const uint4 x1 = reinterpret_cast<const uint4 *>(src)[2 * c + 1];
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t o8[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t lo = f32x2_to_e4m3x2(bf16_lo(w[2 * e]) / s_q, bf16_hi(w[2 * e]) / s_q);
            const uint32_t hi = f32x2_to_e4m3x2(bf16_lo(w[2 * e + 1]) / s_q, bf16_hi(w[2 * e + 1]) / s_q);
            o8[e] = lo | (hi << 16);
        }
        val = make_uint4(o8[0], o8[1], o8[2], o8[3]);
    } else {
        val = reinterpret_cast<const uint4 *>(src)[c];
    }
    const uint32_t a = (is_v ? vbuf : kbuf) + (c / CPB) * Sh::kBoxBytes + swz<RB>(t, c % CPB);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(val.x), "r"(val.y), "r"(val.z),
                 "r"(val.w)
                 : "memory");
    const int64_t phys = physical_block(p, b, p_new / p.block_size);
    const int64_t off = ((phys * p.block_size + p_new % p.block_size) * p.num_kv_heads + hkv) *
                        (int64_t)(D * (KV8 ? 1 : 2));  // bytes
    reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(is_v ? sp.v_cache : sp.k_cache) + off)[c] = val;
}

// Zero this head's V rows past the end of a partial stage (whole rows, any
// swizzle): their scores are -inf, but 0 * NaN would still poison O.
template <class Sh>
__device__ __forceinline__ void zero_v_tail(uint32_t vbuf, int nvalid, int lane) {
    constexpr int RB = Sh::kRowBytes;
    constexpr int CPB = RB / 16;
    for (int idx = lane; idx < (kTok - nvalid) * CPB * Sh::kHalves; idx += 32) {
        const int hf = idx / ((kTok - nvalid) * CPB);
        const int rem = idx % ((kTok - nvalid) * CPB);
        const int t = nvalid + rem / CPB, c = rem % CPB;
        const uint32_t a = vbuf + hf * Sh::kBoxBytes + t * RB + c * 16;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
    }
}

// One 16-token stage of one warp: S^T = K Q^T, the online-softmax update of
// (m_run, l_acc, oacc) with tokens >= nvalid masked, and O^T += V^T P^T.
// kbuf / vbuf are this head's 16 rows of the stage's K and V boxes.
template <class Sh, int D, bool KV8>
__device__ __forceinline__ void stage_math(uint32_t kbuf, uint32_t vbuf, int nvalid,
                                           const uint32_t (&qb)[D / 16][2], float sl2,
                                           float (&oacc)[D / 16][4], float (&m_run)[2],
                                           float (&l_acc)[2], int lane) {
    constexpr int RB = Sh::kRowBytes;
    constexpr int KS = D / 16;
    const int g = lane >> 2;
    const int lj = lane >> 3, lr = lane & 7;  // ldmatrix: matrix lj, row lr

    // S^T = K Q^T : rows = tokens, cols = query heads of the group
    // two accumulators (even / odd k-steps) halve the dependent MMA chain
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    float sd[4] = {0.f, 0.f, 0.f, 0.f};
    if (KV8) {
        // one ldmatrix.x4 = 16 tokens x 32 d codes; each 32-bit register holds 4
        // consecutive codes of one token, widened to the A fragment of k-step
        // (low pair -> k 2qd..+1, high pair -> k 2qd+8..+9)
        // (S^T row r is token fp8_token(r), the order V's fragments arrive in)
        const int t = fp8_token(lr + ((lj & 1) << 3));
#pragma unroll
        for (int kk = 0; kk < KS / 2; ++kk) {
            const int chunk = 2 * kk + (lj >> 1);
            uint32_t fr[4];
            ldsm_x4(kbuf + swz<RB>(t, chunk), fr);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t ra = fr[2 * h2], rb = fr[2 * h2 + 1];
                const uint32_t af[4] = {e4m3x2_to_f16x2(ra), e4m3x2_to_f16x2(rb),
                                        e4m3x2_to_f16x2(ra >> 16), e4m3x2_to_f16x2(rb >> 16)};
                mma_f16(h2 ? sd : sc, af, qb[2 * kk + h2][0], qb[2 * kk + h2][1]);
            }
        }
    } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int t = lr + ((lj & 1) << 3);
            const int chunk = 2 * ks + (lj >> 1);
            const uint32_t a = kbuf + (chunk >> 3) * Sh::kBoxBytes + swz<128>(t, chunk & 7);
            uint32_t fr[4];
            ldsm_x4(a, fr);
            mma_bf16((ks & 1) ? sd : sc, fr, qb[ks][0], qb[ks][1]);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[e] += sd[e];
    // scores in base 2, masked past the end; sc[0..1] row g, sc[2..3] row g+8
    // (tokens g, g + 8; FP8: fp8_token of them)
    const int tok0 = KV8 ? fp8_token(g) : g, tok1 = KV8 ? fp8_token(g + 8) : g + 8;
    const float x0 = tok0 < nvalid ? sc[0] * sl2 : -INFINITY;
    const float x1 = tok0 < nvalid ? sc[1] * sl2 : -INFINITY;
    const float x2 = tok1 < nvalid ? sc[2] * sl2 : -INFINITY;
    const float x3 = tok1 < nvalid ? sc[3] * sl2 : -INFINITY;
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
    const float p0 = exp2f(x0 - m_run[0]), p1 = exp2f(x1 - m_run[1]);
    const float p2 = exp2f(x2 - m_run[0]), p3 = exp2f(x3 - m_run[1]);
    l_acc[0] += p0 + p2;
    l_acc[1] += p1 + p3;
    // bf16 caches: P = P_hi + P_lo, both bf16, two MMAs: the PV product carries
    // ~16 bits of P; FP8 caches: P in fp16, one MMA
    uint32_t h01, h23, r01 = 0u, r23 = 0u;
    if (KV8) {
        // fp16 P (11 significant bits): one MMA; a weight is off by at most
        // 2^-11 relative, an output by at most 2^-11 max|v|
        h01 = pack_f16(p0, p1);
        h23 = pack_f16(p2, p3);
    } else {
        h01 = pack_bf16(p0, p1);
        h23 = pack_bf16(p2, p3);
        r01 = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        r23 = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
    }
    const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);  // P^T, tokens 0-7 / 8-15
    const uint32_t bl0 = KV8 ? 0u : movmatrix_trans(r01), bl1 = KV8 ? 0u : movmatrix_trans(r23);

    // O^T += V^T P^T : rows = d, cols = query heads
    if (KV8) {
        // V codes through a transposed byte ldmatrix, two 16-d tiles at a time:
        // this lane gets d = g and g + 8 of tokens 4qd .. 4qd+3, whose widened
        // pairs are the A fragment of O^T (rows d in order) at k 2qd.. / 2qd+8..
        // under the token order of fp8_token
#pragma unroll
        for (int mm = 0; mm < KS / 2; ++mm) {
            uint32_t fr[4];
            ldsm_b8_x2_trans(vbuf + swz<RB>(lane & 15, 2 * mm + (lane >> 4)), fr);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t ra = fr[2 * h2], rb = fr[2 * h2 + 1];
                const uint32_t af[4] = {e4m3x2_to_f16x2(ra), e4m3x2_to_f16x2(rb), e4m3x2_to_f16x2(ra >> 16),
                                        e4m3x2_to_f16x2(rb >> 16)};
                mma_f16(oacc[2 * mm + h2], af, bh0, bh1);
            }
        }
    } else {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int t = lr + ((lj >> 1) << 3);
            const int chunk = 2 * mt + (lj & 1);
            const uint32_t a = vbuf + (chunk >> 3) * Sh::kBoxBytes + swz<128>(t, chunk & 7);
            uint32_t fr[4];
            ldsm_x4_trans(a, fr);
            mma_bf16(oacc[mt], fr, bh0, bh1);
            mma_bf16(oacc[mt], fr, bl0, bl1);
        }
    }
}

// End of a warp's token range: l summed over the 8 token lanes, o = O * vsc / l
// and lse = (m + log2 l) ln 2 for the G query heads. Rows go to o_dst (f32,
// row stride D) at row prow + n, or, with o_dst null, to the final output
// (f32 or bf16); lse to l_dst[prow + n] unless l_dst is null.
template <int D, int G, bool KV8>
__device__ __forceinline__ void write_rows(const float (&oacc)[D / 16][4], float (&l_acc)[2],
                                           const float (&m_run)[2], float vsc, int64_t prow,
                                           float *o_dst, void *out, int out_dtype, float *l_dst,
                                           int lane) {
    constexpr int KS = D / 16;
    const int g = lane >> 2, qd = lane & 3;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_acc[0] += __shfl_xor_sync(0xffffffffu, l_acc[0], off);
        l_acc[1] += __shfl_xor_sync(0xffffffffu, l_acc[1], off);
    }
    const int n0 = 2 * qd, n1 = 2 * qd + 1;
    const float inv0 = vsc / l_acc[0], inv1 = vsc / l_acc[1];
    const float lse0 = (m_run[0] + log2f(l_acc[0])) * 0.6931471805599453f;
    const float lse1 = (m_run[1] + log2f(l_acc[1])) * 0.6931471805599453f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        // rows of O^T held by this thread: d = 16mt + g and + 8
        const int d0 = 16 * mt + g;
        const int d1 = d0 + 8;
        const float v00 = oacc[mt][0] * inv0, v01 = oacc[mt][2] * inv0;
        const float v10 = oacc[mt][1] * inv1, v11 = oacc[mt][3] * inv1;
        if (o_dst != nullptr) {
            if (n0 < G) {
                o_dst[(prow + n0) * D + d0] = v00;
                o_dst[(prow + n0) * D + d1] = v01;
            }
            if (n1 < G) {
                o_dst[(prow + n1) * D + d0] = v10;
                o_dst[(prow + n1) * D + d1] = v11;
            }
        } else if (out_dtype == KF_F32) {
            float *dst = static_cast<float *>(out);
            if (n0 < G) {
                dst[(prow + n0) * D + d0] = v00;
                dst[(prow + n0) * D + d1] = v01;
            }
            if (n1 < G) {
                dst[(prow + n1) * D + d0] = v10;
                dst[(prow + n1) * D + d1] = v11;
            }
        } else {
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(out);
            if (n0 < G) {
                dst[(prow + n0) * D + d0] = __float2bfloat16_rn(v00);
                dst[(prow + n0) * D + d1] = __float2bfloat16_rn(v01);
            }
            if (n1 < G) {
                dst[(prow + n1) * D + d0] = __float2bfloat16_rn(v10);
                dst[(prow + n1) * D + d1] = __float2bfloat16_rn(v11);
            }
        }
    }
    if (g == 0 && l_dst != nullptr) {
        if (n0 < G) l_dst[prow + n0] = lse0;
        if (n1 < G) l_dst[prow + n1] = lse1;
    }
}

// FUSED = false: one split's partial into out_partial (empty split -> 0, -inf).
// FUSED = true: the whole decode step. ctx_lens are the pre-append lengths;
// CTAs of empty splits exit at once; the tail split appends the new K/V row;
// a request with one non-empty split writes its final rows directly, others
// go through the workspace and the last CTA merges.
template <int D, int HPC, int G, int NS, bool FUSED, bool KV8>
// (FP8 caches with up to 4 KV heads per CTA: three CTAs per SM is the design --
// a 64 KiB ring each -- so registers are capped for it)
__global__ void __launch_bounds__(TcShape<D, HPC, NS, KV8>::kThreads, (KV8 && HPC <= 4) ? 3 : 1)
decode_tc_kernel(const DecodeParams p, const StepParams sp, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v) {
    using Sh = TcShape<D, HPC, NS, KV8>;
    constexpr int RB = Sh::kRowBytes;
    constexpr int KS = D / 16;  // k-steps of Q.K and m-tiles of O^T

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128B swizzle wants 1024-aligned boxes
    const uint32_t bars = base + NS * Sh::kStageBytes;  // full[NS] then empty[NS]

    const int s = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = hg * HPC;
    const int Hq = p.num_q_heads;
    const bool report = threadIdx.x == 0 && s == 0 && hg == 0;

    // Loads that do not depend on the context length go out first, so that
    // their latencies overlap that of the length: the producer's first 32 table
    // entries (a split starts at logical block s * chunk_blocks), the
    // consumers' query rows and, for FP8 caches, their KV head's scales.
    int64_t tab_base = -1;
    int32_t tab_ent = -1;
    const int g = lane >> 2;
    const int qd = lane & 3;
    const int hkv = h0 + (warp < HPC ? warp : 0);
    const int hq = hkv * G;  // first query head of a consumer warp's KV head
    uint32_t qb[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) qb[ks][0] = qb[ks][1] = 0u;
    float k_sc = 1.f, v_sc = 1.f;
    if (warp == HPC) {
        tab_base = (int64_t)s * p.chunk_blocks;
        const int64_t e = tab_base + lane;
        tab_ent = e < p.bt_stride ? p.block_tables[(int64_t)b * p.bt_stride + e] : -1;
    } else {
        if (g < G) {
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + ((int64_t)b * Hq + hq + g) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (KV8) {
                    const uint2 v = reinterpret_cast<const uint2 *>(qrow)[4 * ks + qd];
                    qb[ks][0] = v.x;
                    qb[ks][1] = v.y;
                } else {
                    qb[ks][0] = qrow[8 * ks + qd];
                    qb[ks][1] = qrow[8 * ks + 4 + qd];
                }
            }
        }
        if (KV8) {
            k_sc = p.k_scale[hkv];
            v_sc = p.v_scale[hkv];
        }
    }

    // token range of this split; in the fused step the range covers the new token too
    int64_t p_new = -1;  // position the step appends (fused only)
    int n_ne = 0;
    SplitRange r;
    if (FUSED) {
        const int64_t before = p.ctx_lens[b];
        const int64_t cap = (int64_t)p.bt_stride * p.block_size;
        int64_t L = before + 1;
        if (before < 0 || L > cap) {
            if (report) raise_error(p.err, before < 0 ? KF_DEVERR_CONTEXT_LEN : KF_DEVERR_APPEND_POS);
            L = before < 0 ? 0 : cap;
        } else {
            p_new = before;
        }
        if (L > p.max_context_len && report) raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
        n_ne = nonempty_splits(p, L);
        if (s >= n_ne) return;  // no tokens: nothing written, not counted
        const int64_t span = (int64_t)p.chunk_blocks * p.block_size;
        r.t_begin = (int64_t)s * span;
        r.t_end = r.t_begin + span < L ? r.t_begin + span : L;
    } else {
        r = split_range(p, b, s, report);
    }
    const int64_t row0 = ((int64_t)s * p.batch + b) * Hq + (int64_t)h0 * G;  // first partial row
    if (!FUSED && (r.t_begin >= r.t_end || (*(volatile unsigned int *)p.err & KF_DEVERR_TIMEOUT))) {
        for (int i = threadIdx.x; i < HPC * G * D; i += blockDim.x) p.out_partial[row0 * D + i] = 0.f;
        for (int i = threadIdx.x; i < HPC * G; i += blockDim.x) p.lse_partial[row0 + i] = -INFINITY;
        return;
    }
    const int64_t sb0 = r.t_begin / kTok;
    const int n_sub = (int)((r.t_end + kTok - 1) / kTok - sb0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bars + 8 * i, 1);              // full: producer's expect_tx arrival
            mbar_init(bars + 8 * (NS + i), HPC);     // empty: one arrival per consumer warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    bool ok = true;
    if (warp == HPC) {
        // ------------------------------ producer ------------------------------
        // The whole warp walks the stages: table entries come 32 at a time (one
        // coalesced load, lane e holds logical block base + e), so a TMA issue
        // never waits on a dependent load; lane 0 waits for slots and issues.
        const int bs_shift = block_shift(p.block_size);
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
                    tma_load_4d(dst + hf * Sh::kBoxBytes, &tmap_k, 64 * hf, slot, h0, (int)phys, full);
                    tma_load_4d(dst + (Sh::kHalves + hf) * Sh::kBoxBytes, &tmap_v, 64 * hf, slot, h0,
                                (int)phys, full);
                }
            }
        }
        if (!FUSED) return;
    } else {
        // ------------------------------- consumers --------------------------------
        // Q^T as B fragments (loaded above as load_q_raw does; prep_q's scaling
        // written out here: as calls the FP8 instantiation with three CTAs per SM
        // spills a register)
        // FP8 cache: the products run in fp16. q (bf16, 8 significant bits) goes to
        // fp16 exactly after an exact power-of-two scaling 2^qe that puts the
        // warp's largest |q| in [2^14, 2^15); 2^-qe goes into the score scale
        float qe_scale = 1.f;
        if (KV8) {
            float mx = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_lo(qb[ks][0])), fabsf(bf16_hi(qb[ks][0]))),
                                     fmaxf(fabsf(bf16_lo(qb[ks][1])), fabsf(bf16_hi(qb[ks][1])))));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const int qe = (mx > 0.f && isfinite(mx)) ? 14 - ilogbf(mx) : 0;
            const float up = ldexpf(1.f, qe);
            qe_scale = ldexpf(1.f, -qe);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qb[ks][0] = pack_f16(bf16_lo(qb[ks][0]) * up, bf16_hi(qb[ks][0]) * up);
                qb[ks][1] = pack_f16(bf16_lo(qb[ks][1]) * up, bf16_hi(qb[ks][1]) * up);
            }
        }
        // per-head dequantisation scales of an FP8 cache
        const float sl2 = KV8 ? p.scale_log2 * k_sc * qe_scale : p.scale_log2;
        const float vsc = KV8 ? v_sc : 1.f;

        float oacc[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_acc[2] = {0.f, 0.f};
        const uint32_t head_off = warp * (kTok * RB);  // this head's 16 rows in a box

        for (int i = 0; i < n_sub; ++i) {
            const int st = i % NS;
            if (!mbar_wait(bars + 8 * st, (i / NS) & 1)) {
                raise_error(p.err, KF_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            const uint32_t kbuf = base + st * Sh::kStageBytes + head_off;
            const uint32_t vbuf = kbuf + Sh::kHalves * Sh::kBoxBytes;
            const int64_t t_base = (sb0 + i) * kTok;
            const int64_t rem_tok = r.t_end - t_base;
            const int nvalid = rem_tok < kTok ? (int)rem_tok : kTok;
            bool wrote_smem = false;
            if (FUSED && p_new >= t_base && p_new < t_base + kTok) {
                append_row<Sh, D, KV8>(p, sp, b, hkv, p_new, (int)(p_new - t_base), kbuf, vbuf, lane);
                wrote_smem = true;
                __syncwarp();
            }
            if (nvalid < kTok) {
                zero_v_tail<Sh>(vbuf, nvalid, lane);
                wrote_smem = true;
                __syncwarp();
            }
            stage_math<Sh, D, KV8>(kbuf, vbuf, nvalid, qb, sl2, oacc, m_run, l_acc, lane);
            // generic smem writes above must be ordered before the next TMA into this stage
            if (wrote_smem) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (NS + st));
        }

        if (ok) {
            // destination: the partial slot, or (fused, single split) the final rows
            const bool direct = FUSED && n_ne == 1 && sp.n_ex == 0;
            const int64_t prow = direct ? (int64_t)b * Hq + (int64_t)hq
                                        : row0 + (int64_t)warp * G;  // row of query head n = 0
            float *o_dst = FUSED ? (direct ? nullptr : sp.ws_o) : p.out_partial;
            float *l_dst = FUSED ? (direct ? sp.lse_out : sp.ws_lse) : p.lse_partial;
            write_rows<D, G, KV8>(oacc, l_acc, m_run, vsc, prow, o_dst, sp.out, sp.out_dtype, l_dst, lane);
        }
        if (!FUSED) return;
    }

    // ----------------------- fused: count, last CTA merges -----------------------
    // (with extra partials even a request of one non-empty split merges: its
    // single CTA counts itself as the last)
    if (FUSED && n_ne + sp.n_ex > 1) {
        __shared__ int sm_last;
        __threadfence();  // this CTA's partial is visible before the count
        __syncthreads();
        unsigned int *ctr = sp.counters + (int64_t)b * p.num_kv_heads + hg;
        if (threadIdx.x == 0) {
            const unsigned int old = atomicAdd(ctr, 1u);
            sm_last = old == (unsigned int)(n_ne - 1);
            if (sm_last) *ctr = 0u;  // every other CTA of the group has counted: reset for the next step
        }
        __syncthreads();
        if (sm_last) {
            __threadfence();
            if (ok) merge_group<D, HPC * G>(p, sp, b, h0 * G, n_ne, reinterpret_cast<float *>(smem_raw + (base - raw)));
        }
    }
}


// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 4-D view (d, slot, head, block) of a [num_blocks, bs, Hkv, D] cache with
// boxes of (64 bf16 | D codes) x 16 slots x hpc heads x 1 block.
inline bool encode_cache_map(EncodeFn fn, CUtensorMap *map, const void *cache, int64_t num_blocks,
                             int block_size, int num_kv_heads, int head_dim, int hpc, bool kv8) {
    const cuuint64_t esz = kv8 ? 1 : 2;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)block_size,
                                (cuuint64_t)num_kv_heads, (cuuint64_t)num_blocks};
    const cuuint64_t row = (cuuint64_t)num_kv_heads * head_dim * esz;  // bytes between slots
    const cuuint64_t strides[3] = {row, (cuuint64_t)head_dim * esz, row * block_size};
    const cuuint32_t box[4] = {kv8 ? (cuuint32_t)head_dim : 64u, (cuuint32_t)kTok, (cuuint32_t)hpc, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = (kv8 && head_dim == 64) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return fn(map, kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int HPC, int G, int NS, bool FUSED, bool KV8>
cudaError_t launch_t(const DecodeParams &p, const StepParams &sp, cudaStream_t stream,
                     const CUtensorMap &mk, const CUtensorMap &mv) {
    using Sh = TcShape<D, HPC, NS, KV8>;
    // the dynamic shared-memory opt-in is per device; set it once per device
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        e = cudaFuncSetAttribute(decode_tc_kernel<D, HPC, G, NS, FUSED, KV8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    const dim3 grid(p.num_splits, p.num_kv_heads / HPC, p.batch);
    decode_tc_kernel<D, HPC, G, NS, FUSED, KV8><<<grid, Sh::kThreads, Sh::kSmemBytes, stream>>>(p, sp, mk, mv);
    return cudaGetLastError();
}

// Ring depth: about 96 KiB of loads in flight per CTA for bf16 caches (two
// CTAs per SM), 64 KiB for FP8 caches, whose per-stage instruction chain is
// longer, so that three CTAs fit per SM; 3 to 8 stages.
template <int D, int HPC, bool KV8>
constexpr int stages_for() {
    constexpr int st = TcShape<D, HPC, 1, KV8>::kStageBytes;
    constexpr int ring = KV8 ? 65536 : 98304;
    return ring / st < 3 ? 3 : (ring / st > 8 ? 8 : ring / st);
}

template <int D, int HPC, bool FUSED, bool KV8>
cudaError_t launch_g(const DecodeParams &p, const StepParams &sp, cudaStream_t stream,
                     const CUtensorMap &mk, const CUtensorMap &mv) {
    constexpr int NS = stages_for<D, HPC, KV8>();
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: return launch_t<D, HPC, 1, NS, FUSED, KV8>(p, sp, stream, mk, mv);
        case 2: return launch_t<D, HPC, 2, NS, FUSED, KV8>(p, sp, stream, mk, mv);
        case 4: return launch_t<D, HPC, 4, NS, FUSED, KV8>(p, sp, stream, mk, mv);
        case 8: return launch_t<D, HPC, 8, NS, FUSED, KV8>(p, sp, stream, mk, mv);
    }
    return cudaErrorInvalidValue;
}

// KV heads per CTA: 4 (two CTAs per SM) where it divides Hkv, measured best on
// the 32/8-head workloads; KF_TC_HPC overrides it for tuning.
inline int heads_per_cta(int num_kv_heads) {
    const char *env = getenv("KF_TC_HPC");  // read per call
    const int forced = env ? atoi(env) : 0;
    if (forced > 0 && num_kv_heads % forced == 0 && (forced == 1 || forced == 2 || forced == 4 || forced == 8))
        return forced;
    for (int h : {4, 8, 2, 1})
        if (num_kv_heads % h == 0) return h;
    return 1;
}

template <bool KV8>
int smem_bytes(int head_dim, int hpc) {
    if (head_dim == 128) {
        switch (hpc) {
            case 8: return TcShape<128, 8, stages_for<128, 8, KV8>(), KV8>::kSmemBytes;
            case 4: return TcShape<128, 4, stages_for<128, 4, KV8>(), KV8>::kSmemBytes;
            case 2: return TcShape<128, 2, stages_for<128, 2, KV8>(), KV8>::kSmemBytes;
            default: return TcShape<128, 1, stages_for<128, 1, KV8>(), KV8>::kSmemBytes;
        }
    }
    switch (hpc) {
        case 8: return TcShape<64, 8, stages_for<64, 8, KV8>(), KV8>::kSmemBytes;
        case 4: return TcShape<64, 4, stages_for<64, 4, KV8>(), KV8>::kSmemBytes;
        case 2: return TcShape<64, 2, stages_for<64, 2, KV8>(), KV8>::kSmemBytes;
        default: return TcShape<64, 1, stages_for<64, 1, KV8>(), KV8>::kSmemBytes;
    }
}

template <bool FUSED, bool KV8>
cudaError_t launch_any(const DecodeParams &p, const StepParams &sp, cudaStream_t stream, void *encode) {
    if (p.batch == 0) return cudaSuccess;
    const int hpc = heads_per_cta(p.num_kv_heads);
    EncodeFn fn = reinterpret_cast<EncodeFn>(encode);
    CUtensorMap mk, mv;
    if (!encode_cache_map(fn, &mk, p.k_cache, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim,
                          hpc, KV8) ||
        !encode_cache_map(fn, &mv, p.v_cache, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim,
                          hpc, KV8))
        return cudaErrorInvalidValue;
    if (p.head_dim == 128) {
        switch (hpc) {
            case 8: return launch_g<128, 8, FUSED, KV8>(p, sp, stream, mk, mv);
            case 4: return launch_g<128, 4, FUSED, KV8>(p, sp, stream, mk, mv);
            case 2: return launch_g<128, 2, FUSED, KV8>(p, sp, stream, mk, mv);
            default: return launch_g<128, 1, FUSED, KV8>(p, sp, stream, mk, mv);
        }
    }
    switch (hpc) {
        case 8: return launch_g<64, 8, FUSED, KV8>(p, sp, stream, mk, mv);
        case 4: return launch_g<64, 4, FUSED, KV8>(p, sp, stream, mk, mv);
        case 2: return launch_g<64, 2, FUSED, KV8>(p, sp, stream, mk, mv);
        default: return launch_g<64, 1, FUSED, KV8>(p, sp, stream, mk, mv);
    }
}

inline StepParams step_params(const StepArgs &a) {
    StepParams sp;
    sp.k_new = a.k_new;
    sp.v_new = a.v_new;
    sp.k_cache = a.k_cache;
    sp.v_cache = a.v_cache;
    sp.ws_o = a.ws_o;
    sp.ws_lse = a.ws_lse;
    sp.counters = a.counters;
    sp.out = a.out;
    sp.lse_out = a.lse_out;
    sp.out_dtype = a.out_dtype;
    sp.ex_o = a.ex_o;
    sp.ex_lse = a.ex_lse;
    sp.n_ex = a.n_ex;
    return sp;
}

}  // namespace tc
}  // namespace kf
