// kf_multiquery_tc05w.cu -- multi-query paged attention on tcgen05 with
// 128-token KV tiles and two 128-row query tiles per CTA: the same contract as
// kf_multiquery.cu, for requests with more than 128 (query, head) rows per KV
// head (the shared-prefix pass of cascade attention, long prefill chunks).
//
// What it computes: "Mathematical Formulation of Chunked Attention" of
// "Disaggregated Inference Architecture: Paged KV-Cache Tiering, Chunked
// Prefill, and Asynchronous Overlap" (ultrainstinct.tech): query j of a chunk
// of C whose tokens are the last C of the L cached ones attends to tokens
// [0, L - C + j] (causal), or all L (non-causal: cascade attention, "What
// FlashInfer brings: JIT and cascade attention", blog.lo0.es). Output: the
// split partials (o, lse).
//
// Why this shape: the 64-token-tile kernel (kf_multiquery_tc05.cu) issues
// N = 64 score MMAs, which reach two thirds of the tensor rate, and its one
// MMA thread waits on six barriers per 64 tokens, each costing a few hundred
// cycles while the MMAs' operand reads keep shared memory busy. Here per 128
// tokens the thread waits on four, and every MMA is N = 128.
//
// One CTA per (split, KV head, request x 256 query rows); 10 warps:
//   warps 0-3 / 4-7  softmax of query tile 0 / 1: thread r of warpgroup t
//                owns row r of tile t. Per KV tile it loads its 128 scores from
//                TMEM, masks them, runs the base-2 online softmax (lazy
//                rescale: the running max moves only when a tile exceeds it by
//                more than 8, and then the thread rescales its O row in TMEM),
//                and writes its 128 weights as bf16 pairs over the first 64
//                columns of its own scores in TMEM (the O rescale comes after
//                the weights, when the scores are no longer held in registers).
//   warp 8       TMA producer: one 5-D box per cache block into a ring of
//                128-token slots (5 at D = 128), K_j, V_j, K_j+1, ... in turn.
//   warp 9       MMA issuer and TMEM owner. Per KV tile j and query tile t:
//                  O_t += P_t V_{j-1}   (A = P_t from TMEM, B = V, MN-major)
//                  S_t  = Q_t K_j^T     (A = Q_t, B = K, both K-major smem)
//                issued in that order into the same TMEM columns (P over S):
//                MMAs of one thread run in issue order, so S_j is written only
//                after PV_{j-1} has read P_{j-1}. Tile 0's pair is issued as
//                soon as its softmax is done, while tile 1's softmax runs, and
//                the other way round, so the tensor core and the exponential
//                unit take turns on the two tiles.
// TMEM (512 columns): S_t / P_t at 128 t, O_t at 256 + D t.
// Barriers: full/empty per ring slot, q_ready, fin (after the last MMA), and per
// tile s_full (commit after S_t) and p_full (the softmax wrote P_t). When a
// softmax warpgroup sees s_full for tile j, PV_{j-1} of its tile has completed
// (the commit tracks every earlier MMA), so a rescale of O needs no other wait;
// the epilogue waits on fin. Every wait is bounded; a wait that gives up sets
// KF_DEVERR_TIMEOUT, and the CTA drains its copies and MMAs and frees its TMEM
// before it returns. V rows past the range in the last tile are zeroed in
// shared memory (0 * NaN would poison the product); masked scores are selected
// to -inf, never multiplied.
//
// Precision: scores and O accumulate in fp32; P enters the PV product as bf16
// (relative error <= 2^-9 per weight); l sums the unrounded fp32 weights.
#include <stdlib.h>
#include <string.h>

#include "kf_mq_tc05.cuh"

namespace kf {
namespace {

using namespace tc;
using namespace mq5;

constexpr int kRowsW = 128;  // query rows per tile
constexpr int kTileW = 128;  // tokens per KV tile

template <int D>
struct WShape {
    static constexpr int kHalves = D / 64;
    static constexpr int kQHalfBytes = kRowsW * 128;             // 16 KiB
    static constexpr int kQTileBytes = kHalves * kQHalfBytes;
    static constexpr int kQBytes = 2 * kQTileBytes;
    static constexpr int kAtomBytes = kHalves * 1024;            // 8 tokens x D
    static constexpr int kSlotBytes = kTileW / 8 * kAtomBytes;   // 128 tokens x D
    // ring: two slots feed the MMAs while the rest load (TMA latency under load
    // is about a microsecond, a tile's MMAs take under one): 5 x 32 KiB at D 128
    static constexpr int kSlots = D == 128 ? 5 : 12;
    static constexpr int kSmemBytes = kQBytes + kSlots * kSlotBytes + 1024;
    // NPW TMA producer warps: warp 8 (K items, or every item when NPW = 1) and
    // warp 10 (V items). TMA instructions issued by the lanes of one warp are
    // taken one after another (~90 cycles per box); different warps' overlap.
    static constexpr int threads(int npw) { return npw == 2 ? 352 : 320; }
    static constexpr int kProducer = 8, kIssuer = 9, kProducer2 = 10;
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
    __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + (uint32_t)D * t; }
    // one CTA per SM, so the 512-column allocation always succeeds
    static_assert(kSmemBytes > 116 * 1024 && kSmemBytes <= 227 * 1024, "one CTA per SM");
    static_assert(2 * kRowsW * D * 4 <= kSlots * kSlotBytes, "the ring holds both tiles' output rows");
};

template <int D, int G, int NPW>
__global__ void __launch_bounds__(NPW == 2 ? 352 : 320, 1)
mqw_kernel(const MqParams p, const __grid_constant__ CUtensorMap tmap_k,
           const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_q) {
    using Sh = WShape<D>;
    constexpr int NSL = Sh::kSlots;
    constexpr int KS = D / 16;  // K steps of S = Q K^T
    constexpr int KP = kTileW / 16;  // K steps of O += P V

    // barriers: full[NSL], empty[NSL], q_ready, fin, s_full[2], p_full[2], staged[2]
    __shared__ __align__(8) uint64_t bar_mem[2 * NSL + 8];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base, sKV = base + Sh::kQBytes;
    const uint32_t bars = smem_u32(bar_mem);
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (NSL + i); };
    // The ring is two rings: K tiles in slots [0, NK), V tiles in [NK, NSL). Each
    // kind's items reuse only their own slots, in order, so a producer warp that
    // runs ahead of the other can never wait on a slot whose previous item the
    // other warp has yet to issue (a parity wait would then alias).
    constexpr int NK = (NSL + 1) / 2, NV = NSL - NK;
    auto slot_of = [](int i) { return (i & 1) ? NK + (i >> 1) % NV : (i >> 1) % NK; };
    auto phase_of = [](int i) -> uint32_t { return ((i & 1) ? (i >> 1) / NV : (i >> 1) / NK) & 1; };
    const uint32_t q_ready = bars + 8u * (2 * NSL), fin = q_ready + 8;
    auto s_full = [&](int t) { return fin + 8u + 8u * t; };
    auto p_full = [&](int t) { return fin + 24u + 8u * t; };
    auto staged = [&](int t) { return fin + 40u + 8u * t; };

    const int s = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / p.q_tiles, qg = blockIdx.z % p.q_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.num_q_heads;

    // The producer's first loads go out before anything waits on the request's
    // lengths: the two tensor maps' descriptors and the 32 block-table entries
    // from the split's first block (both independent of the lengths; a cold
    // first TMA issue otherwise waits on them).
    const int bs_shift = block_shift(p.block_size);
    int64_t tab_base = -1;
    int32_t tab_ent = -1;
    const bool producer = warp == Sh::kProducer || (NPW == 2 && warp == Sh::kProducer2);
    if (producer) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
        }
        tab_base = ((int64_t)s * p.chunk_blocks * p.block_size) >> bs_shift;
        const int64_t e = tab_base + lane;
        tab_ent = e < p.bt_stride ? __ldg(p.block_tables + (int64_t)b * p.bt_stride + e) : -1;
    }

    const int q0 = p.q_start[b], q1 = p.q_start[b + 1];
    if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens) {  // rows outside q: touch nothing
        if (threadIdx.x == 0 && s == 0 && h == 0 && qg == 0) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        return;
    }
    const int64_t C = (int64_t)q1 - q0;
    int64_t L = p.ctx_lens[b];
    const int64_t cap = (int64_t)p.bt_stride * p.block_size;
    const bool report = threadIdx.x == 0 && s == 0 && h == 0 && qg == 0;
    if (L < 0 || L > cap || C < 0 || (p.causal && C > L)) {
        if (report) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        L = L < 0 ? 0 : (L > cap ? cap : L);
    }
    if (L > p.max_context_len && report) raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
    const int64_t nrow_all = C * G;
    if (threadIdx.x == 0 && s == 0 && h == 0 && qg == p.q_tiles - 1 && nrow_all > (int64_t)p.q_tiles * 2 * kRowsW)
        raise_error(p.err, KF_DEVERR_MAX_CONTEXT);  // more queries than max_query_len covers
    const int64_t row0 = (int64_t)qg * 2 * kRowsW;
    if (row0 >= nrow_all) return;  // beyond this request's queries: nothing to write
    const int64_t nrows = nrow_all - row0 < 2 * kRowsW ? nrow_all - row0 : 2 * kRowsW;
    const int nqt = (int)((nrows + kRowsW - 1) / kRowsW);  // tiles with rows (CTA-uniform)

    // token range: the split, clipped to the context and to the last row's limit
    const int64_t span = (int64_t)p.chunk_blocks * p.block_size;
    int64_t t_lo = (int64_t)s * span, t_hi = t_lo + span;
    const int64_t t_max = p.causal ? L - C + (row0 + nrows - 1) / G + 1 : L;
    if (t_hi > t_max) t_hi = t_max;
    if (t_lo > t_hi) t_lo = t_hi;

    // this thread's row (softmax threads): tile tq, row r of the tile
    const int tq = warp >> 2;
    const int r = threadIdx.x & (kRowsW - 1);
    const bool soft = warp < 8;
    const int64_t row = row0 + (int64_t)tq * kRowsW + r;
    const bool row_ok = soft && row < nrow_all;
    const int64_t qrow = row_ok ? q0 + row / G : 0;
    const int qhead = h * G + (int)(row % G);
    float *const o_row = p.out_partial + (((int64_t)s * p.num_q_tokens + qrow) * Hq + qhead) * D;
    float *const lse_row = p.lse_partial + ((int64_t)s * p.num_q_tokens + qrow) * Hq + qhead;

    if (t_lo >= t_hi || (*(volatile unsigned int *)p.err & KF_DEVERR_TIMEOUT)) {
        if (row_ok) {
            for (int i = 0; i < D; i += 4) *reinterpret_cast<float4 *>(o_row + i) = make_float4(0.f, 0.f, 0.f, 0.f);
            *lse_row = -INFINITY;
        }
        return;
    }
    const int ntiles = (int)((t_hi - t_lo + kTileW - 1) / kTileW);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSL; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        mbar_init(q_ready, 1);  // the producer's arrival, plus the Q boxes' bytes
        mbar_init(fin, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), kRowsW);
            mbar_init(staged(t), kRowsW);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == Sh::kIssuer) tc05::tmem_alloc(smem_u32(&tmem_slot), Sh::kTmemCols);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tm = tmem_slot;
    if (producer) {
        // ------------------------------ producer ------------------------------
        // The whole warp walks its items (K_j = item 2j, V_j = item 2j + 1; with
        // two producer warps each takes one kind): table entries come 32 at a
        // time (one coalesced load, lane e holds logical block base + e); lane 0
        // waits for slots and lane k issues the box of the tile's block k.
        const uint32_t box_bytes = (uint32_t)p.block_size * D * 2;
        const int ifirst = warp == Sh::kProducer ? 0 : 1, istep = NPW;
        if (warp == Sh::kProducer && lane == 0) {
            // Q first, ahead of the ring's fill: one box per query tile with rows,
            // (64 d, G heads, 128 / G tokens, D / 64 halves) landing as the tile's
            // swizzled K-major image (rows = (token, head) pairs). Rows past the
            // request's queries read the next request's q (or zeros past the
            // end); their scores are masked and their rows never stored.
            mbar_arrive_expect_tx(q_ready, (uint32_t)nqt * Sh::kQTileBytes);
            for (int t = 0; t < nqt; ++t)
                tma_load_4d(sQ + t * Sh::kQTileBytes, &tmap_q, 0, h * G,
                            (int)(q0 + (row0 + (int64_t)t * kRowsW) / G), 0, q_ready);
        }
        int last_k = -1, last_v = -1;  // this warp's last K / V tile issued
        for (int i = ifirst; i < 2 * ntiles; i += istep) {
            const int slot = slot_of(i);
            int go = 1;
            if (lane == 0) {
                go = !abort_flag && mbar_wait(empty(slot), phase_of(i) ^ 1);
                if (!go) {
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            const CUtensorMap *map = (i & 1) ? &tmap_v : &tmap_k;
            const int64_t t0 = t_lo + (int64_t)(i >> 1) * kTileW;
            const int64_t ntok = t_hi - t0 < kTileW ? t_hi - t0 : kTileW;
            const int nblk = (int)((ntok + p.block_size - 1) >> bs_shift);  // whole blocks, one box each
            if (lane == 0) mbar_arrive_expect_tx(full(slot), nblk * box_bytes);
            const int64_t lb0 = t0 >> bs_shift;
            if (tab_base < 0 || lb0 + nblk - 1 >= tab_base + 32) {
                tab_base = lb0;
                const int64_t e = lb0 + lane;
                tab_ent = e < p.bt_stride ? p.block_tables[(int64_t)b * p.bt_stride + e] : -1;
            }
            int64_t phys = __shfl_sync(0xffffffffu, tab_ent, (int)(lb0 - tab_base) + (lane < nblk ? lane : 0));
            if (lane < nblk) {
                if (phys < 0 || phys >= p.num_blocks) {
                    raise_error(p.err, KF_DEVERR_BLOCK_ID);
                    phys = 0;
                }
                tma_load_4d(sKV + slot * Sh::kSlotBytes + lane * box_bytes, map, 0, 0, h * Sh::kHalves,
                            (int)phys * (p.block_size / 8), full(slot));
            }
            __syncwarp();
            (i & 1 ? last_v : last_k) = i >> 1;
        }
        if (lane == 0) {
            // drain: the last use of each slot this warp filled has landed
            // before the CTA can exit
            for (int j = last_k - NK + 1 > 0 ? last_k - NK + 1 : 0; j <= last_k; ++j)
                if (!mbar_wait(full(slot_of(2 * j)), phase_of(2 * j))) raise_error(p.err, KF_DEVERR_TIMEOUT);
            for (int j = last_v - NV + 1 > 0 ? last_v - NV + 1 : 0; j <= last_v; ++j)
                if (!mbar_wait(full(slot_of(2 * j + 1)), phase_of(2 * j + 1))) raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
    } else if (warp == Sh::kIssuer) {
        // ------------------------------ MMA issuer -----------------------------
        // Step j: for each query tile t, once its softmax of tile j - 1 is done,
        // O_t += P_t V_{j-1} and then S_t = Q_t K_j^T (the last step has no S).
        if (lane == 0) {
            const uint32_t id_s = tc05::idesc_bf16(kRowsW, kTileW, false, false);
            const uint32_t id_o = tc05::idesc_bf16(kRowsW, D, false, true);
            const uint64_t qdesc0 = tc05::sdesc_sw128(sQ, 16, 1024);
            bool ok = mbar_wait(q_ready, 0);
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (abort_flag) {
                    ok = false;
                    break;
                }
                const bool has_s = j < ntiles, has_pv = j > 0;
                const int kslot = slot_of(2 * j), vslot = has_pv ? slot_of(2 * j - 1) : 0;
                if ((has_s && !mbar_wait(full(kslot), phase_of(2 * j))) ||
                    (has_pv && !mbar_wait(full(vslot), phase_of(2 * j - 1)))) {
                    ok = false;
                    break;
                }
                // one descriptor per operand tile, stepped in 16-byte units
                const uint64_t kd = tc05::sdesc_sw128(sKV + kslot * Sh::kSlotBytes, 16, Sh::kAtomBytes);
                const uint64_t vd = tc05::sdesc_sw128(sKV + vslot * Sh::kSlotBytes, 1024, Sh::kAtomBytes);
                for (int t = 0; t < nqt; ++t) {
                    if (has_pv && !mbar_wait(p_full(t), (j - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc05::fence_after_sync();
                    const uint32_t st = tm + Sh::col_s(t);
                    if (has_pv) {
#pragma unroll
                        for (int kk = 0; kk < KP; ++kk)
                            tc05::mma_ts(tm + Sh::col_o(t), st + 8 * kk,
                                         vd + (uint64_t)(kk * 2 * Sh::kAtomBytes / 16), id_o,
                                         (j > 1 || kk > 0) ? 1u : 0u);
                    }
                    if (has_s) {
                        const uint64_t qd = qdesc0 + (uint64_t)(t * Sh::kQTileBytes / 16);
#pragma unroll
                        for (int kk = 0; kk < KS; ++kk)
                            tc05::mma_ss(st, qd + (uint64_t)(((kk >> 2) * Sh::kQHalfBytes + 32 * (kk & 3)) / 16),
                                         kd + (uint64_t)(((kk >> 2) * 1024 + 32 * (kk & 3)) / 16), id_s,
                                         kk > 0 ? 1u : 0u);
                        tc05::commit(s_full(t));
                    }
                }
                if (!ok) break;
                if (has_s) tc05::commit(empty(kslot));
                if (has_pv) tc05::commit(empty(vslot));
            }
            if (!ok) {
                raise_error(p.err, KF_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            // every MMA issued has completed before TMEM is freed
            tc05::commit(fin);
            if (!mbar_wait(fin, 0)) raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
    } else if (warp < 8) {
        // ------------------------------- softmax --------------------------------
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int64_t lim = row_ok ? (p.causal ? L - C + row / G + 1 : L) : 0;
        const int64_t row_hi = lim < t_hi ? lim : t_hi;  // this row's tokens end here
        const float c = p.scale_log2;
        const uint32_t col_s = Sh::col_s(tq), col_o = Sh::col_o(tq);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        if (tq < nqt) {
            for (int j = 0; j < ntiles; ++j) {
                const int64_t t0 = t_lo + (int64_t)j * kTileW;
                // (the flag is read warp-uniformly: tcgen05.ld/st need the whole warp)
                if (__any_sync(0xffffffffu, abort_flag != 0) || !warp_wait(s_full(tq), j & 1)) {
                    ok = false;
                    break;
                }
                tc05::fence_after_sync();
                uint32_t sa[64], sb[64];  // scores 0-63 and 64-127 of this row
                tc05::tmem_ld64(tm + lane_base + col_s, sa);
                tc05::tmem_ld64(tm + lane_base + col_s + 64, sb);

                const int64_t ntile_tok = t_hi - t0 < kTileW ? t_hi - t0 : kTileW;
                if (ntile_tok < kTileW) {
                    // zero the V rows past the range (each tile's warps zero all of them)
                    const int slot = slot_of(2 * j + 1);
                    if (!warp_wait(full(slot), phase_of(2 * j + 1))) {
                        ok = false;
                        break;
                    }
                    const int nzr = (int)(kTileW - ntile_tok) * 8;  // 16-byte chunks per half
                    const uint32_t vb = sKV + slot * Sh::kSlotBytes;
                    for (int i = r; i < nzr * Sh::kHalves; i += kRowsW) {
                        const int hf = i / nzr, rem = i % nzr;
                        const int t = (int)ntile_tok + rem / 8;
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                         vb + (t >> 3) * Sh::kAtomBytes + hf * 1024 + (t & 7) * 128 + (rem % 8) * 16),
                                     "r"(0u)
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                }
                const int64_t nv64 = row_hi - t0;
                const int nv = nv64 <= 0 ? 0 : (nv64 >= kTileW ? kTileW : (int)nv64);
                // Fast path -- every row of the warp sees the whole tile and the
                // scale is positive: max of the raw scores (times c), one fused
                // multiply-add per weight. Otherwise scores are scaled and masked
                // to -inf first.
                const bool fast = c > 0.f && __all_sync(0xffffffffu, nv == kTileW);
                float mx = -INFINITY;
                if (fast) {
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        mx = max3f(mx, __uint_as_float(sa[i]), __uint_as_float(sa[i + 1]));
                        mx = max3f(mx, __uint_as_float(sb[i]), __uint_as_float(sb[i + 1]));
                    }
                    mx *= c;
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const float xa = i < nv ? __uint_as_float(sa[i]) * c : -INFINITY;
                        const float xb = i + 64 < nv ? __uint_as_float(sb[i]) * c : -INFINITY;
                        sa[i] = __float_as_uint(xa);
                        sb[i] = __float_as_uint(xb);
                        mx = max3f(mx, xa, xb);
                    }
                }
                const bool need = mx > m + kRescaleSlack;
                const float alpha = need ? exp2f(m - mx) : 1.f;  // m = -inf: 0
                if (need) {
                    l *= alpha;
                    m = mx;
                }
                const float mu = m == -INFINITY ? 0.f : m;
                // weights, 32 at a time, as 16 bf16 pairs over the first 64 score columns
                float2 ls = make_float2(0.f, 0.f);
                const float2 c2 = make_float2(c, c), nm = make_float2(-mu, -mu);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 32 * (q4 & 1) + 2 * i;
                        const uint32_t u0 = q4 < 2 ? sa[e] : sb[e], u1 = q4 < 2 ? sa[e + 1] : sb[e + 1];
                        float2 a;
                        if (fast) {
                            a = fma_f32x2(make_float2(__uint_as_float(u0), __uint_as_float(u1)), c2, nm);
                        } else {
                            a = make_float2(__uint_as_float(u0) - mu, __uint_as_float(u1) - mu);
                        }
                        a.x = ex2f(a.x);
                        a.y = ex2f(a.y);
                        ls = add_f32x2(ls, a);
                        pk[i] = pack_bf16(a.x, a.y);
                    }
                    tc05::tmem_st16(tm + lane_base + col_s + 16 * q4, pk);
                }
                l += ls.x + ls.y;
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    // O holds PV_0 .. PV_{j-1} (complete: s_full of tile j came after
                    // them); PV_j waits for p_full below. Done after the weights, so
                    // the scores are no longer live.
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tc05::tmem_ld32(tm + lane_base + col_o + 32 * cc, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc05::tmem_st32(tm + lane_base + col_o + 32 * cc, o);
                    }
                }
                tc05::fence_before_sync();
                mbar_arrive(p_full(tq));
            }
            if (ok && warp_wait(fin, 0)) {
                // Epilogue through shared memory (the KV ring is idle once every MMA
                // is done): each thread writes its normalised O row with 16-byte
                // chunks XOR-swizzled by row, then each warp copies whole rows out,
                // one coalesced 16-byte chunk per lane.
                tc05::fence_after_sync();
                constexpr int CH = D / 4;                       // 16-byte chunks per row
                const uint32_t stage = sKV + tq * (kRowsW * D * 4);
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tc05::tmem_ld32(tm + lane_base + col_o + 32 * cc, o);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int k = 8 * cc + i;
                        float4 v = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                               __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
                        if (!(l > 0.f)) v = make_float4(0.f, 0.f, 0.f, 0.f);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         stage + r * (D * 4) + ((k ^ (r & (CH - 1))) << 4)),
                                     "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                                     : "memory");
                    }
                }
                if (row_ok) *lse_row = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
                // this tile's rows are staged (a bounded wait: a warp that gave up
                // earlier never arrives)
                mbar_arrive(staged(tq));
                if (!warp_wait(staged(tq), 0)) {
                    if (r == 0) raise_error(p.err, KF_DEVERR_TIMEOUT);
                } else
                for (int rr = warp & 3; rr < kRowsW; rr += 4) {
                    const int64_t grow = row0 + (int64_t)tq * kRowsW + rr;
                    if (grow >= nrow_all) break;  // rows ascend: the rest are past the request
                    float *dst = p.out_partial +
                                 (((int64_t)s * p.num_q_tokens + q0 + grow / G) * Hq + h * G + (int)(grow % G)) * D;
                    for (int k = lane; k < CH; k += 32) {
                        float4 v;
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                     : "r"(stage + rr * (D * 4) + ((k ^ (rr & (CH - 1))) << 4))
                                     : "memory");
                        reinterpret_cast<float4 *>(dst)[k] = v;
                    }
                }
            } else {
                if (r == 0) raise_error(p.err, KF_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
        }
    }
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == Sh::kIssuer) {
        tc05::fence_after_sync();
        tc05::tmem_dealloc(tm, Sh::kTmemCols);
    }
}

// 4-D view of q [num_q_tokens, Hq, D] bf16: (d % 64, head, token, d / 64), box
// (64, G, 128 / G, D / 64): one query tile of one KV head's group -- 128 rows of
// (token, head) pairs, each 64-column half a 16 KiB block of 128-byte rows --
// landing in the 128-byte-swizzled K-major layout the score MMA reads.
bool encode_q_map(tc::EncodeFn fn, CUtensorMap *map, const MqParams &p) {
    const int G = p.num_q_heads / p.num_kv_heads, halves = p.head_dim / 64;
    const cuuint64_t head = (cuuint64_t)p.head_dim * 2;
    const cuuint64_t dims[4] = {64, (cuuint64_t)p.num_q_heads, (cuuint64_t)p.num_q_tokens, (cuuint64_t)halves};
    const cuuint64_t strides[3] = {head, head * p.num_q_heads, 128};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(kRowsW / G), (cuuint32_t)halves};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(p.q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G, int NPW>
cudaError_t launch_w(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mq) {
    using Sh = WShape<D>;
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        e = cudaFuncSetAttribute(mqw_kernel<D, G, NPW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch * p.q_tiles);
    mqw_kernel<D, G, NPW><<<grid, Sh::threads(NPW), Sh::kSmemBytes, stream>>>(p, mk, mv, mq);
    return cudaGetLastError();
}

// Two producer warps by default; KF_MQW_PRODUCERS = 1 selects one (read per
// call, for comparisons).
template <int D, int G>
cudaError_t launch_w(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mq) {
    const char *s = getenv("KF_MQW_PRODUCERS");
    if (s && strcmp(s, "1") == 0) return launch_w<D, G, 1>(p, stream, mk, mv, mq);
    return launch_w<D, G, 2>(p, stream, mk, mv, mq);
}

template <int D>
cudaError_t launch_w_g(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mq) {
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: return launch_w<D, 1>(p, stream, mk, mv, mq);
        case 2: return launch_w<D, 2>(p, stream, mk, mv, mq);
        case 4: return launch_w<D, 4>(p, stream, mk, mv, mq);
        case 8: return launch_w<D, 8>(p, stream, mk, mv, mq);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_multiquery_tc05w(MqParams p, cudaStream_t stream, void *encode) {
    if (p.batch == 0 || p.num_q_tokens == 0) return cudaSuccess;
    const int G = p.num_q_heads / p.num_kv_heads;
    const int64_t rows = (int64_t)p.max_query_len * G;
    p.q_tiles = (int)((rows + 2 * kRowsW - 1) / (2 * kRowsW));  // 256 rows per CTA
    if (p.q_tiles < 1) p.q_tiles = 1;
    if ((int64_t)p.batch * p.q_tiles > 65535) return cudaErrorInvalidValue;
    tc::EncodeFn fn = reinterpret_cast<tc::EncodeFn>(encode);
    CUtensorMap mk, mv;
    CUtensorMap mq;
    if (!encode_block_map(fn, &mk, p.k_cache, p) || !encode_block_map(fn, &mv, p.v_cache, p) ||
        !encode_q_map(fn, &mq, p))
        return cudaErrorInvalidValue;
    return p.head_dim == 128 ? launch_w_g<128>(p, stream, mk, mv, mq) : launch_w_g<64>(p, stream, mk, mv, mq);
}

}  // namespace kf
