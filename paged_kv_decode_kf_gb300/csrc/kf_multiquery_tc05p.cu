// kf_multiquery_tc05p.cu -- multi-query paged attention on CTA pairs
// (tcgen05.mma.cta_group::2): the same contract as kf_multiquery.cu, for head
// dimension 128 and more than 128 (query, head) rows per KV head (the
// shared-prefix pass of cascade attention, long prefill chunks).
//
// What it computes: "Mathematical Formulation of Chunked Attention" of
// "Disaggregated Inference Architecture: Paged KV-Cache Tiering, Chunked
// Prefill, and Asynchronous Overlap" (ultrainstinct.tech): query j of a chunk
// of C whose tokens are the last C of the L cached ones attends to tokens
// [0, L - C + j] (causal), or all L (non-causal: cascade attention, "What
// FlashInfer brings: JIT and cascade attention", blog.lo0.es). Output: the
// split partials (o, lse).
//
// Why pairs: an M = 128, N = 128 MMA with both operands in shared memory reads
// 8 KiB per 64 cycles, the whole 128 B/cycle an SM's shared memory delivers, so
// the one-CTA kernels (kf_multiquery_tc05w.cu) stall their tensor pipe on
// operand reads (plus the TMA's writes). Two CTAs on two SMs issuing M = 256
// MMAs together each hold half of every B operand -- 64 of a KV tile's 128
// tokens of K, 64 of V's 128 head-dimension columns -- and each SM reads only
// its half: per 128-token tile an SM reads Q (32 KiB) + half K (16 KiB) for
// the scores and half V (16 KiB) for the output, and its TMA writes 32 KiB,
// against 96 + 32 KiB for one CTA alone. Each CTA also holds only half of every
// tile, so its ring is twice as deep in tiles.
//
// One pair per (split, KV head, request x 256 query rows): CTA c of the pair
// holds rows 128 c .. 128 c + 127 of the 256 (query row-major: row = query * G
// + head within the group). 10 warps per CTA:
//   warps 0-3 / 4-7  softmax warpgroups 0 / 1: WG w handles the KV tiles
//                j = w, w + 2, ... with its own running max, sum and output
//                accumulator O_w (two interleaved halves of the token range,
//                merged in the epilogue), so one WG's exponentials overlap the
//                other's MMAs. Thread r of a WG owns row r of its CTA.
//   warp 8       TMA producer: per tile j, the K half (tokens 64 c .. 64 c + 63
//                of the tile, whole head rows) and the V half (all 128 tokens,
//                columns 64 c .. 64 c + 63), one box per cache block, into a
//                ring of 16 KiB slots (12 of them).
//   warp 9       even CTA: MMA issuer. S_j = Q K_j^T into S_{j%2}; after WG j%2
//                wrote P_j over it, O_{j%2} += P_j V_j, then S_{j+2}. Odd CTA:
//                relays the completion of its own loads to the even CTA's
//                `pfull` barriers (an mbarrier can be waited on only in its own
//                CTA). Both allocate and free the pair's TMEM.
// TMEM (512 columns): S_w / P_w at 128 w, O_w at 256 + 128 w.
//
// Synchronisation. Local barriers in each CTA: full/empty per ring slot (the
// TMA's completion; the pair MMA's commit, multicast to both CTAs), s_full per
// WG and fin (commits, multicast), and the epilogue's exchange barriers. The
// even CTA also holds q_ready and p_full per WG (arrivals of both CTAs' warps)
// and pfull per slot (the odd CTA's relay). A WG that sees s_full for its tile
// j knows PV_{j-2} -- the last MMA into its O before that tile -- has
// completed (S_j was issued after it), so it may rescale O. Every wait is
// bounded; one that gives up sets KF_DEVERR_TIMEOUT, and every path still ends
// with the issuer's fin commit and both CTAs' handshake before TMEM is freed.
// Two pair-wide collectives are hardware waits: the cluster barrier after
// barrier set-up and the pair's TMEM allocation. Both CTAs reach them on every
// path, because every decision to leave before them depends only on the pair's
// (split, head, request, row group), which the two CTAs share.
//
// V rows past the range in the last tile are zeroed in shared memory by the
// CTA that holds them (0 * NaN would poison the product); masked scores are
// selected to -inf, never multiplied.
//
// Precision: scores and O accumulate in fp32; P enters the PV product as bf16
// (relative error <= 2^-9 per weight); l sums the unrounded fp32 weights.
#include <atomic>

#include "kf_mq_tc05.cuh"

namespace kf {
namespace {

using namespace tc;
using namespace mq5;

constexpr int kRowsP = 128;  // query rows per CTA (256 per pair)
constexpr int kTileP = 128;  // tokens per KV tile
constexpr int kDP = 128;     // head dimension

struct PShape {
    static constexpr int kQHalfBytes = kRowsP * 128;  // 128 rows x 64 columns
    static constexpr int kQBytes = 2 * kQHalfBytes;
    static constexpr int kSlotBytes = 16 * 1024;  // 64 tokens x 128 d, or 128 tokens x 64 d
    static constexpr int kSlots = 12;
    static constexpr int kSmemBytes = kQBytes + kSlots * kSlotBytes + 1024;
    static constexpr int kThreads = 352;
    // TMA producers: warp 8 the K halves, warp 10 the V halves (TMA instructions
    // from one warp's lanes are taken one after another; different warps' overlap)
    static constexpr int kProducer = 8, kIssuer = 9, kProducer2 = 10;
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t col_s(int w) { return 128u * w; }
    __host__ __device__ static constexpr uint32_t col_o(int w) { return 256u + 128u * w; }
    static_assert(kSmemBytes <= 227 * 1024 - 1024, "one CTA per SM, with room for the static barriers");
    // epilogue: the staged rows (64 KiB) and the (m, l) exchange fit in the idle ring
    static_assert(kRowsP * kDP * 4 + 4 * kRowsP * 4 <= kSlots * kSlotBytes, "epilogue staging");
};

template <int G>
__global__ void __launch_bounds__(352, 1)
mqp_kernel(const MqParams p, const __grid_constant__ CUtensorMap tmap_k,
           const __grid_constant__ CUtensorMap tmap_vh) {
    using Sh = PShape;
    constexpr int NSL = Sh::kSlots;
    constexpr int D = kDP;

    // barriers: full, empty, pfull [NSL]; q_ready, fin, bye, mlx, staged; s_full[2], p_full[2]
    __shared__ __align__(8) uint64_t bar_mem[3 * NSL + 9];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base, sKV = base + Sh::kQBytes;
    const uint32_t bars = smem_u32(bar_mem);
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (NSL + i); };
    auto pfull = [&](int i) { return bars + 8u * (2 * NSL + i); };
    const uint32_t q_ready = bars + 8u * (3 * NSL), fin = q_ready + 8, bye = q_ready + 16,
                   mlx = q_ready + 24, staged = q_ready + 32;
    auto s_full = [&](int w) { return q_ready + 40u + 8u * w; };
    auto p_full = [&](int w) { return q_ready + 56u + 8u * w; };

    const uint32_t cr = cluster_rank();  // 0: the issuing (even) CTA of the pair
    const int s = blockIdx.x >> 1, h = blockIdx.y;
    const int b = blockIdx.z / p.q_tiles, qp = blockIdx.z % p.q_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.num_q_heads;

    const int bs_shift = block_shift(p.block_size);
    int64_t tab_base = -1;
    int32_t tab_ent = -1;
    const bool producer = warp == Sh::kProducer || warp == Sh::kProducer2;
    if (producer) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_vh)) : "memory");
        }
        tab_base = ((int64_t)s * p.chunk_blocks * p.block_size) >> bs_shift;
        const int64_t e = tab_base + lane;
        tab_ent = e < p.bt_stride ? __ldg(p.block_tables + (int64_t)b * p.bt_stride + e) : -1;
    }

    // Everything up to the cluster barrier depends only on (s, h, b, qp), which
    // both CTAs of the pair share: they leave together or not at all.
    const int q0 = p.q_start[b], q1 = p.q_start[b + 1];
    const bool report = threadIdx.x == 0 && cr == 0 && s == 0 && h == 0 && qp == 0;
    if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens) {  // rows outside q: touch nothing
        if (report) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        return;
    }
    const int64_t C = (int64_t)q1 - q0;
    int64_t L = p.ctx_lens[b];
    const int64_t cap = (int64_t)p.bt_stride * p.block_size;
    if (L < 0 || L > cap || C < 0 || (p.causal && C > L)) {
        if (report) raise_error(p.err, KF_DEVERR_CONTEXT_LEN);
        L = L < 0 ? 0 : (L > cap ? cap : L);
    }
    if (L > p.max_context_len && report) raise_error(p.err, KF_DEVERR_MAX_CONTEXT);
    const int64_t nrow_all = C * G;
    if (threadIdx.x == 0 && cr == 0 && s == 0 && h == 0 && qp == p.q_tiles - 1 &&
        nrow_all > (int64_t)p.q_tiles * 2 * kRowsP)
        raise_error(p.err, KF_DEVERR_MAX_CONTEXT);  // more queries than max_query_len covers
    const int64_t prow0 = (int64_t)qp * 2 * kRowsP;  // the pair's first row
    if (prow0 >= nrow_all) return;                    // beyond this request's queries
    const int64_t pnrows = nrow_all - prow0 < 2 * kRowsP ? nrow_all - prow0 : 2 * kRowsP;

    // token range: the split, clipped to the context and to the pair's last row's limit
    const int64_t span = (int64_t)p.chunk_blocks * p.block_size;
    int64_t t_lo = (int64_t)s * span, t_hi = t_lo + span;
    const int64_t t_max = p.causal ? L - C + (prow0 + pnrows - 1) / G + 1 : L;
    if (t_hi > t_max) t_hi = t_max;
    if (t_lo > t_hi) t_lo = t_hi;

    // this thread's row (softmax threads): WG wg, row r of this CTA
    const int wg = warp >> 2;
    const int r = threadIdx.x & (kRowsP - 1);
    const bool soft = warp < 8;
    const int64_t row = prow0 + (int64_t)cr * kRowsP + r;
    const bool row_ok = soft && row < nrow_all;
    const int64_t qrow = row_ok ? q0 + row / G : 0;
    const int qhead = h * G + (int)(row % G);
    float *const o_row = p.out_partial + (((int64_t)s * p.num_q_tokens + qrow) * Hq + qhead) * D;
    float *const lse_row = p.lse_partial + ((int64_t)s * p.num_q_tokens + qrow) * Hq + qhead;

    if (t_lo >= t_hi) {
        if (row_ok && wg == 0) {
            for (int i = 0; i < D; i += 4) *reinterpret_cast<float4 *>(o_row + i) = make_float4(0.f, 0.f, 0.f, 0.f);
            *lse_row = -INFINITY;
        }
        return;
    }
    const int ntiles = (int)((t_hi - t_lo + kTileP - 1) / kTileP);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSL; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
            mbar_init(pfull(i), 1);
        }
        mbar_init(q_ready, 16);  // 8 softmax warps per CTA
        mbar_init(fin, 1);
        mbar_init(bye, 1);
        mbar_init(mlx, 256);
        mbar_init(staged, 256);
        for (int w = 0; w < 2; ++w) {
            mbar_init(s_full(w), 1);
            mbar_init(p_full(w), 8);  // 4 warps per CTA
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == Sh::kIssuer) tc05::tmem_alloc2(smem_u32(&tmem_slot), Sh::kTmemCols);
    tc05::fence_before_sync();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
    tc05::fence_after_sync();
    const uint32_t tm = tmem_slot;
    const uint16_t both = 0x3;

    if (producer) {
        // ------------------------------ producers -----------------------------
        // Items i = 2j (K half of tile j; warp kProducer) and 2j + 1 (V half;
        // warp kProducer2), each warp's in order, slot i % NSL.
        const uint32_t kbox = (uint32_t)p.block_size * D * 2;   // one block, all 128 columns
        const uint32_t vbox = (uint32_t)p.block_size * 64 * 2;  // one block, 64 columns
        const int ifirst = warp == Sh::kProducer ? 0 : 1;
        int issued = 0;
        for (int i = ifirst; i < 2 * ntiles; i += 2) {
            const int slot = i % NSL;
            int go = 1;
            if (lane == 0) {
                go = !abort_flag && wait_cl(empty(slot), ((i / NSL) & 1) ^ 1);
                if (!go) {
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            const bool isv = i & 1;
            const int64_t t0 = t_lo + (int64_t)(i >> 1) * kTileP;
            int64_t first, ntok;
            if (isv) {
                first = t0;
                ntok = t_hi - t0 < kTileP ? t_hi - t0 : kTileP;
            } else {
                first = t0 + 64 * (int64_t)cr;
                ntok = t_hi - first;
                ntok = ntok < 0 ? 0 : (ntok > 64 ? 64 : ntok);
            }
            const int nblk = (int)((ntok + p.block_size - 1) >> bs_shift);  // whole blocks, one box each
            if (lane == 0) mbar_arrive_expect_tx(full(slot), nblk * (isv ? vbox : kbox));
            if (nblk > 0) {
                // table entries 32 at a time, the window starting at a tile's first
                // block (both halves of a tile then read the same window)
                const int64_t lbt = t0 >> bs_shift;
                if (tab_base < 0 || lbt < tab_base || lbt + (kTileP >> bs_shift) > tab_base + 32) {
                    tab_base = lbt;
                    const int64_t e = lbt + lane;
                    tab_ent = e < p.bt_stride ? p.block_tables[(int64_t)b * p.bt_stride + e] : -1;
                }
                const int off = (int)((first >> bs_shift) - tab_base);
                int64_t phys = __shfl_sync(0xffffffffu, tab_ent, off + (lane < nblk ? lane : 0));
                if (lane < nblk) {
                    if (phys < 0 || phys >= p.num_blocks) {
                        raise_error(p.err, KF_DEVERR_BLOCK_ID);
                        phys = 0;
                    }
                    const uint32_t dst = sKV + slot * Sh::kSlotBytes + lane * (isv ? vbox : kbox);
                    const int grp = (int)phys * (p.block_size / 8);
                    if (isv)
                        tma_load_4d(dst, &tmap_vh, 0, 0, h * 2 + (int)cr, grp, full(slot));
                    else
                        tma_load_4d(dst, &tmap_k, 0, 0, h * 2, grp, full(slot));
                }
            }
            __syncwarp();
            issued = i + 1;
        }
        if (lane == 0) {
            // drain: this warp's copies among the last NSL items have landed
            // before the CTA can exit
            for (int i = issued > NSL ? issued - NSL : 0; i < issued; ++i)
                if (((i - ifirst) & 1) == 0 && !mbar_wait(full(i % NSL), (i / NSL) & 1))
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
    } else if (warp == Sh::kIssuer && cr == 1) {
        // --------------------- relay (odd CTA): loads landed ---------------------
        if (lane == 0) {
            const uint32_t leader_pfull0 = map_to(pfull(0), 0);
            for (int i = 0; i < 2 * ntiles; ++i) {
                if (!mbar_wait(full(i % NSL), (i / NSL) & 1)) {
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
                    abort_flag = 1;
                    break;
                }
                arrive_cluster(leader_pfull0 + 8u * (i % NSL));
            }
        }
    } else if (warp == Sh::kIssuer) {
        // ------------------------- MMA issuer (even CTA) -------------------------
        if (lane == 0) {
            const uint32_t id_s = tc05::idesc_bf16(2 * kRowsP, kTileP, false, false);
            const uint32_t id_o = tc05::idesc_bf16(2 * kRowsP, D, false, true);
            const uint64_t qd = tc05::sdesc_sw128(sQ, 16, 1024);
            // item i's halves are in both CTAs
            auto ready = [&](int i) {
                const int slot = i % NSL;
                const uint32_t par = (i / NSL) & 1;
                return mbar_wait(full(slot), par) && wait_cl(pfull(slot), par);
            };
            auto issue_s = [&](int j) {  // S_j = Q K_j^T into S_{j%2}
                const int slot = (2 * j) % NSL;
                const uint64_t kd = tc05::sdesc_sw128(sKV + slot * Sh::kSlotBytes, 16, 2048);
                const uint32_t st = tm + Sh::col_s(j & 1);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc05::mma2_ss(st, qd + (uint64_t)(((kk >> 2) * Sh::kQHalfBytes + 32 * (kk & 3)) >> 4),
                                  kd + (uint64_t)(((kk >> 2) * 1024 + 32 * (kk & 3)) >> 4), id_s, kk > 0 ? 1u : 0u);
                tc05::commit2(s_full(j & 1), both);
                tc05::commit2(empty(slot), both);
            };
            auto issue_pv = [&](int j) {  // O_{j%2} += P_j V_j
                const int slot = (2 * j + 1) % NSL;
                const uint64_t vd = tc05::sdesc_sw128(sKV + slot * Sh::kSlotBytes, 1024, 1024);
                const uint32_t st = tm + Sh::col_s(j & 1);
#pragma unroll
                for (int kk = 0; kk < kTileP / 16; ++kk)
                    tc05::mma2_ts(tm + Sh::col_o(j & 1), st + 8 * kk, vd + (uint64_t)((kk * 2048) >> 4), id_o,
                                  (j >= 2 || kk > 0) ? 1u : 0u);
                tc05::commit2(empty(slot), both);
            };
            bool ok = wait_cl(q_ready, 0);
            if (ok) tc05::fence_after_sync();
            for (int j = 0; ok && j < 2 && j < ntiles; ++j) {
                ok = ready(2 * j);
                if (ok) {
                    tc05::fence_after_sync();
                    issue_s(j);
                }
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                // V_j and K_{j+2} are normally loaded long before the softmax of
                // tile j is done: wait for them first, so that PV_j and S_{j+2}
                // go out back to back once it is (their slots' previous items
                // were consumed steps ago, so these waits need nothing from step j)
                if (abort_flag || !ready(2 * j + 1) || (j + 2 < ntiles && !ready(2 * (j + 2))) ||
                    !wait_cl(p_full(j & 1), (j >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc05::fence_after_sync();
                issue_pv(j);
                if (j + 2 < ntiles) issue_s(j + 2);
            }
            if (!ok) {
                raise_error(p.err, KF_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            // every MMA issued has completed before either CTA reads O or frees TMEM
            tc05::commit2(fin, both);
            if (!mbar_wait(fin, 0)) raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
    } else {
        // ------------------------------- softmax --------------------------------
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t lead = 0;  // cluster rank of the issuing CTA
        {
            // d-half wg of this row's q -> swizzled Q (K-major, 128-byte rows, 8-row atoms)
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (qrow * Hq + qhead) * D) + 8 * wg;
            const uint32_t qb = sQ + wg * Sh::kQHalfBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = row_ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(qb + ((c ^ (r & 7)) << 4)), "r"(v.x),
                             "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) arrive_cluster(map_to(q_ready, lead));
        }
        const int64_t lim = row_ok ? (p.causal ? L - C + row / G + 1 : L) : 0;
        const int64_t row_hi = lim < t_hi ? lim : t_hi;  // this row's tokens end here
        const float c = p.scale_log2;
        const uint32_t col_s = Sh::col_s(wg), col_o = Sh::col_o(wg);
        const uint32_t my_p_full = map_to(p_full(wg), lead);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = wg, k = 0; j < ntiles; j += 2, ++k) {
            const int64_t t0 = t_lo + (int64_t)j * kTileP;
            if (__any_sync(0xffffffffu, abort_flag != 0) || !warp_wait_cl(s_full(wg), k & 1)) {
                ok = false;
                break;
            }
            tc05::fence_after_sync();
            uint32_t sa[64], sb[64];  // scores of tokens 0-63 and 64-127 of the tile
            tc05::tmem_ld64(tm + lane_base + col_s, sa);
            tc05::tmem_ld64(tm + lane_base + col_s + 64, sb);

            const int64_t ntile_tok = t_hi - t0 < kTileP ? t_hi - t0 : kTileP;
            if (ntile_tok < kTileP) {
                // zero this CTA's V rows past the range (64 columns, 128-byte rows)
                const int slot = (2 * j + 1) % NSL;
                if (!warp_wait(full(slot), ((2 * j + 1) / NSL) & 1)) {
                    ok = false;
                    break;
                }
                const int nzr = (int)(kTileP - ntile_tok) * 8;  // 16-byte chunks
                const uint32_t vb = sKV + slot * Sh::kSlotBytes;
                for (int i = r; i < nzr; i += kRowsP) {
                    const int t = (int)ntile_tok + i / 8;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vb + (t >> 3) * 1024 +
                                                                                (t & 7) * 128 + (i % 8) * 16),
                                 "r"(0u)
                                 : "memory");
                }
                fence_proxy_async_smem();
            }
            const int64_t nv64 = row_hi - t0;
            const int nv = nv64 <= 0 ? 0 : (nv64 >= kTileP ? kTileP : (int)nv64);
            const bool fast = c > 0.f && __all_sync(0xffffffffu, nv == kTileP);
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
            if (k > 0 && __any_sync(0xffffffffu, need)) {
                // O_wg holds PV of this WG's earlier tiles, all complete (the
                // last, PV_{j-2}, was issued before S_j); PV_j waits for p_full.
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
            __syncwarp();
            if (lane == 0) arrive_cluster(my_p_full);
        }
        if (!ok) {
            if (r == 0) raise_error(p.err, KF_DEVERR_TIMEOUT);
            abort_flag = 1;
        } else if (!warp_wait_cl(fin, 0)) {
            if (r == 0) raise_error(p.err, KF_DEVERR_TIMEOUT);
        } else {
            // Epilogue: merge the two WGs' halves of the token range. Both WGs
            // compute the row's factors; WG w combines and stages output columns
            // 64 w .. 64 w + 63, then all eight warps copy whole rows out.
            tc05::fence_after_sync();
            const uint32_t stage = sKV;                             // 128 rows x 512 bytes
            const uint32_t xm = sKV + kRowsP * D * 4, xl = xm + 2 * kRowsP * 4;  // (m, l) of both WGs
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(xm + (wg * kRowsP + r) * 4), "f"(m) : "memory");
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(xl + (wg * kRowsP + r) * 4), "f"(l) : "memory");
            mbar_arrive(mlx);
            if (!warp_wait(mlx, 0)) {
                if (r == 0) raise_error(p.err, KF_DEVERR_TIMEOUT);
            } else {
                float m0, m1, l0, l1;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m0) : "r"(xm + r * 4) : "memory");
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m1) : "r"(xm + (kRowsP + r) * 4) : "memory");
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(l0) : "r"(xl + r * 4) : "memory");
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(l1) : "r"(xl + (kRowsP + r) * 4) : "memory");
                const float M = fmaxf(m0, m1);
                const float a0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
                const float a1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
                const float Lsum = a0 * l0 + a1 * l1;
                const bool any = Lsum > 0.f;
                const float inv = any ? 1.f / Lsum : 0.f;
                const float f0 = a0 * inv, f1 = a1 * inv;
                constexpr int CH = D / 4;  // 16-byte chunks per row
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int col = 64 * wg + 32 * cc;
                    uint32_t o0[32], o1[32];
                    tc05::tmem_ld32(tm + lane_base + Sh::col_o(0) + col, o0);
                    tc05::tmem_ld32(tm + lane_base + Sh::col_o(1) + col, o1);
                    // a WG with no tile (ntiles = 1) never wrote its O: its
                    // columns are selected away, never multiplied by 0
                    const bool u0 = f0 != 0.f, u1 = f1 != 0.f;
                    auto mix = [&](uint32_t x0, uint32_t x1) {
                        return (u0 ? __uint_as_float(x0) * f0 : 0.f) + (u1 ? __uint_as_float(x1) * f1 : 0.f);
                    };
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int kch = col / 4 + i;
                        float4 v;
                        v.x = mix(o0[4 * i], o1[4 * i]);
                        v.y = mix(o0[4 * i + 1], o1[4 * i + 1]);
                        v.z = mix(o0[4 * i + 2], o1[4 * i + 2]);
                        v.w = mix(o0[4 * i + 3], o1[4 * i + 3]);
                        if (!any) v = make_float4(0.f, 0.f, 0.f, 0.f);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         stage + r * (D * 4) + ((kch ^ (r & (CH - 1))) << 4)),
                                     "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                                     : "memory");
                    }
                }
                if (row_ok && wg == 0) *lse_row = any ? (M + log2f(Lsum)) * 0.6931471805599453f : -INFINITY;
                mbar_arrive(staged);
                if (!warp_wait(staged, 0)) {
                    if (r == 0) raise_error(p.err, KF_DEVERR_TIMEOUT);
                } else {
                    for (int rr = warp; rr < kRowsP; rr += 8) {
                        const int64_t grow = prow0 + (int64_t)cr * kRowsP + rr;
                        if (grow >= nrow_all) break;  // rows ascend: the rest are past the request
                        float *dst = p.out_partial +
                                     (((int64_t)s * p.num_q_tokens + q0 + grow / G) * Hq + h * G + (int)(grow % G)) * D;
                        float4 v;
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                     : "r"(stage + rr * (D * 4) + ((lane ^ (rr & (CH - 1))) << 4))
                                     : "memory");
                        reinterpret_cast<float4 *>(dst)[lane] = v;
                    }
                }
            }
        }
    }
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == Sh::kIssuer) {
        // neither CTA frees its TMEM (or exits) while the other may still reach
        // into it: each tells the other it is done and waits for the same
        if (lane == 0) {
            arrive_cluster(map_to(bye, cr ^ 1u));
            if (!wait_cl(bye, 0)) raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
        __syncwarp();
        tc05::fence_after_sync();
        tc05::tmem_dealloc2(tm, Sh::kTmemCols);
    }
}

// 4-D view of a [num_blocks, bs, Hkv, 128] bf16 cache whose box is one block
// of one head's 64-column half: (d % 64, slot % 8, head * 2 + d / 64, 8-slot
// group = block * bs/8 + slot / 8), box (64, 8, 1, bs / 8) = bs * 128 bytes,
// landing as 8-token atoms of 128-byte rows (token t at (t / 8) * 1024 +
// (t % 8) * 128).
bool encode_half_map(tc::EncodeFn fn, CUtensorMap *map, const void *cache, const MqParams &p) {
    const cuuint64_t row = (cuuint64_t)p.num_kv_heads * p.head_dim * 2;  // bytes between slots
    const cuuint64_t dims[4] = {64, 8, (cuuint64_t)p.num_kv_heads * 2, (cuuint64_t)p.num_blocks * (p.block_size / 8)};
    const cuuint64_t strides[3] = {row, 128, 8 * row};
    const cuuint32_t box[4] = {64, 8, 1, (cuuint32_t)p.block_size / 8};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_p(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv) {
    using Sh = PShape;
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        e = cudaFuncSetAttribute(mqp_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * p.num_splits, p.num_kv_heads, p.batch * p.q_tiles);
    cfg.blockDim = dim3(Sh::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Sh::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;  // the pair: cluster ranks 0 and 1 are blockIdx.x 2s and 2s + 1
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mqp_kernel<G>, p, mk, mv);
}

}  // namespace

cudaError_t launch_multiquery_tc05p(MqParams p, cudaStream_t stream, void *encode) {
    if (p.batch == 0 || p.num_q_tokens == 0) return cudaSuccess;
    if (p.head_dim != kDP) return cudaErrorInvalidValue;
    const int G = p.num_q_heads / p.num_kv_heads;
    const int64_t rows = (int64_t)p.max_query_len * G;
    p.q_tiles = (int)((rows + 2 * kRowsP - 1) / (2 * kRowsP));  // 256 rows per pair
    if (p.q_tiles < 1) p.q_tiles = 1;
    if ((int64_t)p.batch * p.q_tiles > 65535 || (int64_t)p.num_splits * 2 > 0x7fffffff)
        return cudaErrorInvalidValue;
    tc::EncodeFn fn = reinterpret_cast<tc::EncodeFn>(encode);
    CUtensorMap mk, mv;
    if (!encode_block_map(fn, &mk, p.k_cache, p) || !encode_half_map(fn, &mv, p.v_cache, p))
        return cudaErrorInvalidValue;
    switch (G) {
        case 1: return launch_p<1>(p, stream, mk, mv);
        case 2: return launch_p<2>(p, stream, mk, mv);
        case 4: return launch_p<4>(p, stream, mk, mv);
        case 8: return launch_p<8>(p, stream, mk, mv);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kf
