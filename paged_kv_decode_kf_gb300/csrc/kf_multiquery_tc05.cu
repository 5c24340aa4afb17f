// kf_multiquery_tc05.cu -- multi-query paged attention on the tcgen05 tensor
// cores: the same contract as kf_multiquery.cu (chunked prefill / speculative
// verify with causal = 1, the shared-prefix pass of cascade attention with
// causal = 0), for query tiles large enough to fill a 128-row MMA.
//
// What it computes: "Mathematical Formulation of Chunked Attention" of
// "Disaggregated Inference Architecture: Paged KV-Cache Tiering, Chunked
// Prefill, and Asynchronous Overlap" (ultrainstinct.tech): each query of a
// chunk attends to the paged history without a mask and to its own chunk
// causally; with the chunk already the last C of L cached tokens, query j
// attends to tokens [0, L - C + j]. Cascade attention ("What FlashInfer
// brings: JIT and cascade attention", blog.lo0.es) is a non-causal call over
// the shared prefix. The output is the split partials (o, lse).
//
// Design: one CTA per (split, KV head, request x 128-row query tile); a row is
// a (query token, query head of the KV head's group) pair, so the G heads of a
// KV head share every K/V tile. 6 warps:
//   warps 0-3  softmax: thread r owns row r -- loads its q row into the
//              swizzled Q tile, and per 64-token tile reads its 64 scores from
//              TMEM, masks them, runs the base-2 online softmax (lazy rescale:
//              the running max moves only when a tile exceeds it by more than
//              8, and then the warp rescales its O rows in TMEM), writes its 64
//              weights as bf16 pairs to TMEM, and in the end writes o = O / l
//              and lse.
//   warp 4     TMA producer: walks the split's blocks through the table and
//              loads K_j and V_j into a ring of 64-token slots, one TMA box per
//              cache block (all bs tokens and all D of one head: 4 KiB at D 128,
//              bs 16; small boxes cap TMA throughput). The cache is viewed as
//              5-D (d % 64, slot % 8, 2 head + d / 64, slot / 8, block) -- the
//              head stride is twice the half stride, so (head, half) is one
//              dimension -- and a box lands as 8-token atoms of 128-byte rows:
//              token t, half c at (t / 8) * 1024 * D/64 + c * 1024 + (t % 8) * 128,
//              128-byte swizzled, which both MMAs read in place (K: K-major,
//              8-row stride 1024 * D/64; V: MN-major, d atoms 1024 apart).
//   warp 5     MMA issuer (one thread) and TMEM owner:
//                S_j  = Q K_j^T   M 128, N 64, K = D: A = Q (smem, K-major),
//                                  B = K tile (smem, K-major), D in TMEM;
//                O   += P_j V_j   M 128, N = D, K 64: A = P (TMEM, bf16),
//                                  B = V tile (smem, MN-major), D in TMEM;
//              issued in the order S_0, S_1, PV_0, S_2, PV_1, ... so that the
//              product of tile j + 1 runs while the softmax of tile j does.
// TMEM (256 columns, two CTAs per SM): S in columns [0, 64), P_j in
// [64 + 32 (j % 2), + 32), O in [128, 128 + D).
// Synchronisation is by mbarriers: full/empty per ring slot (TMA / MMA
// commit), q_ready, s_full (commit) / s_free (softmax read S), p_full[2]
// (softmax wrote P), o_done (commit after each PV). Every wait is bounded; a
// wait that gives up sets KF_DEVERR_TIMEOUT, the CTA drains its copies and
// MMAs and frees its TMEM before it returns. V rows past the range in the
// last tile are zeroed in shared memory (their weights are 0, but 0 * NaN is
// NaN); masked scores are selected to -inf, never multiplied.
//
// Precision: scores and O accumulate in fp32; P enters the PV product as
// bf16 (relative error <= 2^-9 per weight, unbiased rounding), l sums the
// unrounded fp32 weights.
#include <stdlib.h>
#include <string.h>

#include "kf_mq_tc05.cuh"

namespace kf {
namespace {

using namespace tc;
using namespace mq5;

constexpr int kRows = 128;  // query rows per tile: M of both products
constexpr int kTile = 64;   // tokens per KV tile

// Shared-memory and TMEM geometry of a CTA with QT query tiles (QT = 2: both
// tiles read every K/V tile once, one CTA per SM; QT = 1: two CTAs per SM).
// SQ (compact Q, one tile): a request has at most 32 rows per KV head
// (speculative verify: 4 draft tokens x G 4 = 16). Only those rows of Q are
// stored (8 KiB at D 128 instead of 32); the MMA still reads 128 rows of A, and
// the rows past the stored ones read whatever the ring holds there -- they
// only make rows of S, P and O that no warp reads or stores (an MMA row
// depends on its own row of A alone). The room goes to two more ring slots.
template <int D, int QT, bool SQ = false>
struct T5Shape {
    static constexpr int kHalves = D / 64;                       // 64-wide d halves (128-byte rows)
    static constexpr int kQRows = SQ ? 32 : kRows;               // rows of Q stored
    static constexpr int kQHalfBytes = kQRows * 128;             // 16 KiB (4 KiB compact)
    static constexpr int kQTileBytes = kHalves * kQHalfBytes;
    static constexpr int kQBytes = QT * kQTileBytes;
    static constexpr int kAtomBytes = kHalves * 1024;            // 8 tokens x D
    static constexpr int kSlotBytes = kTile / 8 * kAtomBytes;    // 64 tokens x D
    static constexpr int kSlots = (QT == 1 ? (SQ ? 6 : 4) : 8) * (128 / D);
    static_assert(!SQ || QT == 1, "compact Q has one tile");
    static constexpr int kSmemBytes = kQBytes + kSlots * kSlotBytes + 1024;
    static constexpr int kSoftWarps = 4 * QT;
    // NPW TMA producer warps: kProducer (K items, or every item when NPW = 1)
    // and kProducer2 (V items). TMA instructions issued by the lanes of one warp
    // are taken one after another (~90 cycles per box); different warps' overlap.
    static constexpr int kProducer = kSoftWarps, kIssuer = kSoftWarps + 1, kProducer2 = kSoftWarps + 2;
    __host__ __device__ static constexpr int threads(int npw) { return 32 * (kSoftWarps + 1 + npw); }
    // TMEM columns: S_t [64 t, +64), P_t two buffers of 32 at 64 QT + 64 t,
    // O_t D columns at 128 QT + D t
    static constexpr uint32_t kTmemCols = QT == 1 ? 256 : 512;
    __host__ __device__ static constexpr uint32_t col_s(int t) { return 64u * t; }
    __host__ __device__ static constexpr uint32_t col_p(int t) { return 64u * QT + 64u * t; }
    __host__ __device__ static constexpr uint32_t col_o(int t) { return 128u * QT + (uint32_t)D * t; }
    // the allocation always fits: at most 512 / kTmemCols CTAs share an SM
    static_assert(QT == 1 ? kSmemBytes > 80 * 1024 : kSmemBytes > 116 * 1024, "TMEM budget per SM");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};


// Two CTAs per SM with one tile (one with two). A sub-partition's 16384
// registers hold floor(16384 / (32 x regs)) warps, so two seven-warp CTAs (four
// warps on some sub-partitions) cap a thread at 128 registers; at that cap the
// kernel spills a few bytes, which measured faster than one CTA per SM.
template <int D, int G, int QT, int NPW, bool SQ>
__global__ void __launch_bounds__(T5Shape<D, QT, SQ>::threads(NPW), QT == 1 ? 2 : 1)
mq5_kernel(const MqParams p, const __grid_constant__ CUtensorMap tmap_k,
           const __grid_constant__ CUtensorMap tmap_v) {
    using Sh = T5Shape<D, QT, SQ>;
    constexpr int NSL = Sh::kSlots;
    constexpr int KS = D / 16;  // K steps of S = Q K^T

    // barriers: full[NSL], empty[NSL], q_ready, fin, then per tile t:
    // s_full, s_free, p_full[2], o_done
    __shared__ __align__(8) uint64_t bar_mem[2 * NSL + 2 + 5 * QT];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base, sKV = base + Sh::kQBytes;
    const uint32_t bars = smem_u32(bar_mem);
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (NSL + i); };
    const uint32_t q_ready = bars + 8u * (2 * NSL), fin = q_ready + 8;
    auto s_full = [&](int t) { return fin + 8u + 40u * t; };
    auto s_free = [&](int t) { return fin + 16u + 40u * t; };
    auto p_full = [&](int t, int k) { return fin + 24u + 40u * t + 8u * k; };
    auto o_done = [&](int t) { return fin + 40u + 40u * t; };

    const int s = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / p.q_tiles, qg = blockIdx.z % p.q_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.num_q_heads;

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
    if (threadIdx.x == 0 && s == 0 && h == 0 && qg == p.q_tiles - 1 &&
        nrow_all > (int64_t)p.q_tiles * QT * kRows)
        raise_error(p.err, KF_DEVERR_MAX_CONTEXT);  // more queries than max_query_len covers
    const int64_t row0 = (int64_t)qg * QT * kRows;
    if (row0 >= nrow_all) return;  // beyond this request's queries: nothing to write
    const int64_t nrows = nrow_all - row0 < QT * kRows ? nrow_all - row0 : QT * kRows;
    const int nqt = (int)((nrows + kRows - 1) / kRows);  // tiles with rows (CTA-uniform)

    // token range: the split, clipped to the context and to the last row's limit
    const int64_t span = (int64_t)p.chunk_blocks * p.block_size;
    int64_t t_lo = (int64_t)s * span, t_hi = t_lo + span;
    const int64_t t_max = p.causal ? L - C + (row0 + nrows - 1) / G + 1 : L;
    if (t_hi > t_max) t_hi = t_max;
    if (t_lo > t_hi) t_lo = t_hi;

    // this thread's row (softmax threads): tile tq, row r of the tile
    const int tq = warp / 4;
    const int r = threadIdx.x & (kRows - 1);
    const bool soft = warp < Sh::kSoftWarps;
    const int64_t row = row0 + (int64_t)tq * kRows + r;
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
    const int ntiles = (int)((t_hi - t_lo + kTile - 1) / kTile);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSL; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        mbar_init(q_ready, 32 * Sh::kSoftWarps);
        mbar_init(fin, 1);
        for (int t = 0; t < QT; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(s_free(t), kRows);
            mbar_init(p_full(t, 0), kRows);
            mbar_init(p_full(t, 1), kRows);
            mbar_init(o_done(t), 1);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == Sh::kIssuer) tc05::tmem_alloc(smem_u32(&tmem_slot), Sh::kTmemCols);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tm = tmem_slot;

    if (warp == Sh::kProducer || (NPW == 2 && warp == Sh::kProducer2)) {
        // ------------------------------ producer ------------------------------
        // (with two producer warps, warp kProducer takes the K items 2j and
        // warp kProducer2 the V items 2j + 1)
        // The whole warp walks its items: the table entries come 32 at a time
        // (one coalesced load, lane e holds logical block base + e), so no TMA
        // issue waits on a dependent load; lane 0 waits for slots, and lane k
        // issues the box of the tile's block k.
        const int bs_shift = block_shift(p.block_size);
        const uint32_t box_bytes = (uint32_t)p.block_size * D * 2;
        const int ifirst = warp == Sh::kProducer ? 0 : 1, istep = NPW;
        int64_t tab_base = -1;
        int32_t tab_ent = -1;
        int issued = 0;
        for (int i = ifirst; i < 2 * ntiles; i += istep) {
            const int slot = i % NSL;
            int go = 1;
            if (lane == 0) {
                go = !abort_flag && mbar_wait(empty(slot), ((i / NSL) & 1) ^ 1);
                if (!go) {
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            const CUtensorMap *map = (i & 1) ? &tmap_v : &tmap_k;
            const int64_t t0 = t_lo + (int64_t)(i >> 1) * kTile;
            const int64_t ntok = t_hi - t0 < kTile ? t_hi - t0 : kTile;
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
            issued = i + 1;
        }
        if (lane == 0) {
            // drain: this warp's copies among the last NSL items have landed
            // before the CTA can exit
            for (int i = issued > NSL ? issued - NSL : 0; i < issued; ++i)
                if ((i - ifirst) % istep == 0 && !mbar_wait(full(i % NSL), (i / NSL) & 1))
                    raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
    } else if (warp == Sh::kIssuer) {
        // ------------------------------ MMA issuer -----------------------------
        if (lane == 0) {
            const uint32_t id_s = tc05::idesc_bf16(kRows, kTile, false, false);
            const uint32_t id_o = tc05::idesc_bf16(kRows, D, false, true);
            const uint64_t qdesc0 = tc05::sdesc_sw128(sQ, 16, 1024);
            bool ok = mbar_wait(q_ready, 0);
            // O_t += P_t V_i for every tile with rows; then the V slot is free
            auto pv = [&](int i) -> bool {
                const int slot = (2 * i + 1) % NSL;
                if (!mbar_wait(full(slot), ((2 * i + 1) / NSL) & 1)) return false;
                // one descriptor per tile, stepped by 16-byte units (the start-address field)
                const uint64_t vd = tc05::sdesc_sw128(sKV + slot * Sh::kSlotBytes, 1024, Sh::kAtomBytes);
                for (int t = 0; t < nqt; ++t) {
                    if (!mbar_wait(p_full(t, i & 1), (i >> 1) & 1)) return false;
                    tc05::fence_after_sync();
                    const uint32_t pa = tm + Sh::col_p(t) + 32 * (i & 1), od = tm + Sh::col_o(t);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        tc05::mma_ts(od, pa + 8 * kk, vd + (uint64_t)(kk * 2 * Sh::kAtomBytes / 16), id_o,
                                     (i > 0 || kk > 0) ? 1u : 0u);
                    tc05::commit(o_done(t));
                }
                tc05::commit(empty(slot));
                return true;
            };
            for (int j = 0; ok && j < ntiles; ++j) {
                if (abort_flag) {
                    ok = false;
                    break;
                }
                const int slot = (2 * j) % NSL;
                if (!mbar_wait(full(slot), ((2 * j) / NSL) & 1)) {
                    ok = false;
                    break;
                }
                const uint64_t kd = tc05::sdesc_sw128(sKV + slot * Sh::kSlotBytes, 16, Sh::kAtomBytes);
                for (int t = 0; ok && t < nqt; ++t) {
                    if (j > 0 && !mbar_wait(s_free(t), (j - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc05::fence_after_sync();
                    const uint64_t qd = qdesc0 + (uint64_t)(t * Sh::kQTileBytes / 16);
                    const uint32_t sd = tm + Sh::col_s(t);
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk)
                        tc05::mma_ss(sd, qd + (uint64_t)(((kk >> 2) * Sh::kQHalfBytes + 32 * (kk & 3)) / 16),
                                     kd + (uint64_t)(((kk >> 2) * 1024 + 32 * (kk & 3)) / 16), id_s,
                                     kk > 0 ? 1u : 0u);
                    tc05::commit(s_full(t));
                }
                if (!ok) break;
                tc05::commit(empty(slot));
                if (j > 0 && !pv(j - 1)) {
                    ok = false;
                    break;
                }
            }
            if (ok && !abort_flag) ok = pv(ntiles - 1);
            if (!ok) {
                raise_error(p.err, KF_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            // every MMA issued has completed before TMEM is freed
            tc05::commit(fin);
            if (!mbar_wait(fin, 0)) raise_error(p.err, KF_DEVERR_TIMEOUT);
        }
    } else {
        // ------------------------------- softmax --------------------------------
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        {
            // q row -> swizzled Q tile tq (K-major, 128-byte rows, 8-row atoms)
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (qrow * Hq + qhead) * D);
            const uint32_t qb = sQ + tq * Sh::kQTileBytes;
#pragma unroll
            for (int c16 = 0; c16 < D / 8; ++c16) {
                if (r >= Sh::kQRows) break;  // compact Q: rows past the stored ones
                const uint4 v = row_ok ? __ldg(src + c16) : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t a = qb + (c16 >> 3) * Sh::kQHalfBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                                   (((c16 & 7) ^ (r & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
                             "r"(v.w)
                             : "memory");
            }
            fence_proxy_async_smem();
            mbar_arrive(q_ready);
        }
        const int64_t lim = row_ok ? (p.causal ? L - C + row / G + 1 : L) : 0;
        const int64_t row_hi = lim < t_hi ? lim : t_hi;  // this row's tokens end here
        const float c = p.scale_log2;
        const uint32_t col_s = Sh::col_s(tq), col_p = Sh::col_p(tq), col_o = Sh::col_o(tq);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // A warp with no row of the request (a short tile: speculative verify
        // fills 16 of 128 rows) keeps the barrier protocol and its share of the
        // V-tail zeroing but reads no scores and writes no weights: its P lanes
        // hold whatever TMEM held, which reaches only its own rows of O (an MMA
        // row depends on its own row of A alone), and those rows are never stored.
        const bool live = __any_sync(0xffffffffu, row_ok);
        if (tq < nqt) {
            for (int j = 0; j < ntiles; ++j) {
                const int64_t t0 = t_lo + (int64_t)j * kTile;
                // (the flag is read warp-uniformly: tcgen05.ld/st need the whole warp)
                if (__any_sync(0xffffffffu, abort_flag != 0) || !warp_wait(s_full(tq), j & 1)) {
                    ok = false;
                    break;
                }
                uint32_t sr[kTile];
                if (live) {
                    tc05::fence_after_sync();
                    tc05::tmem_ld64(tm + lane_base + col_s, sr);
                    tc05::fence_before_sync();
                }
                mbar_arrive(s_free(tq));

                const int64_t ntile_tok = t_hi - t0 < kTile ? t_hi - t0 : kTile;
                if (ntile_tok < kTile) {
                    // zero the V rows past the range (each tile's warps zero all of them)
                    const int slot = (2 * j + 1) % NSL;
                    if (!warp_wait(full(slot), ((2 * j + 1) / NSL) & 1)) {
                        ok = false;
                        break;
                    }
                    const int nz = (int)(kTile - ntile_tok) * 8 * Sh::kHalves;  // 16-byte chunks
                    const uint32_t vb = sKV + slot * Sh::kSlotBytes;
                    for (int i = r; i < nz; i += kRows) {
                        const int hf = i / ((int)(kTile - ntile_tok) * 8);
                        const int rem = i % ((int)(kTile - ntile_tok) * 8);
                        const int t = (int)ntile_tok + rem / 8;
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                         vb + (t >> 3) * Sh::kAtomBytes + hf * 1024 + (t & 7) * 128 + (rem % 8) * 16),
                                     "r"(0u)
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                }
                if (!live) {
                    mbar_arrive(p_full(tq, j & 1));
                    continue;
                }
                const int64_t nv64 = row_hi - t0;
                const int nv = nv64 <= 0 ? 0 : (nv64 >= kTile ? kTile : (int)nv64);
                // Fast path -- every row of the warp sees the whole tile and the
                // scale is positive: the max of the raw scores (times c), and one
                // fused multiply-add per weight below. Otherwise scores are scaled
                // and masked to -inf first. Rows past the request (zero q, so
                // zero scores against the tile's in-context keys) do not force
                // the masked path.
                const bool fast = c > 0.f && __all_sync(0xffffffffu, nv == kTile || !row_ok);
                float mx = -INFINITY;
                if (fast) {
#pragma unroll
                    for (int i = 0; i < kTile; i += 2)
                        mx = max3f(mx, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
                    mx *= c;
                } else {
#pragma unroll
                    for (int i = 0; i < kTile; ++i) {
                        const float x = i < nv ? __uint_as_float(sr[i]) * c : -INFINITY;
                        sr[i] = __float_as_uint(x);
                        mx = fmaxf(mx, x);
                    }
                }
                const bool need = mx > m + kRescaleSlack;
                const float alpha = need ? exp2f(m - mx) : 1.f;  // m = -inf: 0
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    // O holds PV_0 .. PV_{j-1}: rescale this warp's rows once they are done
                    if (!warp_wait(o_done(tq), (j - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc05::fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tc05::tmem_ld32(tm + lane_base + col_o + 32 * cc, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc05::tmem_st32(tm + lane_base + col_o + 32 * cc, o);
                    }
                }
                if (need) {
                    l *= alpha;
                    m = mx;
                }
                const float mu = m == -INFINITY ? 0.f : m;
                uint32_t pr[kTile / 2];
                float2 ls = make_float2(0.f, 0.f);
                if (fast) {
                    const float2 c2 = make_float2(c, c), nm = make_float2(-mu, -mu);
#pragma unroll
                    for (int i = 0; i < kTile / 2; ++i) {
                        float2 a = fma_f32x2(make_float2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                                             c2, nm);
                        a.x = ex2f(a.x);
                        a.y = ex2f(a.y);
                        ls = add_f32x2(ls, a);
                        pr[i] = pack_bf16(a.x, a.y);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kTile / 2; ++i) {
                        const float p0 = ex2f(__uint_as_float(sr[2 * i]) - mu);
                        const float p1 = ex2f(__uint_as_float(sr[2 * i + 1]) - mu);
                        ls = add_f32x2(ls, make_float2(p0, p1));
                        pr[i] = pack_bf16(p0, p1);
                    }
                }
                l += ls.x + ls.y;
                tc05::tmem_st32(tm + lane_base + col_p + 32 * (j & 1), pr);
                tc05::fence_before_sync();
                mbar_arrive(p_full(tq, j & 1));
            }
            // The epilogue waits for fin (one phase, committed after the last MMA):
            // a parity wait on o_done could alias -- this warpgroup can get here
            // with the last two PVs still pending, and two phases back has the
            // parity it waits for. (Every other wait here is at most one phase
            // behind its barrier.)
            if (ok && !live) {
                // nothing to store; the issuer waits for the last MMA before TMEM is freed
            } else if (ok && warp_wait(fin, 0)) {
                tc05::fence_after_sync();
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tc05::tmem_ld32(tm + lane_base + col_o + 32 * cc, o);
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(o_row + 32 * cc + i) =
                                l > 0.f ? make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                                                      __uint_as_float(o[i + 2]) * inv,
                                                      __uint_as_float(o[i + 3]) * inv)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (row_ok) *lse_row = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
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

template <int D, int G, int QT, int NPW, bool SQ>
cudaError_t launch_t5(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv) {
    using Sh = T5Shape<D, QT, SQ>;
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        e = cudaFuncSetAttribute(mq5_kernel<D, G, QT, NPW, SQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch * p.q_tiles);
    mq5_kernel<D, G, QT, NPW, SQ><<<grid, Sh::threads(NPW), Sh::kSmemBytes, stream>>>(p, mk, mv);
    return cudaGetLastError();
}

// Compact Q when a request has at most 32 rows per KV head, with one producer
// warp: its six-slot ring keeps enough in flight, and at two CTAs per SM a
// seventh warp would cap a thread at 128 registers and spill (speculative
// verify: 162.5 us against 167.7 with two producers, 170.3 without compact Q).
// Otherwise two producer warps (181.8 -> 168.5 us there before compact Q).
// KF_MQW_PRODUCERS = 1 or 2 and KF_MQ_COMPACT_Q = 0 override (read per call).
template <int D, int G, int QT>
cudaError_t launch_t5(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv) {
    const char *s = getenv("KF_MQW_PRODUCERS");
    const char *c = getenv("KF_MQ_COMPACT_Q");
    const bool sq = QT == 1 && (int64_t)p.max_query_len * G <= 32 && !(c && strcmp(c, "0") == 0);
    const bool one = s ? strcmp(s, "1") == 0 : sq;
    if (QT == 1 && sq)
        return one ? launch_t5<D, G, 1, 1, true>(p, stream, mk, mv) : launch_t5<D, G, 1, 2, true>(p, stream, mk, mv);
    return one ? launch_t5<D, G, QT, 1, false>(p, stream, mk, mv) : launch_t5<D, G, QT, 2, false>(p, stream, mk, mv);
}

template <int D, int QT>
cudaError_t launch_t5_g(const MqParams &p, cudaStream_t stream, const CUtensorMap &mk, const CUtensorMap &mv) {
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: return launch_t5<D, 1, QT>(p, stream, mk, mv);
        case 2: return launch_t5<D, 2, QT>(p, stream, mk, mv);
        case 4: return launch_t5<D, 4, QT>(p, stream, mk, mv);
        case 8: return launch_t5<D, 8, QT>(p, stream, mk, mv);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_multiquery_tc05(MqParams p, cudaStream_t stream, void *encode) {
    if (p.batch == 0 || p.num_q_tokens == 0) return cudaSuccess;
    const int G = p.num_q_heads / p.num_kv_heads;
    const int64_t rows = (int64_t)p.max_query_len * G;
    // One 128-row tile per CTA (two CTAs per SM) by default: two independent
    // MMA issuers per SM measured faster than one CTA holding two tiles, whose
    // single issuer spends most of a tile in barrier waits. KF_MQ_TILES = 2
    // selects two tiles per CTA (only when a request has more than 128 rows).
    const char *force = getenv("KF_MQ_TILES");
    const int QT = force && force[0] == '2' && rows > kRows ? 2 : 1;
    p.q_tiles = (int)((rows + QT * kRows - 1) / (QT * kRows));
    if (p.q_tiles < 1) p.q_tiles = 1;
    if ((int64_t)p.batch * p.q_tiles > 65535) return cudaErrorInvalidValue;
    tc::EncodeFn fn = reinterpret_cast<tc::EncodeFn>(encode);
    CUtensorMap mk, mv;
    if (!encode_block_map(fn, &mk, p.k_cache, p) || !encode_block_map(fn, &mv, p.v_cache, p))
        return cudaErrorInvalidValue;
    if (p.head_dim == 128)
        return QT == 2 ? launch_t5_g<128, 2>(p, stream, mk, mv) : launch_t5_g<128, 1>(p, stream, mk, mv);
    return QT == 2 ? launch_t5_g<64, 2>(p, stream, mk, mv) : launch_t5_g<64, 1>(p, stream, mk, mv);
}

}  // namespace kf
