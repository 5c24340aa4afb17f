"""Pins of the fp64 oracle to facts other than itself.

Each pin checks the oracle (loaded as `lib`) against something the pages or
the mathematics fix: hand-derived worked examples (tests/golden), closed forms
(context length 1, identical keys, zero scale, one dominant key, constant
values per KV head), invariants (physical-block permutation, split/merge
equality, merge associativity, score-shift invariance) and an independent
library computation (scipy's logsumexp/softmax over a contiguous copy made by
numpy indexing). The planted-mistake tests run every pin against mutated
builds of the oracle and require each mutation to be caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from paged_kv_decode_kf_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_examples.json")


def _bf16(a) -> np.ndarray:
    """Exact bf16 bit patterns of a float array (values must be bf16-exact)."""
    t = torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(a, dtype=np.float32)), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def _widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> float64 via torch (independent of the oracle's widening)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def _small(batch=3, hq=4, hkv=2, d=16, bs=4, lengths=(5, 9, 16), seed=7, spare=3):
    w = wl.Workload(name="pin", batch=batch, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                    block_size=bs, lengths=wl.Fixed(tuple(lengths)), seed=seed, spare_blocks=spare)
    inp = wl.make_inputs(w, "cpu")
    # attention below runs over ctx_before tokens; the tables cover ctx_before + 1
    return w, inp


def _arrays(inp):
    return (wl.bf16_bits(inp.q), wl.bf16_bits(inp.k_cache), wl.bf16_bits(inp.v_cache),
            inp.block_tables.numpy(), inp.ctx_after.numpy())


def _gather(cache_bits, bt_row, bs, h, L):
    """Contiguous [L, D] float64 copy of one request/head by numpy indexing."""
    t = np.arange(L)
    blocks = bt_row[t // bs]
    return _widen(cache_bits[blocks, t % bs, h, :])


def _load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_bf16_widening(lib):
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F81: 1.0 + 2 ** -7, 0x0001: 2.0 ** -133,
             0x7F80: math.inf, 0x0000: 0.0, 0x4049: 3.140625}
    for bits, val in cases.items():
        assert oracle.bf16_to_f64(bits, lib=lib) == val, hex(bits)


def pin_golden_two_token(lib):
    g = _load_golden()["two_token_softmax"]
    out, lse = oracle.attention(_bf16(g["q"]), _bf16(g["k_cache"]), _bf16(g["v_cache"]),
                                np.array(g["block_tables"], np.int32), np.array(g["ctx_lens"], np.int32),
                                g["scale"], lib=lib)
    np.testing.assert_allclose(out, np.array(g["expect_out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(g["expect_lse"]), rtol=0, atol=1e-13)


def pin_golden_gqa(lib):
    g = _load_golden()["gqa_two_blocks"]
    args = (_bf16(g["q"]), _bf16(g["k_cache"]), _bf16(g["v_cache"]),
            np.array(g["block_tables"], np.int32), np.array(g["ctx_lens"], np.int32))
    out, lse = oracle.attention(*args, g["scale"], lib=lib)
    np.testing.assert_allclose(out, np.array(g["expect_out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(g["expect_lse"]), rtol=0, atol=1e-13)
    S, maxL = g["splits"], g["max_context_len"]
    for s, (lo, hi) in enumerate(g["expect_split_ranges"]):
        assert oracle.split_range(3, g["block_size"], S, maxL, s, lib=lib) == (lo, hi)
    o_p, lse_p = oracle.decode_partials(*args, g["scale"], S, max_context_len=maxL, lib=lib)
    for head, key in ((0, "expect_partials_head0"), (3, "expect_partials_head3")):
        np.testing.assert_allclose(o_p[:, 0, head, 0], g[key]["o"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse_p[:, 0, head], g[key]["lse"], rtol=0, atol=1e-13)
    m_out, m_lse = oracle.merge_partials(o_p, lse_p, lib=lib)
    np.testing.assert_allclose(m_out, np.array(g["expect_out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(m_lse, np.array(g["expect_lse"]), rtol=0, atol=1e-13)


def pin_golden_merge(lib):
    g = _load_golden()["merge_closed_form"]
    o, lse = oracle.merge(np.array(g["o_parts"], float), np.array(g["lse_parts"]), lib=lib)
    np.testing.assert_allclose(o, g["expect_out"], rtol=0, atol=1e-14)
    assert abs(lse - g["expect_lse"]) < 1e-14
    o2, lse2 = oracle.merge(np.array(g["o_parts"] + [[0, 0]], float),
                            np.array(g["lse_parts"] + [-math.inf]), lib=lib)
    np.testing.assert_allclose(o2, g["expect_out"], rtol=0, atol=1e-14)
    assert abs(lse2 - g["expect_lse"]) < 1e-14


def pin_golden_append(lib):
    g = _load_golden()["append_fresh_block"]
    nb, bs, hkv, d = g["num_blocks"], g["block_size"], g["num_kv_heads"], g["head_dim"]
    rng = np.random.default_rng(3)
    k = rng.integers(0, 2 ** 16, size=(nb, bs, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(nb, bs, hkv, d), dtype=np.uint16)
    kn = rng.integers(0, 2 ** 16, size=(1, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 2 ** 16, size=(1, hkv, d), dtype=np.uint16)
    k2, v2, skipped = oracle.append(k, v, kn, vn, np.array(g["block_tables"], np.int32),
                                    np.array(g["ctx_before"], np.int32), lib=lib)
    assert skipped == 0
    blk, slot = g["expect_block"], g["expect_slot"]
    ek, ev = k.copy(), v.copy()
    ek[blk, slot] = kn[0]
    ev[blk, slot] = vn[0]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


def pin_context_len_one(lib):
    w, inp = _small(lengths=(0, 0, 0))
    q, k, v, bt, _ = _arrays(inp)
    ctx = np.ones(w.batch, np.int32)
    out, lse = oracle.attention(q, k, v, bt, ctx, w.scale, lib=lib)
    G = w.group
    for b in range(w.batch):
        for h in range(w.num_q_heads):
            k0 = _gather(k, bt[b], w.block_size, h // G, 1)[0]
            v0 = _gather(v, bt[b], w.block_size, h // G, 1)[0]
            assert np.array_equal(out[b, h], v0)
            s0 = w.scale * float(np.dot(_widen(q[b, h]), k0))
            assert abs(lse[b, h] - s0) <= 1e-12 * max(1.0, abs(s0))


def pin_identical_keys(lib):
    w, inp = _small(lengths=(6, 13, 30))
    q, k, v, bt, ctx = _arrays(inp)
    k = k.copy()
    k[:] = k[0:1, 0:1]            # every slot of every block holds the same key rows
    out, lse = oracle.attention(q, k, v, bt, ctx, w.scale, lib=lib)
    G = w.group
    for b in range(w.batch):
        L = int(ctx[b])
        for h in range(w.num_q_heads):
            V = _gather(v, bt[b], w.block_size, h // G, L)
            kk = _widen(k[0, 0, h // G])
            s = w.scale * float(np.dot(_widen(q[b, h]), kk))
            np.testing.assert_allclose(out[b, h], V.mean(axis=0), rtol=0, atol=1e-12)
            assert abs(lse[b, h] - (s + math.log(L))) <= 1e-12 * max(1.0, abs(s + math.log(L)))


def pin_scale_zero(lib):
    w, inp = _small(lengths=(3, 20, 11))
    q, k, v, bt, ctx = _arrays(inp)
    out, lse = oracle.attention(q, k, v, bt, ctx, 0.0, lib=lib)
    for b in range(w.batch):
        L = int(ctx[b])
        for h in range(w.num_q_heads):
            V = _gather(v, bt[b], w.block_size, h // w.group, L)
            np.testing.assert_allclose(out[b, h], V.mean(axis=0), rtol=0, atol=1e-12)
            assert abs(lse[b, h] - math.log(L)) <= 1e-12


def pin_dominant_key(lib):
    """K at one token = 8*q (exact in bf16): its score beats every other by
    hundreds, so o equals that token's V to fp64 precision. Catches a wrong
    K/V token pairing, a wrong sign and a wrong block."""
    w, inp = _small(batch=1, hq=1, hkv=1, d=32, bs=4, lengths=(21,))
    q, k, v, bt, ctx = _arrays(inp)
    L = int(ctx[0])
    qv = _widen(q[0, 0])
    for t_star in (0, 3, 4, 11, L - 1):
        kk = k.copy()
        kk[:] = _bf16(np.zeros(kk.shape, np.float32))            # all other keys 0
        blk, slot = bt[0][t_star // w.block_size], t_star % w.block_size
        kk[blk, slot, 0] = _bf16((8.0 * qv).astype(np.float32))
        out, _ = oracle.attention(q, kk, v, bt, ctx, 1.0, lib=lib)
        V = _gather(v, bt[0], w.block_size, 0, L)
        np.testing.assert_allclose(out[0, 0], V[t_star], rtol=0, atol=1e-12)


def pin_head_mapping(lib):
    """Every token of KV head j holds V = j + 1, so query head h must return
    floor(h / G) + 1 (contiguous query-head groups)."""
    w, inp = _small(batch=2, hq=8, hkv=2, d=8, bs=4, lengths=(9, 14))
    q, k, v, bt, ctx = _arrays(inp)
    v = v.copy()
    for j in range(w.num_kv_heads):
        v[:, :, j, :] = _bf16(np.full(v[:, :, j, :].shape, j + 1.0, np.float32))
    out, _ = oracle.attention(q, k, v, bt, ctx, w.scale, lib=lib)
    for h in range(w.num_q_heads):
        np.testing.assert_allclose(out[:, h, :], h // w.group + 1.0, rtol=0, atol=1e-12)


def pin_permutation_invariance(lib):
    """Re-scattering the same logical tokens under another physical
    permutation leaves the result bit-identical."""
    w, inp = _small(lengths=(7, 18, 25))
    q, k, v, bt, ctx = _arrays(inp)
    out, lse = oracle.attention(q, k, v, bt, ctx, w.scale, lib=lib)
    nb = k.shape[0]
    perm = np.random.default_rng(11).permutation(nb)          # old physical p -> new perm[p]
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.attention(q, k2, v2, bt2, ctx, w.scale, lib=lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_split_ranges(lib):
    for L, bs, S, maxL in ((0, 16, 3, 10), (1, 16, 1, 1), (37, 16, 3, 100), (100, 16, 3, 100),
                           (101, 32, 7, 4000), (4096, 16, 9, 4096), (5, 4, 8, 5)):
        n_max = -(-maxL // bs)
        chunk = max(1, -(-n_max // S))
        prev = 0
        for s in range(S):
            lo, hi = oracle.split_range(L, bs, S, maxL, s, lib=lib)
            assert lo == prev and lo <= hi, (L, bs, S, maxL, s, lo, hi)
            assert hi - lo <= chunk * bs
            if hi > lo:
                assert lo % (chunk * bs) == 0 and lo == s * chunk * bs
            prev = hi
        assert prev == L


def pin_split_merge(lib):
    w, inp = _small(batch=3, hq=4, hkv=2, d=16, bs=4, lengths=(1, 22, 47))
    q, k, v, bt, ctx = _arrays(inp)
    out, lse = oracle.attention(q, k, v, bt, ctx, w.scale, lib=lib)
    for S, maxL in ((1, 48), (2, 48), (3, 48), (5, 60), (8, 48), (13, 48), (40, 200)):
        o_p, lse_p = oracle.decode_partials(q, k, v, bt, ctx, w.scale, S, max_context_len=maxL, lib=lib)
        m_out, m_lse = oracle.merge_partials(o_p, lse_p, lib=lib)
        np.testing.assert_allclose(m_out, out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(m_lse, lse, rtol=1e-13, atol=1e-13)
        # every split is either empty (o = 0, lse = -inf) or finite
        empty = np.isneginf(lse_p)
        assert np.all(o_p[empty] == 0.0)
        assert np.all(np.isfinite(lse_p[~empty]))


def pin_merge_properties(lib):
    rng = np.random.default_rng(5)
    o = rng.standard_normal((4, 6))
    lse = rng.standard_normal(4) * 3
    a, la = oracle.merge(o[:2], lse[:2], lib=lib)
    b, lb = oracle.merge(o[2:], lse[2:], lib=lib)
    ab, lab = oracle.merge(np.stack([a, b]), np.array([la, lb]), lib=lib)
    full, lfull = oracle.merge(o, lse, lib=lib)
    np.testing.assert_allclose(ab, full, rtol=0, atol=1e-13)
    assert abs(lab - lfull) < 1e-13
    p = [2, 0, 3, 1]
    rev, lrev = oracle.merge(o[p], lse[p], lib=lib)
    np.testing.assert_allclose(rev, full, rtol=0, atol=1e-13)
    dup, ldup = oracle.merge(np.stack([o[0], o[0]]), np.array([lse[0], lse[0]]), lib=lib)
    np.testing.assert_allclose(dup, o[0], rtol=0, atol=1e-15)
    assert abs(ldup - (lse[0] + math.log(2))) < 1e-14
    single, lsingle = oracle.merge(o[1:2], lse[1:2], lib=lib)
    np.testing.assert_allclose(single, o[1], rtol=0, atol=1e-15)
    assert lsingle == lse[1]
    none, lnone = oracle.merge(np.zeros((3, 6)), np.full(3, -math.inf), lib=lib)
    assert np.all(none == 0.0) and lnone == -math.inf
    # weights e^{lse_i}: closed form against direct normalised weights
    wts = np.exp(lse - lse.max())
    np.testing.assert_allclose(full, (wts[:, None] * o).sum(0) / wts.sum(), rtol=0, atol=1e-13)
    # an empty partial first and one partial 895 above another: the weights
    # are e^{lse_i - max}, so the result is the top partial exactly (e^-895
    # is 0 in double); a shift by any lse but the maximum yields -inf here or
    # overflows
    top, ltop = oracle.merge(np.stack([np.zeros(6), o[0], o[1]]), np.array([-math.inf, 5.0, 900.0]), lib=lib)
    np.testing.assert_array_equal(top, o[1])
    assert ltop == 900.0


def pin_shift_invariance(lib):
    """Adding a constant c to every score (via a constant key component)
    leaves o unchanged and adds c to lse; with c = 2048 an oracle without the
    max subtraction overflows."""
    w, inp = _small(batch=1, hq=2, hkv=1, d=8, bs=4, lengths=(14,))
    q, k, v, bt, ctx = _arrays(inp)
    q2 = q.copy()
    q2[..., 0] = _bf16(np.full(q2[..., 0].shape, 64.0, np.float32))
    k_lo = k.copy()
    k_lo[..., 0] = _bf16(np.zeros(k_lo[..., 0].shape, np.float32))
    k_hi = k.copy()
    k_hi[..., 0] = _bf16(np.full(k_hi[..., 0].shape, 32.0, np.float32))
    o_lo, l_lo = oracle.attention(q2, k_lo, v, bt, ctx, 1.0, lib=lib)
    o_hi, l_hi = oracle.attention(q2, k_hi, v, bt, ctx, 1.0, lib=lib)
    np.testing.assert_allclose(o_hi, o_lo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_hi, l_lo + 64.0 * 32.0, rtol=1e-14, atol=0)


def pin_scipy_brute_force(lib):
    from scipy.special import logsumexp, softmax
    w, inp = _small(batch=2, hq=6, hkv=3, d=16, bs=8, lengths=(17, 40))
    q, k, v, bt, ctx = _arrays(inp)
    out, lse = oracle.attention(q, k, v, bt, ctx, w.scale, lib=lib)
    for b in range(w.batch):
        L = int(ctx[b])
        for h in range(w.num_q_heads):
            K = _gather(k, bt[b], w.block_size, h // w.group, L)
            V = _gather(v, bt[b], w.block_size, h // w.group, L)
            s = w.scale * (K @ _widen(q[b, h]))
            np.testing.assert_allclose(out[b, h], softmax(s) @ V, rtol=0, atol=1e-12)
            assert abs(lse[b, h] - logsumexp(s)) <= 1e-12 * max(1.0, abs(lse[b, h]))


def pin_append_random(lib):
    w, inp = _small(batch=4, hq=4, hkv=2, d=8, bs=4, lengths=(3, 4, 0, 10))
    q, k, v, bt, _ = _arrays(inp)
    kn, vn = wl.bf16_bits(inp.k_new), wl.bf16_bits(inp.v_new)
    ctx0 = inp.ctx_before.numpy()
    k2, v2, skipped = oracle.append(k, v, kn, vn, bt, ctx0, lib=lib)
    assert skipped == 0
    ek, ev = k.copy(), v.copy()
    for b in range(w.batch):
        p = int(ctx0[b])
        blk = bt[b, p // w.block_size]
        ek[blk, p % w.block_size] = kn[b]
        ev[blk, p % w.block_size] = vn[b]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    # an out-of-range position is skipped and writes nothing
    k3, v3, skipped = oracle.append(k, v, kn[:1], vn[:1], bt[:1], np.array([bt.shape[1] * w.block_size], np.int32), lib=lib)
    assert skipped == 1 and np.array_equal(k3, k) and np.array_equal(v3, v)


# ----------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# ----------------------------------------------------------------------------

def _torch_e4m3_table():
    """Values of all 256 E4M3 codes decoded by torch's float8_e4m3fn (an
    implementation independent of the oracle)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_decode(lib):
    # values fixed by the OCP E4M3 definition
    spec = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
            0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in spec.items():
        assert oracle.e4m3_to_f64(c, lib=lib) == v, hex(c)
    assert math.isnan(oracle.e4m3_to_f64(0x7F, lib=lib)) and math.isnan(oracle.e4m3_to_f64(0xFF, lib=lib))
    table = _torch_e4m3_table()
    mine = np.array([oracle.e4m3_to_f64(c, lib=lib) for c in range(256)])
    assert np.array_equal(np.isnan(mine), np.isnan(table))
    fin = ~np.isnan(table)
    assert np.array_equal(mine[fin], table[fin])


def pin_e4m3_encode(lib):
    """The code is the nearest finite E4M3 value (brute force over the table),
    ties to the even code, saturating at +-448; NaN -> 0x7F."""
    table = _torch_e4m3_table()
    finite = [c for c in range(256) if not np.isnan(table[c])]
    rng = np.random.default_rng(17)
    xs = np.concatenate([rng.standard_normal(3000) * 4, rng.standard_normal(1000) * 200,
                         rng.standard_normal(1000) * 0.01, rng.uniform(-460, 460, 500)]).astype(np.float32)
    # exact halfway points between neighbouring positive codes, and their negatives
    pos = sorted({table[c] for c in finite if table[c] > 0})
    mids = np.array([(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])], dtype=np.float64)
    xs = np.concatenate([xs, mids.astype(np.float32), -mids.astype(np.float32)])
    for x in xs:
        xd = float(x)
        if abs(xd) >= 448:
            want = 0x7E | (0x80 if xd < 0 else 0)
        else:
            best = min(abs(table[c] - xd) for c in finite)
            cands = [c for c in finite if abs(table[c] - xd) == best and (table[c] != 0 or c == (0x80 if np.signbit(xd) else 0))]
            cands = [c for c in cands if (c & 0x80) == (0x80 if np.signbit(xd) else 0)] or cands
            want = min(cands, key=lambda c: (c & 1, c))      # ties: even mantissa
        assert oracle.e4m3_from_f32(x, lib=lib) == want, (xd, hex(want))
    assert oracle.e4m3_from_f32(float("nan"), lib=lib) == 0x7F
    assert oracle.e4m3_from_f32(float("inf"), lib=lib) == 0x7E
    assert oracle.e4m3_from_f32(float("-inf"), lib=lib) == 0xFE
    assert oracle.e4m3_from_f32(1e30, lib=lib) == 0x7E


def _fp8_small(hq=4, hkv=2, d=16, bs=4, lengths=(5, 13, 22), seed=9):
    w, inp = _small(batch=len(lengths), hq=hq, hkv=hkv, d=d, bs=bs, lengths=lengths, seed=seed)
    rng = np.random.default_rng(seed)
    nb = inp.k_cache.shape[0]
    kc = rng.integers(0, 256, size=(nb, bs, hkv, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(nb, bs, hkv, d), dtype=np.uint8)
    # no NaN codes in the pool
    kc[(kc & 0x7F) == 0x7F] ^= 1
    vc[(vc & 0x7F) == 0x7F] ^= 1
    ks = (2.0 ** -rng.integers(3, 7, size=hkv)).astype(np.float32)
    vs = (2.0 ** -rng.integers(3, 7, size=hkv)).astype(np.float32)
    return w, inp, kc, vc, ks, vs


def pin_fp8_attention_is_dequantised_attention(lib):
    """Attention over E4M3 codes equals the bf16 attention over a cache that
    holds decode(code) * scale (exact in bf16 for power-of-two scales)."""
    w, inp, kc, vc, ks, vs = _fp8_small()
    q, _, _, bt, ctx = _arrays(inp)
    table = _torch_e4m3_table()
    kd = (table[kc] * ks[None, None, :, None]).astype(np.float32)
    vd = (table[vc] * vs[None, None, :, None]).astype(np.float32)
    out8, lse8 = oracle.attention_fp8(q, kc, vc, ks, vs, bt, ctx, w.scale, lib=lib)
    out16, lse16 = oracle.attention(q, _bf16(kd), _bf16(vd), bt, ctx, w.scale, lib=lib)
    np.testing.assert_allclose(out8, out16, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse8, lse16, rtol=1e-13, atol=1e-13)
    # and the split partials merge back to it
    o_p, l_p = oracle.decode_partials_fp8(q, kc, vc, ks, vs, bt, ctx, w.scale, 4, max_context_len=30, lib=lib)
    m_o, m_l = oracle.merge_partials(o_p, l_p, lib=lib)
    np.testing.assert_allclose(m_o, out8, rtol=0, atol=1e-12)


def pin_fp8_append(lib):
    """The new row's codes are E4M3(float(x) / scale) of its own KV head;
    nothing else changes."""
    w, inp, kc, vc, ks, vs = _fp8_small(lengths=(3, 4, 10))
    _, _, _, bt, _ = _arrays(inp)
    kn = _bf16(np.array([[[1.0, -2.0, 0.5, 288.0] * 4] * 2] * 3, np.float32))
    vn = _bf16(np.array([[[0.25, 3.0, -0.125, 2.0 ** -10] * 4] * 2] * 3, np.float32))
    ctx0 = inp.ctx_before.numpy()
    k2, v2, skipped = oracle.append_fp8(kc, vc, kn, vn, ks, vs, bt, ctx0, lib=lib)
    assert skipped == 0
    ek, ev = kc.copy(), vc.copy()
    knf, vnf = _widen(kn).astype(np.float32), _widen(vn).astype(np.float32)
    for b in range(w.batch):
        p = int(ctx0[b])
        blk = bt[b, p // w.block_size]
        for h in range(w.num_kv_heads):
            for d in range(w.head_dim):
                xk = knf[b, h, d] / np.float32(ks[h])
                xv = vnf[b, h, d] / np.float32(vs[h])
                ek[blk, p % w.block_size, h, d] = torch.tensor(min(max(float(xk), -448.0), 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).item()
                ev[blk, p % w.block_size, h, d] = torch.tensor(min(max(float(xv), -448.0), 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


# ----------------------------------------------------------------------------
# multi-query (chunked prefill / shared prefix) attention
# ----------------------------------------------------------------------------

def pin_golden_chunk(lib):
    g = _load_golden()["chunk_causal"]
    args = (_bf16(g["q"]), np.array(g["q_start"], np.int32), _bf16(g["k_cache"]), _bf16(g["v_cache"]),
            np.array(g["block_tables"], np.int32), np.array(g["ctx_lens"], np.int32), g["scale"])
    for causal, key in ((True, "causal"), (False, "full")):
        o, l = oracle.multiquery_partials(*args, causal, lib=lib)
        np.testing.assert_allclose(o[0], np.array(g["expect_%s_out" % key]), rtol=0, atol=1e-13)
        np.testing.assert_allclose(l[0], np.array(g["expect_%s_lse" % key]), rtol=0, atol=1e-13)


def _mq_case(lengths=(9, 30, 17), chunks=(3, 1, 5), hq=4, hkv=2, d=16, bs=4, seed=21):
    w, inp = _small(batch=len(lengths), hq=hq, hkv=hkv, d=d, bs=bs, lengths=lengths, seed=seed)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    rng = np.random.default_rng(seed)
    q = _bf16(np.round(rng.standard_normal((int(q_start[-1]), hq, d)) * 8) / 8)
    _, k, v, bt, ctx = _arrays(inp)
    return w, q, q_start, k, v, bt, ctx


def pin_multiquery_causal_rows(lib):
    """Causal query j of a chunk of C equals plain attention over the first
    L - C + j + 1 tokens; with C = 1 it is the decode partial itself."""
    w, q, qs, k, v, bt, ctx = _mq_case()
    o, l = oracle.multiquery_partials(q, qs, k, v, bt, ctx, w.scale, True, 3, max_context_len=32, lib=lib)
    m_o, m_l = oracle.merge_partials(o, l, lib=lib)
    for b in range(len(ctx)):
        C = int(qs[b + 1] - qs[b])
        for j in range(C):
            n = int(qs[b]) + j
            lim = np.array([int(ctx[b]) - C + j + 1], np.int32)
            ref_o, ref_l = oracle.attention(q[n:n + 1], k, v, bt[b:b + 1], lim, w.scale, lib=lib)
            np.testing.assert_allclose(m_o[n], ref_o[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(m_l[n], ref_l[0], rtol=1e-13, atol=1e-13)
    # C = 1 for every request: the decode partials, split by split
    qs1 = np.arange(len(ctx) + 1, dtype=np.int32)
    q1 = q[:len(ctx)]
    o1, l1 = oracle.multiquery_partials(q1, qs1, k, v, bt, ctx, w.scale, True, 3, max_context_len=32, lib=lib)
    od, ld = oracle.decode_partials(q1, k, v, bt, ctx, w.scale, 3, max_context_len=32, lib=lib)
    assert np.array_equal(o1, od) and np.array_equal(l1, ld)


def pin_multiquery_noncausal_rows(lib):
    w, q, qs, k, v, bt, ctx = _mq_case(seed=23)
    o, l = oracle.multiquery_partials(q, qs, k, v, bt, ctx, w.scale, False, lib=lib)
    for b in range(len(ctx)):
        for n in range(int(qs[b]), int(qs[b + 1])):
            ref_o, ref_l = oracle.attention(q[n:n + 1], k, v, bt[b:b + 1], ctx[b:b + 1], w.scale, lib=lib)
            np.testing.assert_allclose(o[0, n], ref_o[0], rtol=0, atol=1e-12)


def pin_cascade_merge(lib):
    """Shared prefix attended once (non-causal, one table) merged with each
    request's own suffix equals attention over prefix + suffix."""
    bs, P = 4, 12                                 # prefix: 3 shared blocks
    w, inp = _small(batch=3, hq=4, hkv=2, d=16, bs=bs, lengths=(P + 2, P + 7, P + 12), seed=29)
    q, k, v, bt, ctx = _arrays(inp)
    shared = bt[0, :P // bs].copy()
    full_bt = bt.copy()
    full_bt[:, :P // bs] = shared                 # every request's table starts with the shared blocks
    o_full, l_full = oracle.attention(q, k, v, full_bt, ctx, w.scale, lib=lib)
    qs = np.array([0, 3], np.int32)
    o_p, l_p = oracle.multiquery_partials(q, qs, k, v, shared[None, :], np.array([P], np.int32), w.scale, False,
                                          2, lib=lib)
    suffix_bt = np.full_like(bt, -1)
    suffix_bt[:, :bt.shape[1] - P // bs] = full_bt[:, P // bs:]
    o_s, l_s = oracle.decode_partials(q, k, v, suffix_bt, ctx - P, w.scale, 2, lib=lib)
    m_o, m_l = oracle.merge_partials(np.concatenate([o_p, o_s]), np.concatenate([l_p, l_s]), lib=lib)
    np.testing.assert_allclose(m_o, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m_l, l_full, rtol=1e-13, atol=1e-13)


PINS = [
    pin_bf16_widening, pin_golden_two_token, pin_golden_gqa, pin_golden_merge, pin_golden_append,
    pin_context_len_one, pin_identical_keys, pin_scale_zero, pin_dominant_key, pin_head_mapping,
    pin_permutation_invariance, pin_split_ranges, pin_split_merge, pin_merge_properties,
    pin_shift_invariance, pin_scipy_brute_force, pin_append_random,
    pin_e4m3_decode, pin_e4m3_encode, pin_fp8_attention_is_dequantised_attention, pin_fp8_append,
    pin_golden_chunk, pin_multiquery_causal_rows, pin_multiquery_noncausal_rows, pin_cascade_merge,
]
