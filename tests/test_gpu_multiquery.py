"""GPU parity of multi-query paged attention (chunked prefill / speculative
verify, causal; shared-prefix pass of cascade attention, non-causal)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import HostView, check_lse, check_out, check_partials, mq_impl
from paged_kv_decode_kf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kf():
    import __graft_entry__ as g
    g.build()
    from paged_kv_decode_kf_gb300 import kf
    assert kf.kf_get_device_error() == 0
    return kf


@pytest.fixture(autouse=True)
def no_device_error(kf):
    yield
    assert kf.kf_get_device_error() == 0, "a kernel raised a device error"


def _case(lengths, chunks, hq=32, hkv=8, d=128, bs=16, seed=5):
    """Contexts of L_b tokens (chunk included) with C_b query tokens each."""
    w = wl.Workload(name="mq", batch=len(lengths), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                    lengths=wl.Fixed(tuple(L - 1 for L in lengths)), seed=seed, spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + 1)
    q = torch.randn((int(q_start[-1]), hq, d), generator=gen, device="cuda", dtype=torch.bfloat16)
    return w, dev, q, torch.tensor(q_start, device="cuda")


def _host(dev, q, qs):
    return (wl.bf16_bits(q), qs.cpu().numpy(), wl.bf16_bits(dev.k_cache), wl.bf16_bits(dev.v_cache),
            dev.block_tables.cpu().numpy(), dev.ctx_after.cpu().numpy())


CASES = {
    "spec_verify": ((300, 1000, 77, 4096), (4, 4, 4, 4)),
    "mixed_chunks": ((9, 30, 17, 100, 64), (3, 1, 5, 32, 64)),
    "long_chunk": ((2048, 700), (128, 700)),
}


IMPLS = ["mma", "tc05", "tc05x2", "tc05w", "tc05p"]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("S", [1, 3])
def test_multiquery(kf, name, causal, S, impl):
    lengths, chunks = CASES[name]
    w, dev, q, qs = _case(lengths, chunks)
    hq_, qs_h, k, v, bt, ctx = _host(dev, q, qs)
    maxL, maxC = int(max(lengths)), int(max(chunks))
    with mq_impl(impl):
        o_p, l_p = kf.kf_paged_multiquery_attention(q, qs, dev.k_cache, dev.v_cache, dev.block_tables,
                                                    dev.ctx_after, causal, maxL, maxC, w.scale, S)
    out, lse = kf.kf_merge_partials(o_p, l_p)
    ref_po, ref_pl = oracle.multiquery_partials(hq_, qs_h, k, v, bt, ctx, w.scale, causal, S, max_context_len=maxL)
    check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, name + " partials")
    ref_o, ref_l = oracle.merge_partials(ref_po, ref_pl)
    check_out(out.cpu().numpy(), ref_o, name + " out")
    check_lse(lse.cpu().numpy(), ref_l, name + " lse")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (8, 1)])
@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32)])
def test_multiquery_shapes(kf, hq, hkv, d, bs, impl):
    w, dev, q, qs = _case((40, 97, 33), (7, 2, 33), hq=hq, hkv=hkv, d=d, bs=bs, seed=hq + hkv + d)
    hq_, qs_h, k, v, bt, ctx = _host(dev, q, qs)
    with mq_impl(impl):
        o_p, l_p = kf.kf_paged_multiquery_attention(q, qs, dev.k_cache, dev.v_cache, dev.block_tables,
                                                    dev.ctx_after, True, 97, 33, w.scale, 2)
    ref_po, ref_pl = oracle.multiquery_partials(hq_, qs_h, k, v, bt, ctx, w.scale, True, 2, max_context_len=97)
    check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, "mq shapes")


@pytest.mark.parametrize("mode", ["concurrent", "serial", "calls"])
@pytest.mark.parametrize("impl", IMPLS)
def test_cascade_prefix_plus_suffix(kf, impl, mode):
    """Prefix attended once for all requests, merged with each suffix, equals
    decode attention over each request's full table -- as the prefix pass and
    the suffix step on two streams then one merge, as three launches in a row
    (prefix pass, prefix merge, kf_decode_step_merge_partials), or four."""
    from paged_kv_decode_kf_gb300.step import CascadeStep
    w = wl.scaled(wl.CONFIGS["cascade"], batch=6, lengths=wl.Fixed((5, 70, 300, 1, 16, 999)))
    dev = wl.make_inputs(w, "cuda")
    hv_k, hv_v = wl.bf16_bits(dev.k_cache), wl.bf16_bits(dev.v_cache)
    step = CascadeStep(dev, fused_suffix=mode != "calls", concurrent=mode == "concurrent")
    with mq_impl(impl):
        step.run()
    torch.cuda.synchronize()
    k2, v2, _ = oracle.append(hv_k, hv_v, wl.bf16_bits(dev.k_new), wl.bf16_bits(dev.v_new),
                              dev.block_tables.cpu().numpy(), dev.ctx_before.cpu().numpy())
    ref_o, ref_l = oracle.attention(wl.bf16_bits(dev.q), k2, v2, dev.block_tables.cpu().numpy(),
                                    dev.ctx_after.cpu().numpy(), w.scale)
    check_out(step.out.cpu().numpy(), ref_o, "cascade out")
    check_lse(step.lse.cpu().numpy(), ref_l, "cascade lse")


def test_cascade_concurrent_streams(kf):
    """The concurrent cascade step forks its suffix step onto a second stream
    and joins before the merge: run on a caller's non-default stream, on the
    current stream, or given a raw stream handle (then one stream, in order),
    it gives the same output and lse bit for bit."""
    from paged_kv_decode_kf_gb300.step import CascadeStep
    w = wl.scaled(wl.CONFIGS["cascade"], batch=6, lengths=wl.Fixed((5, 70, 300, 1, 16, 999)))
    dev = wl.make_inputs(w, "cuda")
    step = CascadeStep(dev)
    assert step.concurrent
    step.run()
    torch.cuda.synchronize()
    ref_o, ref_l = step.out.clone(), step.lse.clone()
    s = torch.cuda.Stream()
    for how in ("torch stream", "raw handle"):
        step.out.zero_()
        step.lse.zero_()
        s.wait_stream(torch.cuda.current_stream())
        step.run(s if how == "torch stream" else s.cuda_stream)
        s.synchronize()
        assert torch.equal(step.out, ref_o) and torch.equal(step.lse, ref_l), how


@pytest.mark.parametrize("impl", IMPLS)
def test_multiquery_rejects_bad_q_start(kf, impl):
    w, dev, q, qs = _case((40, 50), (3, 3))
    bad = torch.tensor([0, 3, 99], dtype=torch.int32, device="cuda")   # past num_q_tokens
    with mq_impl(impl):
        kf.kf_paged_multiquery_attention(q, bad, dev.k_cache, dev.v_cache, dev.block_tables, dev.ctx_after,
                                         True, 50, 3, w.scale, 1)
    assert kf.kf_get_device_error() & kf.KF_DEVERR_CONTEXT_LEN


def test_cascade_full_size_sampled(kf):
    """The cascade workload at full size (64 requests behind a 16384-token
    shared prefix, 4 query heads per KV head: 256 rows per KV head, the
    tcgen05 kernel's shape) in the launch configuration the benchmark times;
    sampled requests against the oracle over their whole tables."""
    from paged_kv_decode_kf_gb300.step import CascadeStep
    w = wl.CONFIGS["cascade"]
    dev = wl.make_inputs(w, "cuda")
    reqs = [0, 1, 31, 62, 63]
    hv = HostView(dev, reqs)
    step = CascadeStep(dev)
    step.run()
    torch.cuda.synchronize()
    k2, v2 = hv.appended()
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, w.scale)
    check_out(step.out.float().cpu().numpy()[reqs], ref_o, "cascade full out")
    check_lse(step.lse.cpu().numpy()[reqs], ref_l, "cascade full lse")


def test_decode_step_merge_partials_extra_slots(kf):
    """One split plus extra partials (the single work unit counts itself as the
    last and merges); an extra slot with lse = -inf is skipped without reading
    its o (NaN here); bf16 output."""
    from paged_kv_decode_kf_gb300.step import CascadeStep
    w = wl.scaled(wl.CONFIGS["cascade"], batch=5, lengths=wl.Fixed((40, 3, 200, 17, 64)))
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    step = CascadeStep(dev, suffix_splits=1)
    step.prefix()
    Sp = step.Sp
    B, Hq, D = w.batch, w.num_q_heads, w.head_dim
    ex_o = torch.cat([step.out_partial[:Sp], torch.full((1, B, Hq, D), float("nan"), device="cuda")])
    ex_l = torch.cat([step.lse_partial[:Sp], torch.full((1, B, Hq), float("-inf"), device="cuda")])
    ws = kf.make_workspace(B, Hq, w.num_kv_heads, D, 1)
    out, lse = kf.kf_decode_step_merge_partials(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache,
                                                dev.suffix_tables, dev.suffix_ctx_before, step.max_suffix, w.scale,
                                                1, ex_o, ex_l, ws, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    k2, v2 = hv.appended()
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, w.scale)
    check_out(out.float().cpu().numpy(), ref_o, "merge_partials out")
    check_lse(lse.cpu().numpy(), ref_l, "merge_partials lse")
    al = lambda x: (x + 255) // 256 * 256
    off = al(B * Hq * D * 4) + al(B * Hq * 4)    # workspace: partials (1 split), lse, counters
    assert int(ws[off:off + B * w.num_kv_heads * 4].view(torch.int32).abs().sum()) == 0, "counters not reset"


def test_chunk_full_size_sampled(kf):
    """The chunked-prefill workload at full size (4 requests, 1024 causal chunk
    queries each over U[4K,12K] cached tokens: 4096 rows per KV head, the wide
    tcgen05 kernel) in the configuration the benchmark times; queries at the
    chunk's start, middle and end against the oracle over their own limits."""
    from paged_kv_decode_kf_gb300.step import ChunkStep
    w = wl.CONFIGS["chunk"]
    dev = wl.make_inputs(w, "cuda")
    step = ChunkStep(dev)
    step.run()
    torch.cuda.synchronize()
    C = w.chunk
    reqs = [0, w.batch - 1]
    hv = HostView(dev, reqs)
    for idx, b in enumerate(reqs):
        L = int(hv.ctx_after[idx])
        js = [0, 1, C // 2, C - 2, C - 1]
        rows = [b * C + j for j in js]
        q = wl.bf16_bits(dev.q_chunk[rows])
        bt = np.repeat(hv.tables[0][idx:idx + 1], len(js), axis=0)
        lim = np.array([L - C + j + 1 for j in js], np.int32)
        ref_o, ref_l = oracle.attention(q, hv.k, hv.v, bt, lim, w.scale)
        check_out(step.out[rows].cpu().numpy(), ref_o, "chunk out, request %d" % b)
        check_lse(step.lse[rows].cpu().numpy(), ref_l, "chunk lse, request %d" % b)


def test_specverify_full_size_sampled(kf):
    """The speculative-verify workload at full size (64 requests of U[3.5K,4K]
    cached tokens, 4 draft queries each, causal: 16 rows per KV head, the
    one-tile tcgen05 kernel) in the configuration the benchmark times; every
    draft query of sampled requests against the oracle over its own limit."""
    from paged_kv_decode_kf_gb300.step import ChunkStep
    w = wl.CONFIGS["specverify"]
    dev = wl.make_inputs(w, "cuda")
    step = ChunkStep(dev)
    step.run()
    torch.cuda.synchronize()
    C = w.chunk
    reqs = [0, 17, w.batch - 1]
    hv = HostView(dev, reqs)
    for idx, b in enumerate(reqs):
        L = int(hv.ctx_after[idx])
        rows = [b * C + j for j in range(C)]
        q = wl.bf16_bits(dev.q_chunk[rows])
        bt = np.repeat(hv.tables[0][idx:idx + 1], C, axis=0)
        lim = np.array([L - C + j + 1 for j in range(C)], np.int32)
        ref_o, ref_l = oracle.attention(q, hv.k, hv.v, bt, lim, w.scale)
        check_out(step.out[rows].cpu().numpy(), ref_o, "specverify out, request %d" % b)
        check_lse(step.lse[rows].cpu().numpy(), ref_l, "specverify lse, request %d" % b)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("causal", [True, False])
def test_multiquery_nonfinite_garbage_past_context(kf, impl, causal):
    """Slots past each request's end (same blocks) and unused blocks hold
    NaN/Inf: results must be unaffected -- with query tiles whose warps hold
    no row (4 tokens x G 4 = 16 of 128 rows), partly filled warps (12 and 44
    rows) and full ones."""
    lengths, chunks = (300, 1000, 77, 4096, 45, 130), (4, 4, 3, 4, 11, 32)
    w, dev, q, qs = _case(lengths, chunks, seed=11)
    bt = dev.block_tables.cpu().numpy()
    L = dev.ctx_after.cpu().numpy()
    used = set()
    for b in range(w.batch):
        n = -(-int(L[b]) // w.block_size)
        used |= set(bt[b, :n].tolist())
        last = bt[b, n - 1]
        for t in range(int(L[b]) % w.block_size or w.block_size, w.block_size):
            dev.k_cache[last, t] = float("nan")
            dev.v_cache[last, t] = float("inf") if t % 2 else float("nan")
    for p in range(dev.num_blocks):
        if p not in used:
            dev.k_cache[p] = float("nan")
            dev.v_cache[p] = float("nan")
    hq_, qs_h, k, v, bt_h, ctx = _host(dev, q, qs)
    maxL, maxC = int(max(lengths)), int(max(chunks))
    for S in (1, 3):
        with mq_impl(impl):
            o_p, l_p = kf.kf_paged_multiquery_attention(q, qs, dev.k_cache, dev.v_cache, dev.block_tables,
                                                        dev.ctx_after, causal, maxL, maxC, w.scale, S)
        ref_po, ref_pl = oracle.multiquery_partials(hq_, qs_h, k, v, bt_h, ctx, w.scale, causal, S,
                                                    max_context_len=maxL)
        check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, "garbage partials")
