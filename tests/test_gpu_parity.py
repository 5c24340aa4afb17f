"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bar: KV append bit-exact; every output within max|err| <= 8e-3 and
mean|err| <= 1e-3; lse within 1e-4 * max(1, |lse|); empty partials exactly
(0, -inf). Both decode kernels (tensor-core "tc", CUDA-core "simt") are
checked.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import HostView, check_lse, check_out, check_partials, decode_impl
from paged_kv_decode_kf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
IMPLS = ["tc", "simt"]


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


def _host_all(inp):
    return HostView(inp, range(inp.workload.batch))


# ----------------------------------------------------------------------------
# the tiny workload, every output element
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("S", [1, 3])
def test_tiny_workload(kf, impl, S):
    w = wl.CONFIGS["tiny"]
    host = wl.make_inputs(w, "cpu")
    dev = host.to("cuda")
    q, bt, ctx = wl.bf16_bits(host.q), host.block_tables.numpy(), host.ctx_after.numpy()
    with decode_impl(impl):
        kf.kf_append_kv(dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, dev.ctx_before)
        o_p, l_p = kf.kf_paged_decode_attention(dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                                                dev.ctx_after, dev.max_ctx_after, w.scale, S)
        out, lse = kf.kf_merge_partials(o_p, l_p)
        out16, _ = kf.kf_merge_partials(o_p, l_p, out_dtype=torch.bfloat16, want_lse=False)
    k2, v2, _ = oracle.append(wl.bf16_bits(host.k_cache), wl.bf16_bits(host.v_cache),
                              wl.bf16_bits(host.k_new), wl.bf16_bits(host.v_new),
                              host.block_tables.numpy(), host.ctx_before.numpy())
    assert np.array_equal(wl.bf16_bits(dev.k_cache), k2)
    assert np.array_equal(wl.bf16_bits(dev.v_cache), v2)
    ref_po, ref_pl = oracle.decode_partials(q, k2, v2, bt, ctx, w.scale, S, max_context_len=dev.max_ctx_after)
    check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, "tiny partials")
    ref_o, ref_l = oracle.attention(q, k2, v2, bt, ctx, w.scale)
    check_out(out.cpu().numpy(), ref_o, "tiny out")
    check_lse(lse.cpu().numpy(), ref_l, "tiny lse")
    check_out(out16.float().cpu().numpy(), ref_o, "tiny out bf16")


# ----------------------------------------------------------------------------
# oracle-sized versions of the large workloads: several tiles, ragged tails
# ----------------------------------------------------------------------------

SMALL = {
    "llama8b": (1, 17, 250, 777, 3840),
    "longctx": (12345, 40, 8191),
    "shard4": (3000, 64, 0, 15, 16),
    "ragged": (31, 32, 63, 1000, 4095, 0, 64),
}


def _small(name):
    lens = SMALL[name]
    return wl.scaled(wl.CONFIGS[name], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=5)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("splits", ["plan", 1, 7])
def test_small_workloads(kf, impl, name, splits):
    from paged_kv_decode_kf_gb300.step import DecodeStep
    w = _small(name)
    dev = wl.make_inputs(w, "cuda")
    tables = [dev.block_tables] + [s.block_tables for s in dev.shards]
    if dev.tail_tables is not None:
        tables.append(dev.tail_tables)
    hv = HostView(dev, range(w.batch), tables)
    with decode_impl(impl):
        step = DecodeStep(dev, num_splits=None if splits == "plan" else splits)
        step.run()
    torch.cuda.synchronize()
    if w.shards:
        k2, v2 = hv.appended(table=len(tables) - 1, ctx_before=dev.tail_ctx_before.cpu().numpy())
    else:
        k2, v2 = hv.appended()
    # the append, checked on the rows it should write
    used = sorted({int(x) for x in dev.block_tables.cpu().numpy().ravel() if x >= 0})
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    assert np.array_equal(wl.bf16_bits(dev.k_cache.index_select(0, idx)), k2)
    assert np.array_equal(wl.bf16_bits(dev.v_cache.index_select(0, idx)), v2)
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, w.scale)
    check_out(step.out.cpu().numpy(), ref_o, name + " out")
    check_lse(step.lse.cpu().numpy(), ref_l, name + " lse")
    S = step.num_splits
    for j, (bt, ctx, max_ctx) in enumerate(step.views):
        tab = hv.tables[0] if not w.shards else hv.tables[1 + j]
        ref_po, ref_pl = oracle.decode_partials(hv.q, k2, v2, tab, ctx.cpu().numpy(), w.scale, S,
                                                max_context_len=max_ctx)
        check_partials(step.out_partial[j * S:(j + 1) * S].cpu().numpy(),
                       step.lse_partial[j * S:(j + 1) * S].cpu().numpy(), ref_po, ref_pl,
                       "%s view %d" % (name, j))


# ----------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration, sampled rows
# ----------------------------------------------------------------------------

def _sample_requests(dev, k=6):
    L = dev.ctx_after.cpu().numpy()
    order = np.argsort(L)
    pick = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    if dev.workload.name == "ragged":
        pick |= {0, 5}                       # two of the fresh-block appends
    rng = np.random.default_rng(dev.workload.seed)
    while len(pick) < min(k, dev.workload.batch):
        pick.add(int(rng.integers(0, dev.workload.batch)))
    return sorted(pick)


@pytest.mark.parametrize("name", ["llama8b", "longctx", "shard4", "ragged"])
def test_full_size_sampled(kf, name):
    from paged_kv_decode_kf_gb300.step import DecodeStep
    w = wl.CONFIGS[name]
    dev = wl.make_inputs(w, "cuda")
    reqs = _sample_requests(dev)
    tables = [dev.block_tables] + [s.block_tables for s in dev.shards]
    if dev.tail_tables is not None:
        tables.append(dev.tail_tables)
    hv = HostView(dev, reqs, tables)
    k_before, v_before = dev.k_cache.clone(), dev.v_cache.clone()
    step = DecodeStep(dev)
    step.run()
    torch.cuda.synchronize()

    # append: every request's new row landed, and nothing else changed
    bt = dev.block_tables.cpu().numpy()
    pos = dev.ctx_before.cpu().numpy().astype(np.int64)
    phys = torch.tensor(bt[np.arange(w.batch), pos // w.block_size], dtype=torch.long, device="cuda")
    slot = torch.tensor(pos % w.block_size, dtype=torch.long, device="cuda")
    assert torch.equal(dev.k_cache[phys, slot], dev.k_new) and torch.equal(dev.v_cache[phys, slot], dev.v_new)
    dev.k_cache[phys, slot] = k_before[phys, slot]
    dev.v_cache[phys, slot] = v_before[phys, slot]
    assert torch.equal(dev.k_cache, k_before) and torch.equal(dev.v_cache, v_before)
    dev.k_cache[phys, slot] = dev.k_new
    dev.v_cache[phys, slot] = dev.v_new
    del k_before, v_before

    if w.shards:
        k2, v2 = hv.appended(table=len(tables) - 1, ctx_before=dev.tail_ctx_before.cpu().numpy()[reqs])
    else:
        k2, v2 = hv.appended()
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, w.scale)
    check_out(step.out.cpu().numpy()[reqs], ref_o, name + " out")
    check_lse(step.lse.cpu().numpy()[reqs], ref_l, name + " lse")
    S = step.num_splits
    for j, (bt_j, ctx, max_ctx) in enumerate(step.views):
        tab = hv.tables[0] if not w.shards else hv.tables[1 + j]
        ref_po, ref_pl = oracle.decode_partials(hv.q, k2, v2, tab, ctx.cpu().numpy()[reqs], w.scale, S,
                                                max_context_len=max_ctx)
        check_partials(step.out_partial[j * S:(j + 1) * S].cpu().numpy()[:, reqs],
                       step.lse_partial[j * S:(j + 1) * S].cpu().numpy()[:, reqs], ref_po, ref_pl,
                       "%s view %d" % (name, j))


# ----------------------------------------------------------------------------
# edge cases
# ----------------------------------------------------------------------------

def _attend(kf, dev, ctx, S, max_ctx=None, table=None):
    bt = dev.block_tables if table is None else table
    mc = int(ctx.max().item()) if max_ctx is None else max_ctx
    o_p, l_p = kf.kf_paged_decode_attention(dev.q, dev.k_cache, dev.v_cache, bt, ctx, mc,
                                            dev.workload.scale, S)
    out, lse = kf.kf_merge_partials(o_p, l_p)
    return o_p, l_p, out, lse


@pytest.mark.parametrize("impl", IMPLS)
def test_empty_contexts_and_excess_splits(kf, impl):
    """Context 0 (every split empty -> merged out 0, lse -inf) beside short
    requests, with far more splits than blocks."""
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=4, lengths=wl.Fixed((0, 1, 20, 47)))
    dev = wl.make_inputs(w, "cuda")
    ctx = torch.tensor([0, 1, 20, 47], dtype=torch.int32, device="cuda")
    hv = _host_all(dev)
    for S in (1, 3, 40):
        with decode_impl(impl):
            o_p, l_p, out, lse = _attend(kf, dev, ctx, S)
        ref_po, ref_pl = oracle.decode_partials(hv.q, hv.k, hv.v, hv.tables[0], ctx.cpu().numpy(),
                                                w.scale, S, max_context_len=47)
        check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, "S=%d" % S)
        ref_o, ref_l = oracle.attention(hv.q, hv.k, hv.v, hv.tables[0], ctx.cpu().numpy(), w.scale)
        assert np.all(out[0].cpu().numpy() == 0.0) and np.all(np.isneginf(lse[0].cpu().numpy()))
        check_out(out[1:].cpu().numpy(), ref_o[1:], "S=%d" % S)
        check_lse(lse.cpu().numpy(), ref_l, "S=%d" % S)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (32, 8), (64, 8)])
@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32), (64, 32), (128, 16)])
def test_shape_sweep(kf, impl, hq, hkv, d, bs):
    w = wl.Workload(name="sweep", batch=3, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                    lengths=wl.Fixed((5, 2 * bs + 3, 9 * bs)), seed=77 + hq + hkv + d + bs, spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    hv = _host_all(dev)
    for S in (1, 4):
        with decode_impl(impl):
            o_p, l_p, out, lse = _attend(kf, dev, dev.ctx_after, S)
        ref_po, ref_pl = oracle.decode_partials(hv.q, hv.k, hv.v, hv.tables[0], hv.ctx_after, w.scale, S,
                                                max_context_len=dev.max_ctx_after)
        check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, "sweep")
        ref_o, ref_l = oracle.attention(hv.q, hv.k, hv.v, hv.tables[0], hv.ctx_after, w.scale)
        check_out(out.cpu().numpy(), ref_o, "sweep out")
        check_lse(lse.cpu().numpy(), ref_l, "sweep lse")


@pytest.mark.parametrize("impl", IMPLS)
def test_nonfinite_garbage_past_context(kf, impl):
    """Slots past each request's end (same blocks) and unused blocks hold
    NaN/Inf: results must be unaffected."""
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=3, lengths=wl.Fixed((17, 33, 100)), spare_blocks=4)
    dev = wl.make_inputs(w, "cuda")
    hv = _host_all(dev)
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
    for S in (1, 5):
        with decode_impl(impl):
            o_p, l_p, out, lse = _attend(kf, dev, dev.ctx_after, S)
        ref_o, ref_l = oracle.attention(hv.q, hv.k, hv.v, hv.tables[0], hv.ctx_after, w.scale)
        check_out(out.cpu().numpy(), ref_o, "garbage out")
        check_lse(lse.cpu().numpy(), ref_l, "garbage lse")


@pytest.mark.parametrize("impl", IMPLS)
def test_longest_context(kf, impl):
    """One request at the largest context of the workloads (256K + 1)."""
    w = wl.scaled(wl.CONFIGS["longctx"], batch=1, lengths=wl.Fixed((262144,)))
    dev = wl.make_inputs(w, "cuda")
    hv = _host_all(dev)
    S = kf.kf_choose_num_splits(1, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                dev.max_ctx_after, dev.ctx_after.cpu().numpy())
    assert S > 1
    with decode_impl(impl):
        o_p, l_p, out, lse = _attend(kf, dev, dev.ctx_after, S)
    ref_o, ref_l = oracle.attention(hv.q, hv.k, hv.v, hv.tables[0], hv.ctx_after, w.scale)
    check_out(out.cpu().numpy(), ref_o, "256K out")
    check_lse(lse.cpu().numpy(), ref_l, "256K lse")


@pytest.mark.parametrize("hpc", ["1", "2", "4", "8"])
def test_heads_per_cta_variants(kf, hpc, monkeypatch):
    monkeypatch.setenv("KF_TC_HPC", hpc)
    w = wl.scaled(wl.CONFIGS["ragged"], batch=4, lengths=wl.Fixed((100, 31, 700, 64)))
    dev = wl.make_inputs(w, "cuda")
    hv = _host_all(dev)
    with decode_impl("tc"):
        o_p, l_p, out, lse = _attend(kf, dev, dev.ctx_after, 3)
    ref_o, ref_l = oracle.attention(hv.q, hv.k, hv.v, hv.tables[0], hv.ctx_after, w.scale)
    check_out(out.cpu().numpy(), ref_o, "hpc out")
    check_lse(lse.cpu().numpy(), ref_l, "hpc lse")


def test_merge_kernel_alone(kf):
    """The merge on partials produced by the oracle (rounded to fp32), with
    empty partials and an all-empty row; f32 and bf16 outputs."""
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=3, lengths=wl.Fixed((40, 300, 9)))
    host = wl.make_inputs(w, "cpu")
    hv = _host_all(host)
    ctx = hv.ctx_after.copy()
    ctx[2] = 0
    po, pl = oracle.decode_partials(hv.q, hv.k, hv.v, hv.tables[0], ctx, w.scale, 6,
                                    max_context_len=int(ctx.max()))
    po32 = torch.tensor(po.astype(np.float32), device="cuda")
    pl32 = torch.tensor(pl.astype(np.float32), device="cuda")
    ref_o, ref_l = oracle.merge_partials(po32.double().cpu().numpy(), pl32.double().cpu().numpy())
    out, lse = kf.kf_merge_partials(po32, pl32)
    check_out(out.cpu().numpy(), ref_o, "merge f32")
    check_lse(lse.cpu().numpy(), ref_l, "merge lse")
    assert np.all(out[2].cpu().numpy() == 0) and np.all(np.isneginf(lse[2].cpu().numpy()))
    out16, _ = kf.kf_merge_partials(po32, pl32, out_dtype=torch.bfloat16, want_lse=False)
    # bf16 output is the fp32 result rounded to nearest even
    assert torch.equal(out16, out.to(torch.bfloat16))


def test_device_errors_are_reported(kf):
    """Bad values only the GPU sees: reported in the error word, no fault."""
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=2, lengths=wl.Fixed((20, 40)))
    dev = wl.make_inputs(w, "cuda")
    bad = dev.block_tables.clone()
    bad[1, 0] = dev.num_blocks + 5
    for impl in IMPLS:
        with decode_impl(impl):
            _attend(kf, dev, dev.ctx_after, 2, table=bad)
        assert kf.kf_get_device_error() & kf.KF_DEVERR_BLOCK_ID
        over = dev.ctx_after.clone()
        over[0] = dev.block_tables.shape[1] * w.block_size + 1
        with decode_impl(impl):
            _attend(kf, dev, over, 2, max_ctx=int(over.max().item()))
        assert kf.kf_get_device_error() & kf.KF_DEVERR_CONTEXT_LEN
        with decode_impl(impl):
            _attend(kf, dev, dev.ctx_after, 2, max_ctx=10)
        assert kf.kf_get_device_error() & kf.KF_DEVERR_MAX_CONTEXT
    bt = dev.block_tables.cpu().numpy()
    pos = dev.ctx_before.cpu().numpy()
    far = dev.ctx_before.clone()
    far[0] = dev.block_tables.shape[1] * w.block_size     # request 0: past its table
    k0 = dev.k_cache.clone()
    kf.kf_append_kv(dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, far)
    assert kf.kf_get_device_error() & kf.KF_DEVERR_APPEND_POS
    bad_app = dev.block_tables.clone()
    bad_app[1, pos[1] // w.block_size] = -1                 # request 1: bad block at its position
    kf.kf_append_kv(dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, bad_app, dev.ctx_before)
    assert kf.kf_get_device_error() & kf.KF_DEVERR_BLOCK_ID
    assert kf.kf_get_device_error() == 0                     # read clears
    # only the two valid appends wrote (request 1 first, request 0 second)
    changed = set(torch.nonzero(dev.k_cache.ne(k0).any(dim=3).any(dim=2).any(dim=1)).flatten().tolist())
    assert changed == {int(bt[1, pos[1] // w.block_size]), int(bt[0, pos[0] // w.block_size])}


def test_side_stream_and_determinism(kf):
    from paged_kv_decode_kf_gb300.step import DecodeStep
    w = wl.scaled(wl.CONFIGS["ragged"], batch=6, lengths=wl.Fixed((500, 31, 2000, 64, 1, 777)))
    dev = wl.make_inputs(w, "cuda")
    step = DecodeStep(dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run()
        a = step.out.clone()
        step.run()                            # the append rewrites the same rows
        b = step.out.clone()
    s.synchronize()
    assert torch.equal(a, b)
    step.run()
    torch.cuda.synchronize()
    assert torch.equal(a, step.out)
