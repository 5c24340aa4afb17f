"""GPU parity of the decode step on the balanced schedule (num_splits =
KF_SPLITS_BALANCED: the batch's 16-token stages cut into equal runs, one per
CTA of a single wave, runs crossing request boundaries) against the fp64
oracle, for bf16 and FP8 caches, with and without extra partials."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import HostView, check_lse, check_out
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


def _ws(kf, w):
    return kf.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, kf.KF_SPLITS_BALANCED)


def _counters_zero(ws, w):
    n = w.batch * w.num_kv_heads
    return int(ws[:n * 4].view(torch.int32).abs().sum()) == 0   # the counters lead the balanced layout


def _step(kf, dev, ws, out_dtype=torch.float32):
    w = dev.workload
    return kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.ctx_before, dev.max_ctx_after, w.scale, kf.KF_SPLITS_BALANCED, ws,
                             out_dtype=out_dtype)


def _check_bf16(dev, hv, out, lse, what, reqs=None):
    k2, v2 = hv.appended()
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, dev.workload.scale)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    if reqs is not None:
        o, l = o[reqs], l[reqs]
    check_out(o, ref_o, what + " out")
    check_lse(l, ref_l, what + " lse")
    return k2, v2


SMALL = {
    "llama8b": (1, 17, 250, 777, 3840, 15, 16),
    "longctx": (12345, 40, 8191),
    "ragged": (31, 32, 63, 1000, 4095, 0, 64),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_small(kf, name, dtype):
    lens = SMALL[name]
    w = wl.scaled(wl.CONFIGS[name], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=3)
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    ws = _ws(kf, w)
    out, lse = _step(kf, dev, ws, dtype)
    k2, v2 = _check_bf16(dev, hv, out, lse, "%s balanced" % name)
    used = sorted({int(x) for x in dev.block_tables.cpu().numpy().ravel() if x >= 0})
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    assert np.array_equal(wl.bf16_bits(dev.k_cache.index_select(0, idx)), k2)
    assert np.array_equal(wl.bf16_bits(dev.v_cache.index_select(0, idx)), v2)
    assert _counters_zero(ws, w)


def test_many_short_requests(kf):
    """Hundreds of 1- to 40-token requests: a CTA's run spans many requests,
    most of them complete inside it (direct rows), a few cut at its ends."""
    rng = np.random.default_rng(7)
    lens = tuple(int(x) for x in rng.integers(0, 40, size=300))
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    ws = _ws(kf, w)
    out, lse = _step(kf, dev, ws)
    _check_bf16(dev, hv, out, lse, "short requests")
    assert _counters_zero(ws, w)


def test_one_long_request(kf):
    """One request cut into every CTA's run: the merge takes one partial per CTA."""
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=1, lengths=wl.Fixed((50000,)), spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, [0])
    ws = _ws(kf, w)
    out, lse = _step(kf, dev, ws)
    _check_bf16(dev, hv, out, lse, "one long request")
    assert _counters_zero(ws, w)


def test_fewer_stages_than_ctas(kf):
    """A batch with fewer 16-token stages than CTAs (most runs empty)."""
    w = wl.scaled(wl.CONFIGS["ragged"], batch=3, lengths=wl.Fixed((0, 5, 20)), spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    ws = _ws(kf, w)
    out, lse = _step(kf, dev, ws)
    _check_bf16(dev, hv, out, lse, "fewer stages")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (8, 1), (64, 8)])
@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32)])
def test_shape_sweep(kf, hq, hkv, d, bs):
    w = wl.Workload(name="balsweep", batch=5, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                    lengths=wl.Fixed((5, 2 * bs + 3, 9 * bs, 0, 700)), seed=191 + hq + hkv + d + bs,
                    spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    ws = _ws(kf, w)
    out, lse = _step(kf, dev, ws)
    _check_bf16(dev, hv, out, lse, "sweep %d/%d d%d bs%d" % (hq, hkv, d, bs))


def test_repeated_steps_match_split_rule(kf):
    """Consecutive balanced steps agree bit for bit (counters back at zero)
    and match the split-rule step up to rounding: the two partitions round P
    (a bf16 pair, ~16 significant bits) against different running maxima, so
    |o| <= max|v| ~ 4 differs by up to ~4 * 2^-16 per row in the worst case
    and ~1e-6 in practice."""
    w = wl.scaled(wl.CONFIGS["ragged"], batch=6, lengths=wl.Fixed((500, 31, 2000, 64, 1, 777)))
    dev = wl.make_inputs(w, "cuda")
    ws = _ws(kf, w)
    outs = [_step(kf, dev, ws)[0].clone() for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert _counters_zero(ws, w)
    ws6 = kf.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, 6)
    ref, _ = kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                               dev.ctx_before, dev.max_ctx_after, w.scale, 6, ws6)
    assert torch.allclose(outs[0], ref, rtol=0, atol=2e-5)


def test_static_entry(kf):
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=4, lengths=wl.Fixed((100, 3000, 7, 1500)))
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device="cuda")
    kf.kf_decode_step_static(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                             dev.ctx_before, dev.max_ctx_after, w.scale, kf.KF_SPLITS_BALANCED, out, lse_out=lse)
    _check_bf16(dev, hv, out, lse, "static balanced")


def test_extra_partials(kf):
    """kf_decode_step_merge_partials on the balanced schedule: the prefix
    partials of a cascade step (plus an empty slot whose o is NaN) merged with
    each request's suffix runs; bf16 output."""
    from paged_kv_decode_kf_gb300.step import CascadeStep
    w = wl.scaled(wl.CONFIGS["cascade"], batch=7, lengths=wl.Fixed((40, 3, 200, 17, 64, 0, 1500)))
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    step = CascadeStep(dev, suffix_splits=1)
    step.prefix()
    Sp = step.Sp
    B, Hq, D = w.batch, w.num_q_heads, w.head_dim
    ex_o = torch.cat([step.out_partial[:Sp], torch.full((1, B, Hq, D), float("nan"), device="cuda")])
    ex_l = torch.cat([step.lse_partial[:Sp], torch.full((1, B, Hq), float("-inf"), device="cuda")])
    ws = _ws(kf, w)
    out, lse = kf.kf_decode_step_merge_partials(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache,
                                                dev.suffix_tables, dev.suffix_ctx_before, step.max_suffix, w.scale,
                                                kf.KF_SPLITS_BALANCED, ex_o, ex_l, ws, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    _check_bf16(dev, hv, out, lse, "balanced + extras")
    assert _counters_zero(ws, w)


def test_cascade_full_size_balanced(kf):
    """The cascade workload at full size with its suffix step on the balanced
    schedule; sampled requests against the oracle over their whole tables."""
    from paged_kv_decode_kf_gb300.step import CascadeStep
    w = wl.CONFIGS["cascade"]
    dev = wl.make_inputs(w, "cuda")
    reqs = [0, 1, 31, 62, 63]
    hv = HostView(dev, reqs)
    step = CascadeStep(dev, suffix_splits=0)
    step.run()
    torch.cuda.synchronize()
    _check_bf16(dev, hv, step.out, step.lse, "cascade balanced", reqs=reqs)


@pytest.mark.parametrize("name", ["llama8b", "longctx", "ragged"])
def test_full_size_sampled(kf, name):
    from paged_kv_decode_kf_gb300.step import DecodeStep
    from test_gpu_parity import _sample_requests
    w = wl.CONFIGS[name]
    dev = wl.make_inputs(w, "cuda")
    reqs = _sample_requests(dev)
    hv = HostView(dev, reqs)
    step = DecodeStep(dev, num_splits=0, fused=True)
    step.run()
    torch.cuda.synchronize()
    _check_bf16(dev, hv, step.out, step.lse, name + " balanced", reqs=reqs)


# ------------------------------- FP8 caches --------------------------------

def _fp8_host(dev):
    return dict(q=wl.bf16_bits(dev.q), k=dev.k_cache.cpu().numpy(), v=dev.v_cache.cpu().numpy(),
                kn=wl.bf16_bits(dev.k_new), vn=wl.bf16_bits(dev.v_new), ks=dev.k_scale.cpu().numpy(),
                vs=dev.v_scale.cpu().numpy(), bt=dev.block_tables.cpu().numpy(),
                c0=dev.ctx_before.cpu().numpy(), c1=dev.ctx_after.cpu().numpy())


@pytest.mark.parametrize("name", sorted(SMALL))
def test_step_fp8(kf, name):
    lens = SMALL[name]
    w = wl.scaled(wl.with_kv_dtype(wl.CONFIGS[name], "fp8"), batch=len(lens), lengths=wl.Fixed(lens),
                  spare_blocks=3)
    dev = wl.make_inputs(w, "cuda")
    h = _fp8_host(dev)
    ws = _ws(kf, w)
    out, lse = kf.kf_decode_step_fp8(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.k_scale,
                                     dev.v_scale, dev.block_tables, dev.ctx_before, dev.max_ctx_after, w.scale,
                                     kf.KF_SPLITS_BALANCED, ws)
    k2, v2, _ = oracle.append_fp8(h["k"], h["v"], h["kn"], h["vn"], h["ks"], h["vs"], h["bt"], h["c0"])
    assert np.array_equal(dev.k_cache.cpu().numpy(), k2) and np.array_equal(dev.v_cache.cpu().numpy(), v2)
    ref_o, ref_l = oracle.attention_fp8(h["q"], k2, v2, h["ks"], h["vs"], h["bt"], h["c1"], w.scale)
    check_out(out.cpu().numpy(), ref_o, name + " fp8 balanced")
    check_lse(lse.cpu().numpy(), ref_l, name + " fp8 balanced")
    assert _counters_zero(ws, w)


def test_fp8_full_size_sampled(kf):
    """llama8b shapes with an FP8 cache, in the configuration the benchmark times."""
    from paged_kv_decode_kf_gb300.step import DecodeStep
    from test_gpu_parity import _sample_requests
    w = wl.with_kv_dtype(wl.CONFIGS["llama8b"], "fp8")
    dev = wl.make_inputs(w, "cuda")
    reqs = _sample_requests(dev, k=4)
    bt = dev.block_tables.cpu().numpy()[reqs]
    used = sorted({int(x) for x in bt.ravel() if x >= 0})
    remap = np.full(dev.num_blocks, -1, np.int64)
    remap[used] = np.arange(len(used))
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    ksub, vsub = dev.k_cache.index_select(0, idx).cpu().numpy(), dev.v_cache.index_select(0, idx).cpu().numpy()
    bt_sub = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    r = torch.tensor(reqs, dtype=torch.long, device="cuda")
    q = wl.bf16_bits(dev.q.index_select(0, r))
    kn, vn = wl.bf16_bits(dev.k_new.index_select(0, r)), wl.bf16_bits(dev.v_new.index_select(0, r))
    c0, c1 = dev.ctx_before.cpu().numpy()[reqs], dev.ctx_after.cpu().numpy()[reqs]
    ks, vs = dev.k_scale.cpu().numpy(), dev.v_scale.cpu().numpy()
    step = DecodeStep(dev, num_splits=0, fused=True)
    step.run()
    torch.cuda.synchronize()
    k2, v2, _ = oracle.append_fp8(ksub, vsub, kn, vn, ks, vs, bt_sub, c0)
    ref_o, ref_l = oracle.attention_fp8(q, k2, v2, ks, vs, bt_sub, c1, w.scale)
    check_out(step.out.cpu().numpy()[reqs], ref_o, "llama8b fp8 balanced")
    check_lse(step.lse.cpu().numpy()[reqs], ref_l, "llama8b fp8 balanced")
