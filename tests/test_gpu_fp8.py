"""GPU parity of the FP8 (E4M3) KV-cache path against the fp64 oracle:
append bit-exact (same quantisation decision, fp32 division then E4M3
nearest-even), attention and the single-launch step within the bf16 path's
tolerances on the dequantised values."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_lse, check_out, check_partials
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


def _fp8(name, lengths, **kw):
    w = wl.scaled(wl.with_kv_dtype(wl.CONFIGS[name], "fp8"), batch=len(lengths), lengths=wl.Fixed(lengths),
                  spare_blocks=3, **kw)
    return w, wl.make_inputs(w, "cuda")


def _host(dev):
    return dict(q=wl.bf16_bits(dev.q), k=dev.k_cache.cpu().numpy(), v=dev.v_cache.cpu().numpy(),
                kn=wl.bf16_bits(dev.k_new), vn=wl.bf16_bits(dev.v_new), ks=dev.k_scale.cpu().numpy(),
                vs=dev.v_scale.cpu().numpy(), bt=dev.block_tables.cpu().numpy(),
                c0=dev.ctx_before.cpu().numpy(), c1=dev.ctx_after.cpu().numpy())


def test_append_fp8_bit_exact(kf):
    w, dev = _fp8("ragged", (31, 32, 63, 1000, 0, 64))
    h = _host(dev)
    # include values that saturate (|x / scale| > 448) and exact ties
    dev.k_new[0, 0, :4] = torch.tensor([100.0, -100.0, 1.0625 / 16, 3 * 2.0 ** -14], dtype=torch.bfloat16)
    h["kn"] = wl.bf16_bits(dev.k_new)
    kf.kf_append_kv_fp8(dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale,
                        dev.block_tables, dev.ctx_before)
    k2, v2, skipped = oracle.append_fp8(h["k"], h["v"], h["kn"], h["vn"], h["ks"], h["vs"], h["bt"], h["c0"])
    assert skipped == 0
    assert np.array_equal(dev.k_cache.cpu().numpy(), k2) and np.array_equal(dev.v_cache.cpu().numpy(), v2)


SMALL = {
    "llama8b": (1, 17, 250, 777, 3840),
    "longctx": (12345, 40, 8191),
    "ragged": (31, 32, 63, 1000, 4095, 0, 64),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("S", [1, 3, 16])
def test_attention_fp8(kf, name, S):
    w, dev = _fp8(name, SMALL[name])
    h = _host(dev)
    o_p, l_p = kf.kf_paged_decode_attention_fp8(dev.q, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale,
                                                dev.block_tables, dev.ctx_after, dev.max_ctx_after, w.scale, S)
    out, lse = kf.kf_merge_partials(o_p, l_p)
    ref_po, ref_pl = oracle.decode_partials_fp8(h["q"], h["k"], h["v"], h["ks"], h["vs"], h["bt"], h["c1"],
                                                w.scale, S, max_context_len=dev.max_ctx_after)
    check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, name + " fp8 partials")
    ref_o, ref_l = oracle.merge_partials(ref_po, ref_pl)
    check_out(out.cpu().numpy(), ref_o, name + " fp8 out")
    check_lse(lse.cpu().numpy(), ref_l, name + " fp8 lse")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (8, 1), (32, 8), (64, 8)])
@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32), (64, 32), (128, 16)])
def test_fp8_shape_sweep(kf, hq, hkv, d, bs):
    w = wl.Workload(name="fp8sweep", batch=3, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                    lengths=wl.Fixed((5, 2 * bs + 3, 9 * bs)), seed=91 + hq + hkv + d + bs, spare_blocks=2,
                    kv_dtype="fp8")
    dev = wl.make_inputs(w, "cuda")
    h = _host(dev)
    for S in (1, 4):
        o_p, l_p = kf.kf_paged_decode_attention_fp8(dev.q, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale,
                                                    dev.block_tables, dev.ctx_after, dev.max_ctx_after, w.scale, S)
        ref_po, ref_pl = oracle.decode_partials_fp8(h["q"], h["k"], h["v"], h["ks"], h["vs"], h["bt"], h["c1"],
                                                    w.scale, S, max_context_len=dev.max_ctx_after)
        check_partials(o_p.cpu().numpy(), l_p.cpu().numpy(), ref_po, ref_pl, "fp8 sweep")


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("S", [1, 5])
def test_step_fp8(kf, name, S):
    w, dev = _fp8(name, SMALL[name])
    h = _host(dev)
    ws = kf.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, S) if S > 1 else None
    out, lse = kf.kf_decode_step_fp8(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.k_scale,
                                     dev.v_scale, dev.block_tables, dev.ctx_before, dev.max_ctx_after, w.scale,
                                     S, ws)
    k2, v2, _ = oracle.append_fp8(h["k"], h["v"], h["kn"], h["vn"], h["ks"], h["vs"], h["bt"], h["c0"])
    assert np.array_equal(dev.k_cache.cpu().numpy(), k2) and np.array_equal(dev.v_cache.cpu().numpy(), v2)
    ref_o, ref_l = oracle.attention_fp8(h["q"], k2, v2, h["ks"], h["vs"], h["bt"], h["c1"], w.scale)
    check_out(out.cpu().numpy(), ref_o, name + " fp8 step")
    check_lse(lse.cpu().numpy(), ref_l, name + " fp8 step")


def test_fp8_nan_codes_past_context(kf):
    """E4M3 NaN codes in slots past the context do not reach the output."""
    w, dev = _fp8("llama8b", (17, 33, 100))
    L = dev.ctx_after.cpu().numpy()
    bt = dev.block_tables.cpu().numpy()
    for b in range(w.batch):
        n = -(-int(L[b]) // w.block_size)
        for t in range(int(L[b]) % w.block_size or w.block_size, w.block_size):
            dev.k_cache[bt[b, n - 1], t] = 0x7F
            dev.v_cache[bt[b, n - 1], t] = 0xFF
    h = _host(dev)
    o_p, l_p = kf.kf_paged_decode_attention_fp8(dev.q, dev.k_cache, dev.v_cache, dev.k_scale, dev.v_scale,
                                                dev.block_tables, dev.ctx_after, dev.max_ctx_after, w.scale, 2)
    out, lse = kf.kf_merge_partials(o_p, l_p)
    ref_o, ref_l = oracle.attention_fp8(h["q"], h["k"], h["v"], h["ks"], h["vs"], h["bt"], h["c1"], w.scale)
    check_out(out.cpu().numpy(), ref_o, "fp8 nan past context")


@pytest.mark.parametrize("name", ["llama8b", "longctx"])
def test_fp8_full_size_sampled(kf, name):
    from paged_kv_decode_kf_gb300.step import DecodeStep
    from test_gpu_parity import _sample_requests
    w = wl.with_kv_dtype(wl.CONFIGS[name], "fp8")
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
    step = DecodeStep(dev, fused=True)
    step.run()
    torch.cuda.synchronize()
    k2, v2, _ = oracle.append_fp8(ksub, vsub, kn, vn, ks, vs, bt_sub, c0)
    ref_o, ref_l = oracle.attention_fp8(q, k2, v2, ks, vs, bt_sub, c1, w.scale)
    check_out(step.out.cpu().numpy()[reqs], ref_o, name + " fp8 full")
    check_lse(step.lse.cpu().numpy()[reqs], ref_l, name + " fp8 full")
