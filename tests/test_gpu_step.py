"""GPU parity of the single-launch decode step (kf_decode_step: append,
split attention and merge in one kernel) against the fp64 oracle."""
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


def _fused(kf, dev, S, out_dtype=torch.float32, ws=None):
    w = dev.workload
    if ws is None and S > 1:
        ws = kf.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, S)
    out, lse = kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                                 dev.ctx_before, dev.max_ctx_after, w.scale, S, ws, out_dtype=out_dtype)
    return out, lse, ws


def _plan(kf, dev):
    w = dev.workload
    return kf.kf_choose_num_splits(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                   dev.max_ctx_after, dev.ctx_after.cpu().numpy())


def _check_against_oracle(dev, hv, out, lse, reqs=None, what=""):
    k2, v2 = hv.appended()
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, dev.workload.scale)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    if reqs is not None:
        o, l = o[reqs], l[reqs]
    check_out(o, ref_o, what + " out")
    check_lse(l, ref_l, what + " lse")
    return k2, v2


@pytest.mark.parametrize("S", [1, 3, "plan"])
def test_tiny(kf, S):
    w = wl.CONFIGS["tiny"]
    host = wl.make_inputs(w, "cpu")
    dev = host.to("cuda")
    S = _plan(kf, dev) if S == "plan" else S
    out, lse, _ = _fused(kf, dev, S)
    k2, v2, _ = oracle.append(wl.bf16_bits(host.k_cache), wl.bf16_bits(host.v_cache), wl.bf16_bits(host.k_new),
                              wl.bf16_bits(host.v_new), host.block_tables.numpy(), host.ctx_before.numpy())
    assert np.array_equal(wl.bf16_bits(dev.k_cache), k2) and np.array_equal(wl.bf16_bits(dev.v_cache), v2)
    ref_o, ref_l = oracle.attention(wl.bf16_bits(host.q), k2, v2, host.block_tables.numpy(),
                                    host.ctx_after.numpy(), w.scale)
    check_out(out.cpu().numpy(), ref_o, "tiny")
    check_lse(lse.cpu().numpy(), ref_l, "tiny")


SMALL = {
    "llama8b": (1, 17, 250, 777, 3840, 15, 16),
    "longctx": (12345, 40, 8191),
    "ragged": (31, 32, 63, 1000, 4095, 0, 64),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("S", ["plan", 1, 5, 40])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_small(kf, name, S, dtype):
    lens = SMALL[name]
    w = wl.scaled(wl.CONFIGS[name], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=3)
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    S = _plan(kf, dev) if S == "plan" else S
    out, lse, _ = _fused(kf, dev, S, dtype)
    k2, v2 = _check_against_oracle(dev, hv, out, lse, what="%s S=%d" % (name, S))
    used = sorted({int(x) for x in dev.block_tables.cpu().numpy().ravel() if x >= 0})
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    assert np.array_equal(wl.bf16_bits(dev.k_cache.index_select(0, idx)), k2)
    assert np.array_equal(wl.bf16_bits(dev.v_cache.index_select(0, idx)), v2)


@pytest.mark.parametrize("name", ["llama8b", "longctx", "ragged"])
def test_full_size_sampled(kf, name):
    from paged_kv_decode_kf_gb300.step import DecodeStep
    from test_gpu_parity import _sample_requests
    w = wl.CONFIGS[name]
    dev = wl.make_inputs(w, "cuda")
    reqs = _sample_requests(dev)
    hv = HostView(dev, reqs)
    step = DecodeStep(dev, fused=True)      # the benchmark's launch configuration
    step.run()
    torch.cuda.synchronize()
    _check_against_oracle(dev, hv, step.out, step.lse, reqs=reqs, what=name)
    bt = dev.block_tables.cpu().numpy()
    pos = dev.ctx_before.cpu().numpy().astype(np.int64)
    phys = torch.tensor(bt[np.arange(w.batch), pos // w.block_size], dtype=torch.long, device="cuda")
    slot = torch.tensor(pos % w.block_size, dtype=torch.long, device="cuda")
    assert torch.equal(dev.k_cache[phys, slot], dev.k_new) and torch.equal(dev.v_cache[phys, slot], dev.v_new)


def test_repeated_steps_and_three_call_path(kf):
    """The workspace counters return to zero: consecutive steps agree bit for
    bit, and match the three-call path (append, attention, merge)."""
    w = wl.scaled(wl.CONFIGS["ragged"], batch=6, lengths=wl.Fixed((500, 31, 2000, 64, 1, 777)))
    dev = wl.make_inputs(w, "cuda")
    S = 6
    ws = kf.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, S)
    outs = [_fused(kf, dev, S, ws=ws)[0].clone() for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    n_ctr = w.batch * w.num_kv_heads
    assert torch.count_nonzero(ws[-((n_ctr * 4 + 255) // 256 * 256):]).item() == 0
    o_p, l_p = kf.kf_paged_decode_attention(dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.ctx_after,
                                            dev.max_ctx_after, w.scale, S)
    ref, _ = kf.kf_merge_partials(o_p, l_p)
    assert torch.allclose(outs[0], ref, rtol=0, atol=2e-6)


def test_device_errors(kf):
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=2, lengths=wl.Fixed((20, 40)))
    dev = wl.make_inputs(w, "cuda")
    bad = dev.block_tables.clone()
    bad[1, 40 // w.block_size] = -7
    kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, bad, dev.ctx_before,
                      dev.max_ctx_after, w.scale, 2, kf.make_workspace(2, w.num_q_heads, w.num_kv_heads,
                                                                       w.head_dim, 2))
    assert kf.kf_get_device_error() & kf.KF_DEVERR_BLOCK_ID
    full = dev.ctx_before.clone()
    full[0] = dev.block_tables.shape[1] * w.block_size
    kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, full,
                      int(full.max().item()) + 1, w.scale, 1, None)
    assert kf.kf_get_device_error() & kf.KF_DEVERR_APPEND_POS


def test_bounded_wait_gives_up_cleanly(kf):
    """A wait that nothing completes gives up after its bound, sets
    KF_DEVERR_TIMEOUT and returns; the context stays usable: a step run right
    after it matches the oracle."""
    kf.kf_check_bounded_wait()
    assert kf.kf_get_device_error() & kf.KF_DEVERR_TIMEOUT
    assert kf.kf_get_device_error() == 0            # read and cleared
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=3, lengths=wl.Fixed((40, 300, 17)))
    dev = wl.make_inputs(w, "cuda")
    hv = HostView(dev, range(w.batch))
    out, lse, _ = _fused(kf, dev, 2)
    _check_against_oracle(dev, hv, out, lse, what="after a timeout")


@pytest.mark.parametrize("kind", ["fused", "balanced", "cascade", "cascade_serial", "calls"])
def test_graph_captured_step_matches_eager(kind):
    """The step's calls need no host synchronisation and allocate nothing, so
    they capture into a CUDA graph (as the benchmark replays them): a replay
    gives the eager step's output and lse bit for bit."""
    from paged_kv_decode_kf_gb300.step import CascadeStep, DecodeStep
    if kind.startswith("cascade"):
        w = wl.scaled(wl.CONFIGS["cascade"], batch=6, lengths=wl.Fixed((5, 70, 300, 1, 16, 999)))
        dev = wl.make_inputs(w, "cuda")
        step = CascadeStep(dev, concurrent=kind == "cascade")   # the concurrent form forks a second stream
    else:
        w = wl.scaled(wl.CONFIGS["ragged"], batch=5, lengths=wl.Fixed((500, 31, 2000, 64, 777)))
        dev = wl.make_inputs(w, "cuda")
        step = DecodeStep(dev, num_splits=0 if kind == "balanced" else None, fused=kind != "calls")
    step.run()
    torch.cuda.synchronize()
    ref_o, ref_l = step.out.clone(), step.lse.clone()
    step.out.zero_()
    step.lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.out, ref_o) and torch.equal(step.lse, ref_l)


@pytest.mark.parametrize("kind", ["splits", "balanced", "static", "merge_partials", "fp8"])
def test_pinned_host_step_io(kind, kf):
    """The step calls read q, k_new, v_new, block tables and context lengths
    from pinned host memory and write out and lse there (zero-copy): the result
    equals the device-buffer call's bit for bit and matches the oracle."""
    lens = (500, 31, 2000, 64, 1, 777)
    w = wl.scaled(wl.CONFIGS["ragged"], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=3)
    if kind == "fp8":
        w = wl.with_kv_dtype(w, "fp8")
    dev = wl.make_inputs(w, "cuda")
    hv = None if kind == "fp8" else HostView(dev, range(w.batch))
    S = kf.KF_SPLITS_BALANCED if kind == "balanced" else 5
    pin = lambda t: t.cpu().pin_memory()
    h = {n: pin(getattr(dev, n)) for n in ("q", "k_new", "v_new", "block_tables", "ctx_before")}
    shape = (w.batch, w.num_q_heads, w.head_dim)
    ws = None if kind == "static" else kf.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, S)
    n_ex = 2
    ex_o = torch.randn((n_ex,) + shape, device="cuda") if kind == "merge_partials" else None
    ex_l = torch.randn((n_ex, w.batch, w.num_q_heads), device="cuda") if kind == "merge_partials" else None

    def call(src, out, lse):
        args = (src["q"], src["k_new"], src["v_new"], dev.k_cache, dev.v_cache)
        rest = (src["block_tables"], src["ctx_before"], dev.max_ctx_after, w.scale, S)
        if kind == "static":
            kf.kf_decode_step_static(*args, *rest, out, lse_out=lse)
        elif kind == "merge_partials":
            kf.kf_decode_step_merge_partials(*args, *rest, ex_o, ex_l, ws, out=out, lse_out=lse)
        elif kind == "fp8":
            kf.kf_decode_step_fp8(*args, dev.k_scale, dev.v_scale, *rest, ws, out=out, lse_out=lse)
        else:
            kf.kf_decode_step(*args, *rest, ws, out=out, lse_out=lse)

    d = {n: getattr(dev, n) for n in h}
    out_d = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    lse_d = torch.empty(shape[:2], dtype=torch.float32, device="cuda")
    call(d, out_d, lse_d)
    out_h = torch.full(shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.full(shape[:2], float("nan"), dtype=torch.float32).pin_memory()
    call(h, out_h, lse_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    if kind in ("merge_partials", "fp8"):
        return          # their numerics are checked against the oracle in their own tests
    _check_against_oracle(dev, hv, out_h, lse_h, what="pinned host I/O, %s" % kind)


def test_pageable_host_tensor_refused(kf):
    w = wl.scaled(wl.CONFIGS["tiny"], batch=2, lengths=wl.Fixed((20, 40)))
    dev = wl.make_inputs(w, "cuda")
    with pytest.raises(ValueError, match="pinned"):
        kf.kf_decode_step(dev.q.cpu(), dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                          dev.ctx_before, dev.max_ctx_after, w.scale, 1)
