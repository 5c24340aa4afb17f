"""The decode step for callers that cannot allocate device memory.

kf_decode_step needs a scratch workspace from its caller. Callers whose
device memory is reserved once by their own pool allocator, plugin hosts
that hand a library only each call's buffers, and decode loops that cannot
pay for cudaMalloc's implicit synchronisation use kf_decode_step_static
instead: it takes no workspace and allocates nothing, keeping its scratch in
a fixed array inside the library. These tests call it through the C ABI
twice in a row, for each of the three scratch layouts (the balanced
schedule, one split with no scratch, the split rule), and check each result
against kf_decode_step with a workspace and against the fp64 oracle.
"""
import ctypes

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
    return kf


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(kf, dev, S, out, lse):
    w = dev.workload
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kf.raw().kf_decode_step_static(
        _ptr(dev.q), _ptr(dev.k_new), _ptr(dev.v_new), _ptr(dev.k_cache), _ptr(dev.v_cache),
        _ptr(dev.block_tables), dev.block_tables.shape[1], _ptr(dev.ctx_before), dev.max_ctx_after,
        w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, dev.num_blocks,
        ctypes.c_float(w.scale), S, _ptr(out), kf.KF_F32, _ptr(lse), stream)


# 0 = the balanced schedule (counters at the start of the scratch, its size
# from the SM count); 1 = one split (no scratch at all); 6 = the split rule
# (counters after the partials)
@pytest.mark.parametrize("S", [0, 1, 6])
def test_static_scratch_step_matches_workspace_step_and_oracle(kf, S):
    lens = (1, 17, 250, 777, 3840)
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    assert kf.kf_decode_step_workspace_size(B, Hq, Hkv, D, S) <= kf.KF_STATIC_SCRATCH_BYTES
    # host copies for the oracle, taken before any call appends
    hv = HostView(dev, range(B))
    k2, v2 = hv.appended()
    ref_o, ref_l = oracle.attention(hv.q, k2, v2, hv.tables[0], hv.ctx_after, w.scale)

    # the existing entry point, with a workspace the caller allocated
    ws = kf.make_workspace(B, Hq, Hkv, D, S) if S != 1 else None
    ref, ref_lse = kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                                     dev.ctx_before, dev.max_ctx_after, w.scale, S, ws)
    torch.cuda.synchronize()
    assert kf.kf_get_device_error() == 0
    ref_np, ref_lse_np = ref.double().cpu().numpy(), ref_lse.double().cpu().numpy()
    check_out(ref_np, ref_o, "workspace step S=%d" % S)
    check_lse(ref_lse_np, ref_l, "workspace step S=%d" % S)

    for call in range(2):   # the second call finds the first one's leftovers in the array
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        st = _static_call(kf, dev, S, out, lse)
        assert st == kf.KF_OK, st
        torch.cuda.synchronize()
        assert kf.kf_get_device_error() == 0
        what = "static scratch S=%d call %d" % (S, call)
        o, l = out.double().cpu().numpy(), lse.double().cpu().numpy()
        check_out(o, ref_np, what + " vs workspace step")
        check_lse(l, ref_lse_np, what + " vs workspace step")
        check_out(o, ref_o, what + " vs oracle")
        check_lse(l, ref_l, what + " vs oracle")
    # the cache holds exactly the oracle's append (the calls re-wrote the same row)
    after = HostView(dev, range(B))
    assert np.array_equal(after.k, k2) and np.array_equal(after.v, v2)


def test_static_scratch_rejects_oversize(kf):
    # a step whose scratch would not fit in the fixed array is refused before any launch
    B, Hq, Hkv, D, S = 256, 32, 8, 128, 64
    assert kf.kf_decode_step_workspace_size(B, Hq, Hkv, D, S) > kf.KF_STATIC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = _ptr(t)
    st = kf.raw().kf_decode_step_static(p, p, p, p, p, p, 8, p, 4096, B, Hq, Hkv, D, 16, 64,
                                        ctypes.c_float(0.1), S, p, kf.KF_F32, None, None)
    assert st == kf.KF_ERR_UNSUPPORTED


@pytest.mark.parametrize("S", [0, 6])
def test_static_scratch_status_matches_workspace_step(kf, S):
    # an unsupported head_dim gets the same status from both entry points, and
    # neither launches anything
    B, Hq, Hkv, D = 2, 8, 2, 96
    t = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = _ptr(t)
    lib = kf.raw()
    st_static = lib.kf_decode_step_static(p, p, p, p, p, p, 8, p, 128, B, Hq, Hkv, D, 16, 64,
                                          ctypes.c_float(0.1), S, p, kf.KF_F32, None, None)
    st_ws = lib.kf_decode_step(p, p, p, p, p, p, 8, p, 128, B, Hq, Hkv, D, 16, 64, ctypes.c_float(0.1), S,
                               p, t.numel(), p, kf.KF_F32, None, None)
    assert st_static == st_ws == kf.KF_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(t.count_nonzero()) == 0
