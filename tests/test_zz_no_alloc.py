"""The decode step for callers that cannot allocate device memory.

kf_decode_step needs a scratch workspace from its caller. Callers whose
device memory is reserved once by their own pool allocator, plugin hosts
that hand a library only each call's buffers, and decode loops that cannot
pay for cudaMalloc's implicit synchronisation use kf_decode_step_static
instead: it takes no workspace and allocates nothing, keeping its scratch in
a fixed array inside the library. This test calls it through the C ABI twice
in a row and checks each result against kf_decode_step with a workspace.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import check_lse, check_out
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


def test_static_scratch_step_matches_workspace_step(kf):
    lens = (1, 17, 250, 777, 3840)
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=len(lens), lengths=wl.Fixed(lens), spare_blocks=2)
    dev = wl.make_inputs(w, "cuda")
    S = 6
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    assert kf.kf_decode_step_workspace_size(B, Hq, Hkv, D, S) <= kf.KF_STATIC_SCRATCH_BYTES

    # the existing entry point, with a workspace the caller allocated
    ws = kf.make_workspace(B, Hq, Hkv, D, S)
    ref, ref_lse = kf.kf_decode_step(dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables,
                                     dev.ctx_before, dev.max_ctx_after, w.scale, S, ws)
    torch.cuda.synchronize()
    ref_np, ref_lse_np = ref.double().cpu().numpy(), ref_lse.double().cpu().numpy()

    lib = kf.raw()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.kf_decode_step_static(
            _ptr(dev.q), _ptr(dev.k_new), _ptr(dev.v_new), _ptr(dev.k_cache), _ptr(dev.v_cache),
            _ptr(dev.block_tables), dev.block_tables.shape[1], _ptr(dev.ctx_before), dev.max_ctx_after,
            B, Hq, Hkv, D, w.block_size, dev.num_blocks, ctypes.c_float(w.scale), S, _ptr(out),
            kf.KF_F32, _ptr(lse), stream)
        assert st == kf.KF_OK, st
        torch.cuda.synchronize()
        assert kf.kf_get_device_error() == 0
        check_out(out.cpu().numpy(), ref_np, "static scratch call %d" % call)
        check_lse(lse.cpu().numpy(), ref_lse_np, "static scratch call %d" % call)


def test_static_scratch_rejects_oversize(kf):
    # a step whose scratch would not fit in the fixed array is refused before any launch
    B, Hq, Hkv, D, S = 256, 32, 8, 128, 64
    assert kf.kf_decode_step_workspace_size(B, Hq, Hkv, D, S) > kf.KF_STATIC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = _ptr(t)
    st = kf.raw().kf_decode_step_static(p, p, p, p, p, p, 8, p, 4096, B, Hq, Hkv, D, 16, 64,
                                        ctypes.c_float(0.1), S, p, kf.KF_F32, None, None)
    assert st == kf.KF_ERR_UNSUPPORTED
