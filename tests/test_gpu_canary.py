"""Writes stay inside their buffers: outputs, lse, partials and the workspace
are views into larger buffers whose guard bands hold a canary bit pattern
that must survive every call, and every byte of the caches (the spare blocks
included) equals the oracle's append result: only the step's new rows
change."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_lse, check_out
from paged_kv_decode_kf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CANARY = 0x7FA5A5A5  # a NaN bit pattern no kernel writes
GUARD = 64           # guard elements on each side (256 bytes: keeps 16-byte alignment)


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


def guarded(shape, dtype=torch.float32):
    """(inner view, whole buffer): the view sits between two canary bands."""
    n = int(np.prod(shape))
    words = (n * torch.tensor([], dtype=dtype).element_size() + 3) // 4
    buf = torch.full((words + 2 * GUARD,), CANARY, dtype=torch.int32, device="cuda")
    inner = buf[GUARD:GUARD + words].view(torch.uint8)[:n * torch.tensor([], dtype=dtype).element_size()]
    return inner.view(dtype).view(shape), buf, words


def bands_intact(buf, words):
    return bool((buf[:GUARD] == CANARY).all()) and bool((buf[GUARD + words:] == CANARY).all())


def _inputs(kv="bf16"):
    base = wl.CONFIGS["ragged"] if kv == "bf16" else wl.with_kv_dtype(wl.CONFIGS["ragged"], "fp8")
    w = wl.scaled(base, batch=6, lengths=wl.Fixed((500, 31, 2000, 64, 0, 777)), spare_blocks=6)
    return w, wl.make_inputs(w, "cuda")


def _cache_expected(dev, kv):
    if kv == "bf16":
        k2, v2, _ = oracle.append(wl.bf16_bits(dev.k_cache), wl.bf16_bits(dev.v_cache), wl.bf16_bits(dev.k_new),
                                  wl.bf16_bits(dev.v_new), dev.block_tables.cpu().numpy(),
                                  dev.ctx_before.cpu().numpy())
    else:
        k2, v2, _ = oracle.append_fp8(dev.k_cache.cpu().numpy(), dev.v_cache.cpu().numpy(), wl.bf16_bits(dev.k_new),
                                      wl.bf16_bits(dev.v_new), dev.k_scale.cpu().numpy(), dev.v_scale.cpu().numpy(),
                                      dev.block_tables.cpu().numpy(), dev.ctx_before.cpu().numpy())
    return k2, v2


def _cache_now(dev, kv):
    if kv == "bf16":
        return wl.bf16_bits(dev.k_cache), wl.bf16_bits(dev.v_cache)
    return dev.k_cache.cpu().numpy(), dev.v_cache.cpu().numpy()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("S", [1, 4, 0])   # 0: the balanced schedule
def test_step_writes_stay_in_bounds(kf, kv, S):
    w, dev = _inputs(kv)
    B, Hq, D = w.batch, w.num_q_heads, w.head_dim
    k2, v2 = _cache_expected(dev, kv)
    out, out_buf, out_words = guarded((B, Hq, D))
    lse, lse_buf, lse_words = guarded((B, Hq))
    ws = None
    if S != 1:
        n = kf.kf_decode_step_workspace_size(B, Hq, w.num_kv_heads, D, S)
        ws_full = torch.full((n + 2 * 4 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
        ws_full[4 * GUARD:4 * GUARD + n] = 0   # the workspace proper starts zeroed
        ws = ws_full[4 * GUARD:4 * GUARD + n]
    args = (dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache)
    if kv == "bf16":
        kf.kf_decode_step(*args, dev.block_tables, dev.ctx_before, dev.max_ctx_after, w.scale, S, ws, out=out,
                          lse_out=lse)
    else:
        kf.kf_decode_step_fp8(*args, dev.k_scale, dev.v_scale, dev.block_tables, dev.ctx_before,
                              dev.max_ctx_after, w.scale, S, ws, out=out, lse_out=lse)
    torch.cuda.synchronize()
    assert bands_intact(out_buf, out_words) and bands_intact(lse_buf, lse_words)
    if ws is not None:
        assert bool((ws_full[:4 * GUARD] == 0xA5).all()) and bool((ws_full[4 * GUARD + n:] == 0xA5).all())
    kn, vn = _cache_now(dev, kv)
    assert np.array_equal(kn, k2) and np.array_equal(vn, v2)   # every block, the spare ones included
    if kv == "bf16":   # the full caches with the full tables
        ref_o, ref_l = oracle.attention(wl.bf16_bits(dev.q), k2, v2, dev.block_tables.cpu().numpy(),
                                        dev.ctx_after.cpu().numpy(), w.scale)
    else:
        ref_o, ref_l = oracle.attention_fp8(wl.bf16_bits(dev.q), k2, v2, dev.k_scale.cpu().numpy(),
                                            dev.v_scale.cpu().numpy(), dev.block_tables.cpu().numpy(),
                                            dev.ctx_after.cpu().numpy(), w.scale)
    check_out(out.cpu().numpy(), ref_o, "canary step out")
    check_lse(lse.cpu().numpy(), ref_l, "canary step lse")


def test_three_calls_write_stay_in_bounds(kf):
    """kf_append_kv, kf_paged_decode_attention into guarded partial slots, and
    kf_merge_partials into a guarded output."""
    w, dev = _inputs("bf16")
    B, Hq, D, S = w.batch, w.num_q_heads, w.head_dim, 5
    k2, v2 = _cache_expected(dev, "bf16")
    kf.kf_append_kv(dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, dev.ctx_before)
    op, op_buf, op_words = guarded((S, B, Hq, D))
    lp, lp_buf, lp_words = guarded((S, B, Hq))
    kf.kf_paged_decode_attention(dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.ctx_after,
                                 dev.max_ctx_after, w.scale, S, out_partial=op, lse_partial=lp)
    out, out_buf, out_words = guarded((B, Hq, D), torch.bfloat16)
    kf.kf_merge_partials(op, lp, out)
    torch.cuda.synchronize()
    assert bands_intact(op_buf, op_words) and bands_intact(lp_buf, lp_words) and bands_intact(out_buf, out_words)
    kn, vn = _cache_now(dev, "bf16")
    assert np.array_equal(kn, k2) and np.array_equal(vn, v2)
