"""The C-ABI library: loads, exports every declared symbol, host-side checks
and the split planner. No GPU needed: every call here returns before any
CUDA work (argument errors, empty batches, the host-only planner)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kf():
    import __graft_entry__ as g
    g.build()
    from paged_kv_decode_kf_gb300 import kf
    return kf


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kf_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(kf):
    names = declared_functions()
    assert "kf_paged_decode_attention" in names and len(names) >= 8
    lib = kf.raw()
    for n in names:
        assert hasattr(lib, n), n
    # and the shared object's dynamic symbol table has them as exported text
    so = open(kf.LIB_PATH, "rb").read()
    for n in names:
        assert n.encode() in so


def test_status_strings_and_version(kf):
    lib = kf.raw()
    for code in range(5):
        assert lib.kf_status_string(code)
    assert lib.kf_status_string(99) == b"unknown status"
    assert kf.kf_version() >= 100


def _attn(lib, **kw):
    a = dict(q=16, k=16, v=16, bt=16, bt_stride=4, ctx=16, max_ctx=64, batch=2, hq=8, hkv=2, d=128,
             bs=16, nb=8, scale=0.1, S=1, o=16, lse=16, stream=None)
    a.update(kw)
    return lib.kf_paged_decode_attention(a["q"], a["k"], a["v"], a["bt"], a["bt_stride"], a["ctx"],
                                         a["max_ctx"], a["batch"], a["hq"], a["hkv"], a["d"], a["bs"],
                                         a["nb"], a["scale"], a["S"], a["o"], a["lse"], a["stream"])


def test_attention_host_checks(kf):
    lib = kf.raw()
    assert _attn(lib, batch=0) == kf.KF_OK                 # empty batch: nothing to do
    for bad in (dict(q=None), dict(k=None), dict(o=None), dict(lse=None), dict(ctx=None),
                dict(bt=None), dict(batch=-1), dict(S=0), dict(bt_stride=0), dict(nb=0),
                dict(max_ctx=-1), dict(scale=float("nan")), dict(scale=float("inf")),
                dict(q=8), dict(k=24), dict(o=4), dict(hq=0), dict(hkv=0)):
        assert _attn(lib, **bad) == kf.KF_ERR_INVALID, bad
    for bad in (dict(d=96), dict(d=256), dict(bs=8), dict(bs=64), dict(hq=6, hkv=2),
                dict(hq=32, hkv=2), dict(hq=7, hkv=2)):
        assert _attn(lib, **bad) == kf.KF_ERR_UNSUPPORTED, bad


def test_append_and_merge_host_checks(kf):
    lib = kf.raw()
    ok = dict(kn=16, vn=16, kc=16, vc=16, bt=16, st=4, ctx=16, B=2, hkv=2, d=128, bs=16, nb=8)

    def app(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.kf_append_kv(a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["st"], a["ctx"], a["B"],
                                a["hkv"], a["d"], a["bs"], a["nb"], None)
    assert app(B=0) == kf.KF_OK
    for bad in (dict(kn=None), dict(vc=None), dict(ctx=None), dict(B=-3), dict(st=0), dict(nb=0), dict(kc=40)):
        assert app(**bad) == kf.KF_ERR_INVALID, bad
    assert app(d=80) == kf.KF_ERR_UNSUPPORTED and app(bs=48) == kf.KF_ERR_UNSUPPORTED

    def mrg(**kw):
        a = dict(o=16, lse=16, S=2, B=2, hq=4, d=128, out=16, dt=kf.KF_F32, lo=None)
        a.update(kw)
        return lib.kf_merge_partials(a["o"], a["lse"], a["S"], a["B"], a["hq"], a["d"], a["out"], a["dt"],
                                     a["lo"], None)
    assert mrg(B=0) == kf.KF_OK
    for bad in (dict(o=None), dict(lse=None), dict(out=None), dict(S=0), dict(B=-1), dict(hq=0),
                dict(dt=7), dict(out=20)):
        assert mrg(**bad) == kf.KF_ERR_INVALID, bad
    assert mrg(d=32) == kf.KF_ERR_UNSUPPORTED


def test_get_device_error_needs_flags(kf):
    lib = kf.raw()
    assert lib.kf_get_device_error(None, None) == kf.KF_ERR_INVALID


def test_split_planner(kf):
    plan = lambda B, L, lens=None, sms=152: kf.kf_choose_num_splits(B, 32, 8, 128, 16, L, lens, num_sms=sms)
    assert plan(2, 16) == 1                                  # one block: nothing to split
    # long single request on a big GPU is split many ways; a full batch of short ones is not
    assert plan(1, 262144) >= 16
    assert plan(64, 4096) <= plan(1, 4096)
    assert plan(16, 262144) >= plan(256, 262144)
    # host lengths: a batch where one request is long but the rest are short
    lens = np.full(256, 1024, np.int32)
    lens[0] = 131072
    s = plan(256, 131072, lens)
    assert 1 <= s <= 1024
    # deterministic and within range for every workload
    from paged_kv_decode_kf_gb300 import workloads as wl
    for name in wl.CONFIG_ORDER:
        w = wl.CONFIGS[name]
        lay = wl.plan_layout(w)
        L = lay.ctx_after.astype(np.int32)
        a = kf.kf_choose_num_splits(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                    int(L.max()), L, num_sms=152)
        b = kf.kf_choose_num_splits(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                    int(L.max()), L, num_sms=152)
        assert a == b and 1 <= a <= 1024
    assert kf.raw().kf_choose_num_splits_for(0, 32, 8, 128, 16, 100, None, 152) < 1
    assert kf.raw().kf_choose_num_splits_for(2, 32, 8, 96, 16, 100, None, 152) < 1


def test_binding_rejects_host_tensors(kf):
    import torch
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kf.kf_paged_decode_attention(q, q, q, torch.zeros(2, 4, dtype=torch.int32),
                                     torch.ones(2, dtype=torch.int32), 4, 0.1, 1,
                                     out_partial=torch.zeros(1), lse_partial=torch.zeros(1))


def test_step_binding_refuses_pageable_host_tensors(kf):
    """The step calls take pinned host tensors for their per-step inputs and
    outputs (read in place by the kernel); pageable host memory is refused
    before any call."""
    import torch
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    cache = torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16)
    for call in (kf.kf_decode_step, kf.kf_decode_step_static):
        with pytest.raises(ValueError, match="pinned"):
            call(q, q[:, :2], q[:, :2], cache, cache, torch.zeros(2, 2, dtype=torch.int32),
                 torch.ones(2, dtype=torch.int32), 4, 0.1, 1, out=torch.zeros(2, 8, 128))


def test_decode_step_host_checks(kf):
    lib = kf.raw()
    need = kf.kf_decode_step_workspace_size(4, 32, 8, 128, 10)
    al = lambda x: (x + 255) // 256 * 256
    assert need == al(10 * 4 * 32 * 128 * 4) + al(10 * 4 * 32 * 4) + al(4 * 8 * 4)
    assert kf.kf_decode_step_workspace_size(0, 32, 8, 128, 1) == al(0) + al(0) + al(0)
    assert kf.kf_decode_step_workspace_size(4, 32, 8, 128, -1) == 0
    if not torch.cuda.is_available():   # the balanced layout is sized for the current device
        assert kf.kf_decode_step_workspace_size(4, 32, 8, 128, kf.KF_SPLITS_BALANCED) == 0

    def step(**kw):
        a = dict(q=16, kn=16, vn=16, kc=16, vc=16, bt=16, st=8, ctx=16, mc=100, B=4, hq=32, hkv=8, d=128, bs=16,
                 nb=64, scale=0.1, S=10, ws=16, wsb=need, out=16, dt=kf.KF_F32, lse=None)
        a.update(kw)
        return lib.kf_decode_step(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["st"], a["ctx"], a["mc"],
                                  a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["scale"], a["S"], a["ws"],
                                  a["wsb"], a["out"], a["dt"], a["lse"], None)
    assert step(B=0) == kf.KF_OK
    for bad in (dict(ws=None), dict(wsb=need - 1), dict(ws=8), dict(kn=None), dict(out=None), dict(dt=3),
                dict(S=-1), dict(mc=-1), dict(scale=float("nan")), dict(S=0, ws=None), dict(S=0, ws=8)):
        assert step(**bad) == kf.KF_ERR_INVALID, bad
    assert step(S=100000) == kf.KF_ERR_UNSUPPORTED
    big = kf.kf_decode_step_workspace_size(4, 32, 8, 128, 2000)
    assert step(S=2000, wsb=big) == kf.KF_ERR_UNSUPPORTED     # the merge would not fit in shared memory
    assert step(d=96) == kf.KF_ERR_UNSUPPORTED


def test_decode_step_merge_partials_host_checks(kf):
    """The extra-partials step: the host checks of kf_decode_step, plus the
    extra slots (count, pointers, alignment), the workspace it needs even at
    one split, and the shared-memory bound on splits + extras."""
    lib = kf.raw()
    need1 = kf.kf_decode_step_workspace_size(4, 32, 8, 128, 1)

    def step(**kw):
        a = dict(q=16, kn=16, vn=16, kc=16, vc=16, bt=16, st=8, ctx=16, mc=100, B=4, hq=32, hkv=8, d=128, bs=16,
                 nb=64, scale=0.1, S=1, eo=16, el=16, ne=3, ws=16, wsb=need1, out=16, dt=kf.KF_F32, lse=None)
        a.update(kw)
        return lib.kf_decode_step_merge_partials(
            a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["st"], a["ctx"], a["mc"], a["B"], a["hq"],
            a["hkv"], a["d"], a["bs"], a["nb"], a["scale"], a["S"], a["eo"], a["el"], a["ne"], a["ws"], a["wsb"],
            a["out"], a["dt"], a["lse"], None)
    assert step(B=0) == kf.KF_OK
    for bad in (dict(ne=-1), dict(eo=None), dict(el=None), dict(eo=8), dict(ws=None), dict(wsb=need1 - 1),
                dict(kn=None), dict(S=-1), dict(S=0, ws=None)):
        assert step(**bad) == kf.KF_ERR_INVALID, bad
    big = kf.kf_decode_step_workspace_size(4, 32, 8, 128, 1000)
    assert step(S=1000, ne=1000, wsb=big) == kf.KF_ERR_UNSUPPORTED   # merge of 2000 partials does not fit
    assert step(d=96) == kf.KF_ERR_UNSUPPORTED
