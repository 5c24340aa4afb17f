"""Helpers for the GPU parity tests: host copies for the oracle and the
tolerance checks. Inputs reach the oracle straight from the seeded
generator (copied from the device before any kernel of the library runs);
nothing the CUDA path computes is ever fed to the oracle."""
from __future__ import annotations

import os
from contextlib import contextmanager

import numpy as np
import torch

import oracle
from paged_kv_decode_kf_gb300 import workloads as wl

# Tolerances of the decode path against the fp64 oracle: bf16 K/V/q, fp32
# accumulation.
MAX_ABS = 8e-3
MEAN_ABS = 1e-3
LSE_REL = 1e-4


@contextmanager
def _env(var: str, value: str):
    old = os.environ.get(var)
    os.environ[var] = value
    try:
        yield
    finally:
        if old is None:
            os.environ.pop(var, None)
        else:
            os.environ[var] = old


def decode_impl(name: str):
    """Select the decode kernel ("tc" or "simt") for the calls in the block."""
    return _env("KF_DECODE_IMPL", name)


@contextmanager
def mq_impl(name: str):
    """Select the multi-query kernel for the calls in the block: "mma", "tc05"
    (one 128-row query tile per CTA), "tc05x2" (two tiles per CTA, 64-token KV
    tiles), "tc05w" (two tiles, 128-token KV tiles; more than 128 rows),
    "tc05p" (CTA pairs, head_dim 128; any row count) or "auto"."""
    with _env("KF_MQ_IMPL", "tc05" if name == "tc05x2" else name), \
            _env("KF_MQ_TILES", "2" if name == "tc05x2" else "1"):
        yield


class HostView:
    """Host copies of the requests `reqs` of a workload, with their blocks
    compacted into a small pool (the oracle is invariant to physical
    placement). Taken BEFORE the step's append."""

    def __init__(self, inp: wl.DecodeInputs, reqs, tables=None):
        self.reqs = list(reqs)
        tabs = [inp.block_tables] if tables is None else list(tables)
        bt_all = [t.cpu().numpy() for t in tabs]
        used = sorted({int(x) for bt in bt_all for b in self.reqs for x in bt[b] if x >= 0})
        remap = {p: i for i, p in enumerate(used)}
        idx = torch.tensor(used, dtype=torch.long, device=inp.k_cache.device)
        self.k = wl.bf16_bits(inp.k_cache.index_select(0, idx))
        self.v = wl.bf16_bits(inp.v_cache.index_select(0, idx))
        self.tables = []
        for bt in bt_all:
            sub = bt[self.reqs]
            self.tables.append(np.vectorize(lambda x: remap[int(x)] if x >= 0 else -1, otypes=[np.int32])(sub)
                               if sub.size else sub.astype(np.int32))
        r = torch.tensor(self.reqs, dtype=torch.long, device=inp.q.device)
        self.q = wl.bf16_bits(inp.q.index_select(0, r))
        self.k_new = wl.bf16_bits(inp.k_new.index_select(0, r))
        self.v_new = wl.bf16_bits(inp.v_new.index_select(0, r))
        self.ctx_before = inp.ctx_before.cpu().numpy()[self.reqs]
        self.ctx_after = inp.ctx_after.cpu().numpy()[self.reqs]

    def appended(self, table=0, ctx_before=None):
        """Caches after the oracle's own append through table `table`."""
        cb = self.ctx_before if ctx_before is None else ctx_before
        k2, v2, skipped = oracle.append(self.k, self.v, self.k_new, self.v_new, self.tables[table], cb)
        assert skipped == 0
        return k2, v2


def check_out(gpu_out, ref_out, what=""):
    g = np.asarray(gpu_out, dtype=np.float64)
    err = np.abs(g - ref_out)
    assert np.all(np.isfinite(g)), what + ": non-finite output"
    assert err.max() <= MAX_ABS, "%s: max|err| %.3e" % (what, err.max())
    assert err.mean() <= MEAN_ABS, "%s: mean|err| %.3e" % (what, err.mean())
    return err.max(), err.mean()


def check_lse(gpu_lse, ref_lse, what=""):
    g = np.asarray(gpu_lse, dtype=np.float64)
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(g), empty), what + ": empty/non-empty mismatch"
    d = np.abs(g[~empty] - ref_lse[~empty])
    tol = LSE_REL * np.maximum(1.0, np.abs(ref_lse[~empty]))
    assert np.all(d <= tol), "%s: |dlse| %.3e" % (what, (d - tol).max())


def check_partials(o_p, l_p, ref_o, ref_l, what=""):
    """Every partial: empty ones exactly (0, -inf), the rest within tolerance."""
    o_p = np.asarray(o_p, dtype=np.float64)
    l_p = np.asarray(l_p, dtype=np.float64)
    check_lse(l_p, ref_l, what + " partial lse")
    empty = np.isneginf(ref_l)
    assert np.all(o_p[empty] == 0.0), what + ": empty partial o not zero"
    if (~empty).any():
        check_out(o_p[~empty], ref_o[~empty], what + " partial o")
