"""Host logic of the benchmark's roofline fields, on CPU: the committed DRAM
traffic records are looked up by kernel and workload, scaled by the KV bytes
of the launch, and dropped once the kernel's sources no longer match the
digest they were captured from; the L2 note names why no flush runs."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_decode_kf_gb300 import workloads as wl  # noqa: E402


def test_traffic_records_scale_by_kv_bytes():
    rec = json.load(open(os.path.join(ROOT, "profiles", "multiquery_dram_traffic.json")))
    for kernel, rows, name in (("mq5", 16, "specverify"), ("mqw", 4096, "chunk")):
        r = rec["kernels"][kernel]
        if r["kernel_source_digest"] != bench.kernel_source_digest(kernel):
            assert bench.profiled_mq_traffic(name, rows, 1.0) is None   # stale: no traffic claimed
            continue
        per = r["per_workload"][name]
        assert per["dram_bytes_per_launch"] == per["dram_bytes_read"] + per["dram_bytes_write"]
        full = bench.profiled_mq_traffic(name, rows, per["kv_bytes_per_launch"])
        assert full == pytest.approx(per["dram_bytes_per_launch"])
        assert bench.profiled_mq_traffic(name, rows, per["kv_bytes_per_launch"] / 2) == pytest.approx(full / 2)
    # a kernel's record never answers for the other kernel's row counts
    assert bench.profiled_mq_traffic("specverify", 4096, 1.0) is None
    assert bench.profiled_mq_traffic("chunk", 16, 1.0) is None
    assert bench.profiled_mq_traffic("no-such-workload", 16, 1.0) is None


def test_decode_traffic_record():
    rec = json.load(open(os.path.join(ROOT, "profiles", "attention_dram_traffic.json")))
    fused = rec["per_workload_fused"]
    if rec["kernel_source_digest"] != bench.kernel_source_digest():
        assert bench.profiled_traffic("llama8b", "fused", 1.0) is None
        return
    for key, per in fused.items():
        name, _, dt = key.partition("_")
        got = bench.profiled_traffic(name, "fused", per["kv_bytes_per_launch"], dt or "bf16")
        assert got == pytest.approx(per["dram_bytes_per_launch"])
        # traffic at most a few percent above the algorithmic KV bytes: no re-reads
        assert per["dram_bytes_read"] < 1.02 * per["kv_bytes_per_launch"]
    assert bench.profiled_traffic("llama8b", "simt", 1.0) is None


def test_digests_depend_on_their_sources():
    assert bench.kernel_source_digest("decode") == bench.kernel_source_digest()
    assert len({bench.kernel_source_digest(k) for k in bench.DIGEST_SOURCES}) == len(bench.DIGEST_SOURCES)


@pytest.mark.parametrize("name,expect", [("llama8b", "GB of KV"), ("chunk", "inputs a step reads"),
                                         ("tiny", "launch-bound")])
def test_l2_note(name, expect):
    w = wl.CONFIGS[name]
    lay = wl.plan_layout(w)
    kv = float(lay.ctx_after.sum()) * 2 * w.num_kv_heads * w.head_dim * 2
    note = bench.l2_note(kv, wl.make_inputs(w, "cpu") if name != "llama8b" else _q_only(w))
    assert expect in note


class _q_only:
    """The query-side tensors of a workload without building its cache."""
    def __init__(self, w):
        import torch
        self.q = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.bfloat16)
        self.k_new = self.v_new = torch.empty((w.batch, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16)
        self.q_chunk = None
