#!/usr/bin/env python3
"""Benchmark of one paged-KV decode step on GB300: append, split-KV
attention, LSE merge, through the C-ABI library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload ragged|llama8b|longctx|shard4|tiny|cascade|chunk|specverify]
                    [--kv-dtype bf16|fp8] [--num-splits S] [--out-dtype bf16|f32]

Prints one JSON line. The default workload is the largest one-GPU
configuration: the ragged continuous batch (256 requests, 70/25/5 % of them
1K-8K / 8K-64K / 64K-128K tokens, block size 32) with its append. `value` is
KV-read GB/s over all ranks: algorithmic KV bytes (sum_b L_b * 2 * Hkv * D *
2) per step divided by the device time of a step, inputs resident in HBM,
timed with CUDA events between a barrier and a synchronize on both sides, max
over ranks. `e2e` is the same metric through the C ABI with host buffers,
host waiting for each step's result: for the single-launch step, the step
kernel reads its per-step inputs from pinned host memory and writes out and
lse there (zero-copy), and `e2e_copies` is the copy-based run; for the other
paths, one H2D copy of the inputs and one D2H copy of the result per step.
Each carries the split of its time into device step and host launch/wait.
`per_config` (one GPU, default workload) times every decode configuration
(tiny, llama8b, longctx, shard4, ragged): per-step median / p10 / p90 over
at least 50 graph-replayed steps, KV GB/s and its fraction of the measured
HBM peak, next to the fp64 oracle timed on the host cores on a bounded
sample of the same configuration. `--impl reference` times the fp64 CPU
oracle on this machine's host cores on a bounded sample of the same workload.

With N > 1 (torchrun), every rank runs its own copy of the workload on its own
GPU (independent batches, no data-path collective: weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn KV-read GB/s (% of GB300 HBM peak); µs per batch step"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ragged")
    ap.add_argument("--decode-kernel", default="tc", choices=["tc", "simt"])
    ap.add_argument("--path", default="auto",
                    choices=["auto", "fused", "calls", "cascade", "cascade-serial", "cascade-calls"],
                    help="fused: kf_decode_step (one launch); calls: append, attention, merge; "
                         "cascade (shared-prefix workloads): prefix pass and kf_decode_step on two streams at "
                         "once, then one merge; cascade-serial: prefix pass, prefix merge, "
                         "kf_decode_step_merge_partials; cascade-calls: append, prefix pass, suffix decode, merge; "
                         "auto: fused for unsharded workloads with the tensor-core kernel, cascade with a "
                         "shared prefix")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="cache element type (fp8 = E4M3 codes with per-KV-head scales)")
    ap.add_argument("--num-splits", type=int, default=None,
                    help="override the planner's split count (tuning sweeps); 0 = the balanced one-wave "
                         "schedule of the single-launch step (fused and cascade paths)")
    ap.add_argument("--prefix-splits", type=int, default=None,
                    help="cascade workloads: split count of the shared-prefix pass (default: one wave of CTAs)")
    ap.add_argument("--no-graph", action="store_true",
                    help="single-launch step: launch each step from the host instead of replaying a "
                         "CUDA graph of consecutive steps")
    ap.add_argument("--requests", type=int, default=None,
                    help="run only the first N requests of the workload's seeded draw (their own lengths): "
                         "a smaller case of the same mix, for profiler captures")
    ap.add_argument("--out-dtype", default="bf16", choices=["bf16", "f32"],
                    help="element type of the step's output rows (the partials and lse stay fp32)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration table (it runs on one GPU, default workload only)")
    return ap.parse_args()


def default_steps(workload: str) -> int:
    # about one second of timed device work per workload (clock samples land in it)
    return {"tiny": 2000, "llama8b": 4000, "longctx": 800, "shard4": 800, "ragged": 250, "chunk": 1000,
            "specverify": 4000, "cascade": 4000}.get(workload, 200)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy kernel)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def tensor_peak():
    """Dense bf16 tensor throughput: the sustained figure (kernels timed inside
    a long step) of MEASURED_PEAKS.json."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d.get("bf16_tflops_sustained") or d["bf16_tflops"]), "measured (sustained cuBLAS bf16)"
    except Exception:
        return 1700.0, "fallback (sustained bf16)"


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    INTERVAL_MS = 50
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float, more_windows=()):
        """Clocks over the timed region [t0, t1]; `more_windows` are further
        timed regions of the same run (the per-configuration loops), counted in
        when the main region is too short for three samples."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        def within(a, b):
            return [r for r in rows if a - 0.03 <= r[0] <= b + 0.03]
        main = within(t0, t1)
        window = "timed region"
        inside = main
        if len(main) < 3 and more_windows:
            inside = main + [r for a, b in more_windows for r in within(a, b)]
            window = "timed region + the per-configuration timed loops (the timed region alone is %.0f ms)" % (
                (t1 - t0) * 1e3)
        if not inside:
            inside, window = rows[-3:], "last samples (no sample fell inside a timed region)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max([r[2] for r in inside]) if inside else None,
                "reasons": reasons, "samples": len(inside), "samples_in_timed_region": len(main),
                "interval_ms": self.INTERVAL_MS, "window": window}


# ----------------------------------------------------------------------------
# cross-rank aggregation (every rank runs its own copy of the workload)
# ----------------------------------------------------------------------------

def max_over_ranks(x: float) -> float:
    """The maximum of a per-rank float over all ranks (identity without a
    process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, seconds_max: float) -> float:
    """Weak scaling: all ranks' bytes over the slowest rank's time."""
    return bytes_per_rank * world / seconds_max / 1e9


# ----------------------------------------------------------------------------
# profile-derived DRAM traffic of the attention kernel (null if stale)
# ----------------------------------------------------------------------------

# the sources each DRAM-traffic record was captured from
DIGEST_SOURCES = {
    "decode": ("kf_decode_tc.cuh", "kf_decode_tc.cu", "kf_internal.cuh"),
    "mq5": ("kf_multiquery_tc05.cu", "kf_mq_tc05.cuh", "kf_tc05.cuh", "kf_decode_tc.cuh", "kf_internal.cuh"),
    "mqw": ("kf_multiquery_tc05w.cu", "kf_mq_tc05.cuh", "kf_tc05.cuh", "kf_decode_tc.cuh", "kf_internal.cuh"),
    "mqp": ("kf_multiquery_tc05p.cu", "kf_mq_tc05.cuh", "kf_tc05.cuh", "kf_decode_tc.cuh", "kf_internal.cuh"),
}


def kernel_source_digest(which: str = "decode") -> str:
    import hashlib
    h = hashlib.sha256()
    for f in DIGEST_SOURCES[which]:
        with open(os.path.join(ROOT, "paged_kv_decode_kf_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str, kv_bytes_per_launch: float, kv_dtype: str = "bf16"):
    """`kernel` is "tc" (attention launch of the three-call path) or "fused"
    (the single-launch step); records of FP8-cache runs are keyed
    "<workload>_fp8"."""
    path = os.path.join(ROOT, "profiles", "attention_dram_traffic.json")
    if kernel not in ("tc", "fused") or not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel_source_digest") != kernel_source_digest():
            return None
        key = workload if kv_dtype == "bf16" else workload + "_" + kv_dtype
        per = rec.get("per_workload" if kernel == "tc" else "per_workload_fused", {}).get(key)
        if per is None:
            return None
        # scaled to one launch of this run by the KV bytes it processes
        return per["dram_bytes_per_launch"] * kv_bytes_per_launch / per["kv_bytes_per_launch"]
    except Exception:
        return None


def l2_note(kv_bytes: float, dev) -> str:
    """Why no L2 flush runs between timed steps: the inputs a step reads (KV,
    plus the chunk queries of a multi-query step) exceed the L2, or the step is
    launch-bound anyway."""
    q_bytes = sum(t.numel() * t.element_size() for t in (dev.q, dev.q_chunk, dev.k_new, dev.v_new)
                  if t is not None)
    if kv_bytes > L2_BYTES:
        return "no flush: the %.2f GB of KV read per step exceeds the 129 MB L2" % (kv_bytes / 1e9)
    if kv_bytes + q_bytes > L2_BYTES:
        return ("no flush: the %.0f MB of inputs a step reads (KV %.0f MB + queries %.0f MB) exceed the 129 MB L2"
                % ((kv_bytes + q_bytes) / 1e6, kv_bytes / 1e6, q_bytes / 1e6))
    return "inputs fit in L2 (launch-bound case)"


def first_requests(w, n: int):
    """The first `n` requests of workload `w` with the context lengths its
    seeded draw gives them (same heads, dims, block size and cache type)."""
    from paged_kv_decode_kf_gb300 import workloads as wl
    if w.shared_prefix or w.chunk:
        raise SystemExit("--requests applies to the decode workloads")
    lay = wl.plan_layout(w)
    n = max(1, min(n, w.batch))
    return wl.scaled(w, batch=n, lengths=wl.Fixed(tuple(int(x) for x in lay.ctx_before[:n])),
                     name=w.name, seed=w.seed, description=w.description + " (first %d requests)" % n)


def workload_config(w) -> dict:
    """The `config` object of both arms' JSON lines: the workload and its
    sizes, from the seeded layout alone (so the GPU line and the oracle's
    line carry the same object for the same workload)."""
    from paged_kv_decode_kf_gb300 import workloads as wl
    lay = wl.plan_layout(w)
    kvpt = w.kv_bytes_per_token()
    logical = int(lay.ctx_after.astype("int64").sum()) * kvpt
    if w.shared_prefix:     # the prefix once, each request's suffix once
        read = (int(w.shared_prefix) + int((lay.suffix_ctx_before + 1).sum())) * kvpt
    else:
        read = logical
    elt = 2
    q_bytes = w.batch * w.num_q_heads * w.head_dim * elt + 2 * w.batch * w.num_kv_heads * w.head_dim * elt
    if w.chunk:
        q_bytes += w.batch * w.chunk * w.num_q_heads * w.head_dim * elt
    if read > L2_BYTES:
        l2 = "no flush: the %.2f GB of KV read per step exceeds the 129 MB L2" % (read / 1e9)
    elif read + q_bytes > L2_BYTES:
        l2 = ("no flush: the %.0f MB of inputs a step reads (KV %.0f MB + queries %.0f MB) exceed the 129 MB L2"
              % ((read + q_bytes) / 1e6, read / 1e6, q_bytes / 1e6))
    else:
        l2 = "inputs fit in L2 (launch-bound case)"
    return {"workload": w.name + ": " + w.description, "batch": w.batch, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "kv_dtype": w.kv_dtype, "kv_bytes_per_step": read, "logical_kv_bytes_per_step": logical,
            "l2": l2}


def profiled_mq_traffic(workload: str, rows_per_kv_head: int, kv_bytes_per_launch: float, head_dim: int = 128):
    """DRAM traffic of one launch of the tcgen05 multi-query kernel the library
    picks for this many query rows per KV head (the one-tile kernel up to 128,
    the wide one above), scaled to this launch by its KV bytes; None without a
    record for `workload` taken from the current sources of that kernel."""
    path = os.path.join(ROOT, "profiles", "multiquery_dram_traffic.json")
    kernel = "mq5" if rows_per_kv_head <= 128 else "mqw"
    try:
        with open(path) as f:
            rec = json.load(f)["kernels"][kernel]
        if rec.get("kernel_source_digest") != kernel_source_digest(kernel):
            return None
        per = rec.get("per_workload", {}).get(workload)
        if per is None:
            return None
        return per["dram_bytes_per_launch"] * kv_bytes_per_launch / per["kv_bytes_per_launch"]
    except Exception:
        return None


# ----------------------------------------------------------------------------
# reference arm and CPU baseline: the fp64 oracle on the host cores
# ----------------------------------------------------------------------------

def oracle_sample(w, target_s: float):
    """A bounded sample of workload `w` for the oracle: requests (drawn from
    the workload's own length distribution) until the estimated CPU time is
    about `target_s` on this machine's cores."""
    import numpy as np
    import oracle
    from paged_kv_decode_kf_gb300 import workloads as wl
    lay = wl.plan_layout(w)
    threads = oracle.default_threads()
    # rate probe on one short request
    probe = wl.scaled(w, batch=1, lengths=wl.Fixed((int(min(lay.ctx_before.min(), 4096)),)), name="probe")
    pi = wl.make_inputs(probe, "cpu")
    args = (wl.bf16_bits(pi.q), wl.bf16_bits(pi.k_cache), wl.bf16_bits(pi.v_cache), pi.block_tables.numpy(),
            pi.ctx_after.numpy())
    t = time.time()
    oracle.attention(*args, w.scale, threads=threads)
    dt = max(time.time() - t, 1e-4)
    tok_per_s = float(pi.ctx_after.sum()) / dt
    budget = tok_per_s * target_s
    if w.chunk:
        # chunked prefill: one request and the last `c` queries of its chunk (their
        # causal limits are those of the full chunk's last c queries), each query
        # attending to about L tokens
        b = int(np.random.default_rng(w.seed).integers(w.batch))
        L = int(lay.ctx_after[b])
        c = max(1, min(w.chunk, int(budget // L)))
        sample = wl.Workload(name=w.name + "-sample", batch=1, num_q_heads=w.num_q_heads,
                             num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
                             lengths=wl.Fixed((int(lay.ctx_before[b]),)), seed=w.seed + 7919, chunk=c,
                             description=w.description)
        return sample, threads
    order = np.random.default_rng(w.seed).permutation(w.batch)
    chosen, tot = [], 0
    for b in order:
        if chosen and tot + lay.ctx_after[b] > budget:
            break
        chosen.append(int(b))
        tot += int(lay.ctx_after[b])
    lens = tuple(int(lay.ctx_before[b]) for b in chosen)
    sample = wl.scaled(w, batch=len(lens), lengths=wl.Fixed(lens), name=w.name + "-sample", spare_blocks=0)
    return sample, threads


def run_oracle_step(si, threads):
    import oracle
    from paged_kv_decode_kf_gb300 import workloads as wl
    if si.workload.chunk:
        # causal chunk query j of c over L tokens = attention over its first
        # L - c + j + 1 tokens: the c queries as c requests sharing the table,
        # through the threaded decode oracle
        import numpy as np
        c, L = si.workload.chunk, int(si.ctx_after[0])
        bt = np.repeat(si.block_tables.numpy()[:1], c, axis=0)
        lim = (L - c + 1 + np.arange(c)).astype(np.int32)
        return oracle.attention(wl.bf16_bits(si.q_chunk), wl.bf16_bits(si.k_cache), wl.bf16_bits(si.v_cache),
                                bt, lim, si.workload.scale, threads=threads)
    k2, v2, _ = oracle.append(wl.bf16_bits(si.k_cache), wl.bf16_bits(si.v_cache), wl.bf16_bits(si.k_new),
                              wl.bf16_bits(si.v_new), si.block_tables.numpy(), si.ctx_before.numpy())
    return oracle.attention(wl.bf16_bits(si.q), k2, v2, si.block_tables.numpy(), si.ctx_after.numpy(),
                            si.workload.scale, threads=threads)


def sample_kv_bytes(si, w) -> float:
    """KV bytes a sample stands for, in the GPU line's unit: a chunked-prefill
    sample computes c of its request's C chunk queries, so c/C of its KV."""
    kv = float(si.kv_bytes())
    return kv * si.workload.chunk / w.chunk if w.chunk else kv


def cpu_baseline(w, target_s=12.0):
    from paged_kv_decode_kf_gb300 import workloads as wl
    sample, threads = oracle_sample(w, target_s)
    si = wl.make_inputs(sample, "cpu")
    passes = 0
    t = time.time()
    while True:                      # repeat the sample until ~target_s of CPU work
        run_oracle_step(si, threads)
        passes += 1
        dt = time.time() - t
        if dt >= target_s or passes >= 1000:
            break
    kv = sample_kv_bytes(si, w)
    return {"value": kv * passes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d requests of the %s workload (%d tokens, %.2f GB of KV); %d append + "
                      "attention passes in fp64 C over all query heads, %.1f s"
                      % (sample.batch, w.batch, w.name, int(si.ctx_after.sum()), kv / 1e9, passes, dt)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_kv_decode_kf_gb300 import workloads as wl
    w = wl.CONFIGS[args.workload]
    K = args.steps if args.steps is not None else 5
    W = args.warmup
    per_step_s = max(1.0, min(10.0, 120.0 / max(1, K + W)))
    sample, threads = oracle_sample(w, per_step_s)
    si = wl.make_inputs(sample, "cpu")
    for _ in range(W):
        run_oracle_step(si, threads)
    t = time.time()
    for _ in range(K):
        run_oracle_step(si, threads)
    dt = (time.time() - t) / max(K, 1)
    kv = sample_kv_bytes(si, w)
    value = kv / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "run": {"sample_requests": sample.batch, "sample_kv_bytes": kv,
                "path": "fp64 C oracle: append, then attention over every query head, threaded over rows"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "%d of %d requests of %s per step (%.3f GB of KV)"
                                   % (sample.batch, w.batch, w.name, kv / 1e9)},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# every decode configuration in one run
# ----------------------------------------------------------------------------

PER_CONFIG = ("tiny", "llama8b", "longctx", "shard4", "ragged")


def percentile(xs, q: float) -> float:
    """Linear-interpolated percentile q in [0, 100] of a non-empty list."""
    ys = sorted(xs)
    pos = (len(ys) - 1) * q / 100.0
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def step_distribution(step, min_samples: int = 50, target_s: float = 0.3):
    """Per-step device times (ms) of `step` replayed from CUDA graphs.

    A sample is one graph replay of g consecutive steps divided by g, with g
    the smallest count that makes a sample at least 1 ms (g = 1 for a step that
    long on its own), so a replay's own launch cost weighs little. The stream
    first sleeps while the host enqueues every replay and event, so the events
    see device time, not host launch gaps. Returns (samples, g, the wall-clock
    window of the loop)."""
    import torch
    for _ in range(5):
        step.run()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(10):
        step.run()
    b.record()
    torch.cuda.synchronize()
    est_ms = max(a.elapsed_time(b) / 10, 1e-3)
    g = max(1, int(math.ceil(1.0 / est_ms)))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(g):
            step.run()
    graph.replay()
    torch.cuda.synchronize()
    n = int(min(2000, max(min_samples, math.ceil(target_s * 1e3 / (g * est_ms)))))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    t0 = time.time()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(40_000_000)        # ~20 ms at 2 GHz: the host enqueues ahead
    ev[0].record()
    for i in range(n):
        graph.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    t1 = time.time()
    samples = [ev[i].elapsed_time(ev[i + 1]) / g for i in range(n)]
    del graph
    return samples, g, (t0, t1)


def step_phases(step, n: int = 20):
    """Device time of each launch of a multi-launch step (append, attention
    per view, merge), from host-launched steps enqueued behind a stream sleep;
    None for the one-launch step."""
    import torch
    if step.fused:
        return None
    nv = len(step.views)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nv + 3)] for _ in range(n)]
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(40_000_000)
    from paged_kv_decode_kf_gb300 import kf
    i_ = step.inp
    for e in evs:
        e[0].record()
        if step.with_append:
            step.append()
        e[1].record()
        S = step.num_splits
        for j, (bt, ctx, max_ctx) in enumerate(step.views):
            # one attention launch per token-range view, as DecodeStep.attention
            if step.fp8:
                kf.kf_paged_decode_attention_fp8(i_.q, i_.k_cache, i_.v_cache, i_.k_scale, i_.v_scale, bt, ctx,
                                                 max_ctx, step.w.scale, S, step.out_partial[j * S:(j + 1) * S],
                                                 step.lse_partial[j * S:(j + 1) * S])
            else:
                kf.kf_paged_decode_attention(i_.q, i_.k_cache, i_.v_cache, bt, ctx, max_ctx, step.w.scale, S,
                                             step.out_partial[j * S:(j + 1) * S],
                                             step.lse_partial[j * S:(j + 1) * S])
            e[2 + j].record()
        step.merge()
        e[nv + 2].record()
    torch.cuda.synchronize()
    med = lambda k: statistics.median(e[k].elapsed_time(e[k + 1]) for e in evs) * 1e3
    out = {"append_us": med(0)}
    for j in range(nv):
        out["attention_%d_us" % j] = med(1 + j)
    out["merge_us"] = med(nv + 1)
    return out


def per_config_table(device: str, out_dtype, reuse: dict, peak: float, oracle_s: float = 3.0):
    """Every decode configuration on this GPU: per-step distribution, KV GB/s
    and its fraction of `peak`, the per-launch split of multi-launch steps,
    and the fp64 oracle on the host cores on a bounded sample of the same
    configuration. `reuse` maps a configuration name to inputs already on the
    device. Returns (table, timed windows)."""
    import torch
    from paged_kv_decode_kf_gb300 import workloads as wl
    from paged_kv_decode_kf_gb300.step import DecodeStep
    table, windows = {}, []
    for name in PER_CONFIG:
        w = wl.CONFIGS[name]
        dev = reuse.get(name) or wl.make_inputs(w, device)
        step = DecodeStep(dev, fused=not w.shards, out_dtype=out_dtype)
        samples, g, win = step_distribution(step)
        windows.append(win)
        phases = step_phases(step)
        from paged_kv_decode_kf_gb300 import kf
        flags = kf.kf_get_device_error()
        if flags:
            raise RuntimeError("device error word 0x%x after the %s loop" % (flags, name))
        kv = float(dev.kv_bytes())
        med = statistics.median(samples)
        gbs = kv / (med * 1e-3) / 1e9
        cpu = cpu_baseline(w, target_s=oracle_s)
        table[name] = {
            "workload": w.description, "batch": w.batch, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "num_splits": step.num_splits, "kv_bytes_per_step": int(kv),
            "path": ("kf_decode_step (one launch)" if step.fused else
                     "kf_append_kv + kf_paged_decode_attention x%d + kf_merge_partials" % len(step.views)),
            "us_median": med * 1e3, "us_p10": percentile(samples, 10) * 1e3,
            "us_p90": percentile(samples, 90) * 1e3, "samples": len(samples), "steps_per_sample": g,
            "kv_gbs": gbs, "frac": gbs / peak, "launches_per_step": step.launches_per_step,
            "launch_us": phases,
            "oracle": {"value": cpu["value"], "unit": "GB/s", "cores": cpu["cores"], "sample": cpu["sample"]},
            "gpu_over_oracle": gbs / cpu["value"] if cpu["value"] > 0 else None,
        }
        if name not in reuse:
            del step, dev
            torch.cuda.empty_cache()
    return table, windows


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def e2e_breakdown(e2e_step, graph, body, stage_dev, stage_host, res_dev, res_host, step, wall_s, n=50):
    """Where an end-to-end step's time goes: the H2D copy, the device step
    and the D2H copy, each timed alone with events (enqueued ahead, behind a
    stream sleep); the span one step takes
    on the device (events around its graph launch); the host time spent in
    the launch call; and the rest of the wall time (launch latency and the
    host waking from its wait), as medians in us."""
    import torch

    def timed(fn, reps=20):
        # enqueued behind a stream sleep, so the events bracket device time only
        # (not the host's enqueue of each copy or launch)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(10_000_000)
        for a, b in evs:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)

    h2d = timed(lambda: stage_dev.copy_(stage_host, non_blocking=True))
    d2h = timed(lambda: res_host.copy_(res_dev, non_blocking=True))
    dev_step = timed(step.run)
    spans, launches = [], []
    for _ in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t = time.perf_counter()
        a.record()
        if graph is not None:
            graph.replay()
        else:
            body()
        b.record()
        launches.append((time.perf_counter() - t) * 1e6)
        torch.cuda.synchronize()
        spans.append(a.elapsed_time(b) * 1e3)
    span = statistics.median(spans)
    return {"h2d_us": h2d, "step_us": dev_step, "d2h_us": d2h, "device_span_us": span,
            "host_launch_call_us": statistics.median(launches),
            "host_launch_latency_and_wait_us": wall_s * 1e6 - span}


def zero_copy_e2e(step, K: int, world: int, kv_bytes: int, barrier, use_graph: bool):
    """End to end through kf_decode_step with the step's per-step inputs (q,
    k_new, v_new, context lengths, block tables) and its result (out, lse) in
    pinned host memory, which the step kernel reads and writes in place over
    the CPU-GPU link (CUDA unified addressing): no copy launches, the bytes
    still cross the link every step. Each step is one launch (a CUDA graph of
    the call) and the host's wait for the result. Returns the e2e record, with
    whether the result equals the device-buffer step's bit for bit."""
    import copy
    import torch
    from paged_kv_decode_kf_gb300.step import DecodeStep

    inp = copy.copy(step.inp)
    h2d = 0
    for n in ("q", "k_new", "v_new", "ctx_before", "block_tables"):
        t = getattr(inp, n).cpu().pin_memory()
        setattr(inp, n, t)
        h2d += t.numel() * t.element_size()
    zs = DecodeStep(inp, num_splits=step.num_splits, fused=True, out_dtype=step.out.dtype)
    zs.out = torch.empty(zs.out.shape, dtype=zs.out.dtype).pin_memory()
    zs.lse = torch.empty(zs.lse.shape, dtype=torch.float32).pin_memory()
    d2h = zs.out.numel() * zs.out.element_size() + zs.lse.numel() * 4

    zs.run()
    torch.cuda.synchronize()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            zs.run()

    def launch():
        if graph is not None:
            graph.replay()
        else:
            zs.run()

    def one():
        launch()
        torch.cuda.synchronize()

    Ke = max(3, min(K, 400))
    for _ in range(3):
        one()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(Ke):
        one()
    te = (time.perf_counter() - t0) / Ke
    barrier()
    te = max_over_ranks(te)

    step.run()                      # the same step with device buffers
    torch.cuda.synchronize()
    same = bool(torch.equal(zs.out, step.out.cpu()) and torch.equal(zs.lse, step.lse.cpu()))

    def timed(fn, reps=20):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(10_000_000)
        for a, b in evs:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)

    launches = []
    for _ in range(50):
        t = time.perf_counter()
        launch()
        launches.append((time.perf_counter() - t) * 1e6)
        torch.cuda.synchronize()
    step_us = timed(zs.run)
    return {"value": whole_job_gbs(kv_bytes, world, te), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": te * 1e3, "steps": Ke,
            "out_dtype": "bf16" if zs.out.dtype == torch.bfloat16 else "f32",
            "copies_per_step": "none: the step kernel reads q, k_new, v_new, context lengths and block "
                               "tables from pinned host memory and writes out and lse there (zero-copy)",
            "launch": ("one CUDA graph of the kf_decode_step call per step" if graph is not None
                       else "one kf_decode_step call per step") + ", host waits for the result",
            "result_equals_device_buffer_step": same,
            "breakdown": {"step_us": step_us, "step_with_device_buffers_us": timed(step.run),
                          "host_launch_call_us": statistics.median(launches),
                          "host_launch_latency_and_wait_us": te * 1e6 - step_us}}


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    os.environ["KF_DECODE_IMPL"] = args.decode_kernel

    import __graft_entry__ as g
    g.build()
    from paged_kv_decode_kf_gb300 import workloads as wl
    from paged_kv_decode_kf_gb300.step import DecodeStep

    w = wl.CONFIGS[args.workload]
    if args.kv_dtype != "bf16":
        w = wl.with_kv_dtype(w, args.kv_dtype)
    if args.requests is not None:
        w = first_requests(w, args.requests)
    K = args.steps if args.steps is not None else default_steps(args.workload)
    W = max(args.warmup, 3)
    out_dtype = torch.bfloat16 if args.out_dtype == "bf16" else torch.float32
    dev = wl.make_inputs(w, "cuda:%d" % local)
    fused = args.path == "fused" or (args.path == "auto" and not w.shards and not w.shared_prefix
                                     and not w.chunk and args.decode_kernel == "tc")
    if w.kv_dtype == "fp8" and args.decode_kernel != "tc":
        raise SystemExit("the FP8 cache is served by the tensor-core kernel only")
    cascade = bool(w.shared_prefix) and args.path in ("auto", "cascade", "cascade-serial", "cascade-calls")
    chunk = bool(w.chunk)
    if cascade:
        from paged_kv_decode_kf_gb300.step import CascadeStep
        step = CascadeStep(dev, prefix_splits=args.prefix_splits, suffix_splits=args.num_splits,
                           fused_suffix=args.path != "cascade-calls", out_dtype=out_dtype,
                           concurrent=args.path in ("auto", "cascade"))
        kv_bytes = step.unique_kv_bytes()      # the prefix once, each suffix once
    elif chunk:
        from paged_kv_decode_kf_gb300.step import ChunkStep
        step = ChunkStep(dev, num_splits=args.num_splits)
        kv_bytes = dev.kv_bytes()              # each request's cached tokens, once
    else:
        step = DecodeStep(dev, num_splits=args.num_splits, fused=fused, out_dtype=out_dtype)
        kv_bytes = dev.kv_bytes()
    logical_kv_bytes = dev.kv_bytes()          # sum over requests of their whole context
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(W):
        step.run()
    torch.cuda.synchronize()

    # One step with its phases bracketed by events (recorded on the current
    # stream): fused: [the launch]; concurrent cascade, its kernels one after
    # another so that each is timed alone: prefix pass | suffix step | merge;
    # cascade with the fused suffix: prefix pass | prefix merge | suffix step;
    # cascade as calls: append | prefix | suffix | merge; otherwise append,
    # [attention] | merge.
    def one_step(e):
        if step.fused:
            e[0].record()
            step.step_fused()
            e[1].record()
            return
        if cascade:
            if step.concurrent:
                e[0].record()
                step.prefix()
                e[1].record()
                step.suffix_slot()
                e[2].record()
                step.final_merge()
                e[3].record()
                return
            if step.fused_suffix:
                e[0].record()
                step.prefix()
                e[1].record()
                step.prefix_merge()
                e[2].record()
                step.suffix_step()
                e[3].record()
                return
            e[0].record()
            step.append()
            e[1].record()
            step.prefix()
            e[2].record()
            step.suffix()
            e[3].record()
            step.merge()
            e[4].record()
            return
        if step.with_append:
            step.append()
        e[0].record()
        step.attention()
        e[1].record()
        step.merge()

    # Every path's calls are capturable (no host synchronisation, no
    # allocation), so, as a serving loop would, the timed region replays a
    # CUDA graph of n consecutive steps (n the largest divisor of K up to 50):
    # every replay re-runs all of each step's work, without the host launch gap
    # between launches. Events inside the graph would serialise it, so the
    # graph holds the bare steps; per-launch times come from the step time
    # (one launch per step) or, for paths of several launches, from an
    # event-timed pass of host-launched steps right after the timed region.
    def events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(5)]

    graph, g_steps = None, 0
    if not args.no_graph:
        g_steps = max(d for d in range(1, min(K, 50) + 1) if K % d == 0)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(g_steps):
                step.run()
        graph.replay()
        torch.cuda.synchronize()

    # ---- device-timed region ----
    n_att = len(step.views)
    ev = [events() for _ in range(K)] if graph is None else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for _ in range(K // g_steps if graph is not None else 0):
        graph.replay()
    # (a concurrent cascade step runs as it is; its kernels are timed alone
    # after the region)
    concurrent = cascade and step.concurrent
    for i in range(K if graph is None else 0):
        if concurrent:
            step.run()
        else:
            one_step(ev[i])
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    ms = start.elapsed_time(end) / K
    phase_source = "events in the timed region (host launches)"
    if (graph is not None or concurrent) and not step.fused:
        # the stream first sleeps (a bounded clock spin) while the host enqueues
        # every step, so the events see device time, not host launch gaps
        ev = [events() for _ in range(min(K, 20))]
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(40_000_000)   # ~20 ms at 2 GHz
        for e in ev:
            one_step(e)
        torch.cuda.synchronize()
        phase_source = "event-timed pass of %d steps enqueued behind a stream sleep, after the timed region" % len(ev)
        if concurrent:
            phase_source += " (the cascade's kernels one after another, each timed alone)"
    elif graph is not None:
        phase_source = "one launch per step: the graph-replayed step time bounds the launch"
    span = lambda k: sum(e[k].elapsed_time(e[k + 1]) for e in ev) / len(ev)
    if cascade:
        if step.concurrent:     # as (append, prefix, suffix, merge): the append is inside the suffix step
            phase_ms = [0.0, span(0), span(1), span(2)]
        elif step.fused_suffix:
            phase_ms = [0.0, span(0), span(2), span(1)]
        else:
            phase_ms = [span(k) for k in range(4)]
        att_ms = phase_ms[1] + phase_ms[2]
    elif graph is not None and step.fused:
        att_ms = ms
    else:
        att_ms = span(0)
    from paged_kv_decode_kf_gb300 import kf
    flags = kf.kf_get_device_error()
    if flags:
        sys.stderr.write("device error word 0x%x after the timed region\n" % flags)
        sys.exit(1)
    ms = max_over_ranks(ms)
    value = whole_job_gbs(kv_bytes, world, ms * 1e-3)

    # ---- end to end through the C ABI with host buffers ----
    # The step's inputs (q, k_new, v_new, context lengths, block tables) live in
    # one device staging buffer with a pinned host twin, so one H2D copy per
    # step refreshes them all; out and lse share one buffer read back by one
    # D2H copy.
    e2e, e2e_copies = None, None
    if not args.no_e2e:
        names = ["q", "k_new", "v_new", "ctx_before", "ctx_after", "block_tables"]
        for extra in ("prefix_table", "suffix_tables", "suffix_ctx_before", "suffix_ctx_after", "q_chunk",
                      "q_start"):
            if getattr(dev, extra) is not None:
                names.append(extra)
        tensors = [getattr(dev, n) for n in names]
        if w.shards:
            names += ["tail_tables", "tail_ctx_before"]
            tensors += [dev.tail_tables, dev.tail_ctx_before]
            for j, sv in enumerate(dev.shards):
                names += ["shard_bt%d" % j, "shard_ctx%d" % j]
                tensors += [sv.block_tables, sv.ctx_after]
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        stage_dev = torch.empty(off, dtype=torch.uint8, device=dev.q.device)
        stage_host = torch.empty(off, dtype=torch.uint8).pin_memory()
        views = []
        for t, o in zip(tensors, offs):
            nbytes = t.numel() * t.element_size()
            v = stage_dev[o:o + nbytes].view(t.dtype).view(t.shape)
            v.copy_(t)
            stage_host[o:o + nbytes].copy_(t.view(torch.uint8).reshape(-1).cpu())
            views.append(v)
        for n, v in zip(names, views):       # the step now reads its inputs from the staging buffer
            if n.startswith("shard_bt"):
                dev.shards[int(n[8:])].block_tables = v
            elif n.startswith("shard_ctx"):
                dev.shards[int(n[9:])].ctx_after = v
            else:
                setattr(dev, n, v)
        if cascade:
            step_e = CascadeStep(dev, prefix_splits=step.Sp, suffix_splits=step.Ss, fused_suffix=step.fused_suffix,
                                 out_dtype=out_dtype, concurrent=step.concurrent)
        elif chunk:
            step_e = ChunkStep(dev, num_splits=step.S)
        else:
            step_e = DecodeStep(dev, num_splits=step.num_splits, fused=step.fused, out_dtype=out_dtype)
        ob = step_e.out.numel() * step_e.out.element_size()
        res_dev = torch.empty(ob + step_e.lse.numel() * 4, dtype=torch.uint8, device=dev.q.device)
        step_e.out = res_dev[:ob].view(step_e.out.dtype).view(step_e.out.shape)
        step_e.lse = res_dev[ob:].view(torch.float32).view(step_e.lse.shape)
        res_host = torch.empty(res_dev.numel(), dtype=torch.uint8).pin_memory()
        h2d, d2h = off, res_dev.numel()

        def e2e_body():
            stage_dev.copy_(stage_host, non_blocking=True)
            step_e.run()
            res_host.copy_(res_dev, non_blocking=True)

        # as in the timed region: one graph launch per step (the copies from and
        # to pinned memory are captured with the calls), then the host waits for
        # the result, as a decode loop must before it knows the next input
        e2e_graph = None
        if not args.no_graph:
            e2e_body()
            torch.cuda.synchronize()
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph):
                e2e_body()

        def e2e_step():
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_body()
            torch.cuda.synchronize()

        Ke = max(3, min(K, 400))
        for _ in range(3):
            e2e_step()
        barrier()
        torch.cuda.synchronize()
        te0 = time.perf_counter()
        for _ in range(Ke):
            e2e_step()
        te = (time.perf_counter() - te0) / Ke
        barrier()
        te = max_over_ranks(te)
        e2e = {"value": whole_job_gbs(kv_bytes, world, te), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": te * 1e3, "steps": Ke,
               "out_dtype": args.out_dtype,
               "copies_per_step": "1 H2D (pinned, all inputs) + 1 D2H (out and lse)",
               "launch": "one CUDA graph per step (copies + calls), host waits for the result"
               if e2e_graph is not None else "host launches, host waits for the result",
               "breakdown": e2e_breakdown(e2e_step, e2e_graph, e2e_body, stage_dev, stage_host, res_dev, res_host,
                                          step_e, te)}
        if step.fused:
            # the single-launch step also takes its per-step tensors in pinned
            # host memory: the headline e2e, the copy-based run kept beside it
            e2e_copies = e2e
            e2e = zero_copy_e2e(step, K, world, kv_bytes, barrier, not args.no_graph)

    peak, peak_src = hbm_peak()
    per_config, windows = None, []
    if (world == 1 and not args.no_per_config and args.workload == "ragged" and w.kv_dtype == "bf16"
            and args.requests is None
            and args.path == "auto" and args.num_splits is None and args.decode_kernel == "tc"):
        per_config, windows = per_config_table("cuda:%d" % local, out_dtype, {w.name: dev}, peak)
    clk = clocks.stop(t0, t1, windows)
    att_gbs = kv_bytes / (att_ms * 1e-3) / 1e9
    if cascade:
        # Two kernels carry the step: the shared-prefix pass, a dense contraction
        # (every query against every prefix key: 4 D FLOPs per token and query
        # row) bound by the bf16 tensor pipe, and the suffix decode, bound by
        # HBM. The roofline reports the one that takes longer; both are in
        # "kernels".
        tpk, tsrc = tensor_peak()
        pre_s, suf_s = phase_ms[1] * 1e-3, phase_ms[2] * 1e-3
        pre_tf = step.prefix_flops() / pre_s / 1e12
        suf_gbs = step.suffix_kv_bytes() / suf_s / 1e9
        kernels = {"path": "3 launches: the prefix pass and kf_decode_step (append + suffix attention + "
                           "merge of the suffix splits into one slot) on two streams at the same time, then "
                           "one merge of the prefix slots with the suffix slot; the per-kernel times are "
                           "each kernel alone, the step overlaps the first two" if step.concurrent else
                           "3 launches: prefix pass, merge of its partials into one, then "
                           "kf_decode_step_merge_partials (append + suffix attention + merge with the "
                           "prefix partial)" if step.fused_suffix else
                           "4 launches: append, prefix pass, suffix decode, merge",
                   "append_us": phase_ms[0] * 1e3, "prefix_pass_us": phase_ms[1] * 1e3,
                   "suffix_decode_us": phase_ms[2] * 1e3, "merge_us": phase_ms[3] * 1e3,
                   "prefix_pass": {"bound": "tensor", "achieved": pre_tf, "peak": tpk, "unit": "TFLOP/s",
                                   "frac": pre_tf / tpk, "algorithmic_flops": step.prefix_flops(),
                                   "peak_source": tsrc + (", of measured" if tsrc.startswith("measured")
                                                          else ", of fallback")},
                   "suffix_decode": {"bound": "hbm", "achieved": suf_gbs, "peak": peak, "unit": "GB/s",
                                     "frac": suf_gbs / peak, "algorithmic_bytes": step.suffix_kv_bytes()},
                   # the whole step against its two floors: the unique KV bytes at the HBM
                   # peak and the prefix FLOPs at the tensor peak
                   "step": {"us": ms * 1e3, "hbm_floor_us": kv_bytes / (peak * 1e9) * 1e6,
                            "tensor_floor_us": step.prefix_flops() / (tpk * 1e12) * 1e6,
                            "frac_of_hbm_floor": kv_bytes / (peak * 1e9) / (ms * 1e-3)}}
        dom = kernels["prefix_pass"] if pre_s >= suf_s else kernels["suffix_decode"]
        roofline_override = dict(dom, traffic=None,
                                 kernel="shared-prefix multi-query pass" if pre_s >= suf_s
                                 else "suffix decode attention",
                                 peak_source=(lambda src: src + (", of measured" if src.startswith("measured")
                                                                 else ", of fallback"))(
                                     tsrc if pre_s >= suf_s else peak_src),
                                 kernels=kernels)
    elif chunk:
        # every chunk query against its history and the causal part of its
        # chunk: a dense contraction whose bound follows its arithmetic
        # intensity -- the bf16 tensor roofline for long chunks (prefill),
        # HBM for a few queries per request (speculative verify)
        tpk, tsrc = tensor_peak()
        intensity = step.flops() / kv_bytes                    # FLOPs per KV byte read
        if intensity >= tpk * 1e12 / (peak * 1e9):
            tf = step.flops() / (att_ms * 1e-3) / 1e12
            roofline_override = {"bound": "tensor", "achieved": tf, "peak": tpk, "unit": "TFLOP/s",
                                 "frac": tf / tpk, "algorithmic_flops_per_launch": step.flops(),
                                 "peak_source": tsrc + (", of measured" if tsrc.startswith("measured")
                                                        else ", of fallback")}
        else:
            roofline_override = {"bound": "hbm", "achieved": att_gbs, "peak": peak, "unit": "GB/s",
                                 "frac": att_gbs / peak, "algorithmic_bytes_per_launch": kv_bytes,
                                 "peak_source": peak_src + (", of measured" if peak_src.startswith("measured")
                                                            else ", of fallback")}
        roofline_override.update({"traffic": profiled_mq_traffic(w.name, step.C * w.group, kv_bytes, w.head_dim),
                                  "kernel": "multi-query attention (chunk queries, causal)",
                                  "flops_per_kv_byte": intensity, "avg_launch_us": att_ms * 1e3,
                                  # no merge launch with one split and fp32 output
                                  "merge_us": (ms - att_ms) * 1e3 if step.merges else 0.0})
    else:
        roofline_override = None
    per_launch_kv = kv_bytes / n_att
    traffic = profiled_traffic(w.name, "fused" if step.fused else args.decode_kernel, per_launch_kv, w.kv_dtype)
    kname = ("decode step, one launch (append + attention + merge)" if step.fused
             else "shared-prefix multi-query pass + suffix decode attention" if cascade
             else "decode attention (%s)" % args.decode_kernel)
    roofline = {"bound": "hbm", "achieved": att_gbs, "peak": peak, "unit": "GB/s", "frac": att_gbs / peak,
                "traffic": traffic, "kernel": kname,
                "launches_per_step": n_att, "algorithmic_bytes_per_launch": per_launch_kv,
                "avg_launch_us": att_ms * 1e3 / n_att, "peak_source": peak_src + ", of measured"
                if peak_src.startswith("measured") else peak_src + ", of fallback"}

    if roofline_override is not None:
        roofline = roofline_override
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        cfg = workload_config(w)
        # the layout's own count must be what was timed
        assert cfg["kv_bytes_per_step"] == kv_bytes and cfg["logical_kv_bytes_per_step"] == logical_kv_bytes, (
            cfg, kv_bytes, logical_kv_bytes)
        assert cfg["l2"] == l2_note(kv_bytes, dev), (cfg["l2"], l2_note(kv_bytes, dev))
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms, "us_per_step": ms * 1e3, "pct_of_hbm_peak": 100.0 * value / world / peak,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.kv_dtype == "bf16" else "fp8 e4m3 KV, bf16 q",
            "accumulate": "f32", "data": "synthetic",
            "config": cfg,
            "run": {"num_splits": step.num_splits, "out_dtype": args.out_dtype,
                       "decode_kernel": args.decode_kernel,
                       "heads_per_cta_override": os.environ.get("KF_TC_HPC"),
                       "num_splits_source": "planner" if args.num_splits is None else "--num-splits",
                       "step": ("chunk attention (multi-query, causal) + LSE merge" if chunk else
                                "append + split attention + LSE merge"),
                       "path": "kf_decode_step (one launch)" if step.fused else
                               ("kf_paged_multiquery_attention (prefix, once) || kf_decode_step (append + "
                                "suffixes + their merge, second stream), then kf_merge_partials (prefix slots + "
                                "suffix slot)" if step.concurrent else
                                "kf_paged_multiquery_attention (prefix, once) + kf_merge_partials (prefix "
                                "slots into one) + kf_decode_step_merge_partials (append + suffixes + merge)"
                                if step.fused_suffix else
                                "kf_append_kv + kf_paged_multiquery_attention (prefix, once) + "
                                "kf_paged_decode_attention (suffixes) + kf_merge_partials") if cascade else
                               ("kf_paged_multiquery_attention (causal chunks) + kf_merge_partials" if step.merges
                                else "kf_paged_multiquery_attention (causal chunks; one split: its partial slot "
                                     "is the output)") if chunk else
                               "kf_append_kv + kf_paged_decode_attention x%d + kf_merge_partials" % n_att,
                       "launch": ("CUDA graph replay, %d steps per graph" % g_steps if graph is not None
                                  else "host launches, one step at a time"),
                       "launch_times": phase_source,
                       "effective_gbs": logical_kv_bytes / (ms * 1e-3) / 1e9,
                       "parallelism": "replica per GPU" if world > 1 else "1 GPU"},
            "roofline": roofline,
            "e2e": e2e,
            "e2e_copies": e2e_copies,
            "cpu_baseline": cpu,
            "per_config": per_config,
            "clocks": clk,
            "gpu_launches": K * step.launches_per_step,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
