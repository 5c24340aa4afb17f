"""One decode step through the C ABI: append, split attention, merge.

Orchestration of library calls only (buffers come from torch). For a
workload spread over token-range shards, the append goes through the tail
table (the shard holding each request's newest position), each shard's
attention writes its own partial slots, and one merge combines all slots,
as KernelFlume (academ.us/article/2606.29207) section 3.2 describes for
attention nodes.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import kf
from .workloads import DecodeInputs


class DecodeStep:
    """One decode step over `inp`. fused=True runs kf_decode_step (one launch;
    not for sharded workloads); otherwise kf_append_kv, one
    kf_paged_decode_attention per token-range view, kf_merge_partials."""

    def __init__(self, inp: DecodeInputs, num_splits: Optional[int] = None,
                 out_dtype=torch.float32, with_append: bool = True, fused: bool = False):
        self.inp = inp
        w = inp.workload
        self.w = w
        self.with_append = with_append
        if fused and (w.shards or not with_append):
            raise ValueError("the single-launch step covers unsharded workloads with the append")
        self.fused = fused
        B, Hq, D = w.batch, w.num_q_heads, w.head_dim
        dev = inp.q.device
        # host-side bounds, computed once: reading them per step would synchronise
        self.max_ctx = inp.max_ctx_after
        if w.shards:
            self.views = [(s.block_tables, s.ctx_after, int(s.ctx_after.max().item())) for s in inp.shards]
        else:
            self.views = [(inp.block_tables, inp.ctx_after, self.max_ctx)]
        if num_splits is None:
            num_splits = max(self.plan(v[1], v[2]) for v in self.views)
        self.num_splits = int(num_splits)
        slots = self.num_splits * len(self.views)
        self.out_partial = torch.empty((slots, B, Hq, D), dtype=torch.float32, device=dev)
        self.lse_partial = torch.empty((slots, B, Hq), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, Hq, D), dtype=out_dtype, device=dev)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        self.workspace = None
        if fused:
            self.workspace = kf.make_workspace(B, Hq, w.num_kv_heads, D, self.num_splits, dev)

    def plan(self, ctx_lens: torch.Tensor, max_ctx: int) -> int:
        w = self.w
        return kf.kf_choose_num_splits(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                       w.block_size, max_ctx, ctx_lens.cpu().numpy().astype(np.int32),
                                       kv_dtype=w.kv_dtype)

    @property
    def fp8(self) -> bool:
        return self.w.kv_dtype == "fp8"

    def append(self, stream=None) -> None:
        i = self.inp
        if self.fp8:
            bt, ctx = (i.tail_tables, i.tail_ctx_before) if self.w.shards else (i.block_tables, i.ctx_before)
            kf.kf_append_kv_fp8(i.k_new, i.v_new, i.k_cache, i.v_cache, i.k_scale, i.v_scale, bt, ctx, stream)
            return
        if self.w.shards:
            kf.kf_append_kv(i.k_new, i.v_new, i.k_cache, i.v_cache, i.tail_tables, i.tail_ctx_before, stream)
        else:
            kf.kf_append_kv(i.k_new, i.v_new, i.k_cache, i.v_cache, i.block_tables, i.ctx_before, stream)

    def attention(self, stream=None) -> None:
        i, S = self.inp, self.num_splits
        for j, (bt, ctx, max_ctx) in enumerate(self.views):
            if self.fp8:
                kf.kf_paged_decode_attention_fp8(i.q, i.k_cache, i.v_cache, i.k_scale, i.v_scale, bt, ctx,
                                                 max_ctx, self.w.scale, S, self.out_partial[j * S:(j + 1) * S],
                                                 self.lse_partial[j * S:(j + 1) * S], stream)
            else:
                kf.kf_paged_decode_attention(i.q, i.k_cache, i.v_cache, bt, ctx, max_ctx, self.w.scale, S,
                                             self.out_partial[j * S:(j + 1) * S],
                                             self.lse_partial[j * S:(j + 1) * S], stream)

    def merge(self, stream=None) -> None:
        kf.kf_merge_partials(self.out_partial, self.lse_partial, self.out, lse_out=self.lse, stream=stream)

    def step_fused(self, stream=None) -> None:
        i = self.inp
        if self.fp8:
            kf.kf_decode_step_fp8(i.q, i.k_new, i.v_new, i.k_cache, i.v_cache, i.k_scale, i.v_scale,
                                  i.block_tables, i.ctx_before, self.max_ctx, self.w.scale, self.num_splits,
                                  self.workspace, self.out, lse_out=self.lse, stream=stream)
            return
        kf.kf_decode_step(i.q, i.k_new, i.v_new, i.k_cache, i.v_cache, i.block_tables, i.ctx_before,
                          self.max_ctx, self.w.scale, self.num_splits, self.workspace, self.out,
                          lse_out=self.lse, stream=stream)

    def run(self, stream=None) -> None:
        if self.fused:
            self.step_fused(stream)
            return
        if self.with_append:
            self.append(stream)
        self.attention(stream)
        self.merge(stream)

    @property
    def launches_per_step(self) -> int:
        if self.fused:
            return 1
        return int(self.with_append) + len(self.views) + 1
