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
        dev = inp.k_cache.device
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


class CascadeStep:
    """A decode step for requests behind one shared prefix (cascade attention,
    "What FlashInfer brings: JIT and cascade attention", blog.lo0.es): the
    append goes through each request's suffix table; one non-causal
    multi-query pass attends the prefix once for all B queries; decode
    attention covers each request's suffix; one LSE merge combines the two
    sets of partials. With fused_suffix (the default) that is three launches.
    concurrent (the default): the prefix pass on the caller's stream and
    kf_decode_step (append + suffixes + the merge of their own splits, one
    (o, lse) slot per request) on a second stream at the same time -- the
    first is bound by the tensor pipe, the second by HBM -- then one
    kf_merge_partials of the prefix pass's slots with the suffix slot. Not
    concurrent: the prefix pass, a merge of its slots into one prefix partial,
    and kf_decode_step_merge_partials (append + suffixes + the final merge)."""

    def __init__(self, inp: DecodeInputs, prefix_splits: Optional[int] = None,
                 suffix_splits: Optional[int] = None, out_dtype=torch.float32, fused_suffix: bool = True,
                 concurrent: bool = True):
        w = inp.workload
        assert w.shared_prefix and inp.prefix_table is not None
        self.inp, self.w = inp, w
        B, Hq = w.batch, w.num_q_heads
        dev = inp.q.device
        self.P = int(w.shared_prefix)
        self.max_suffix = int(inp.suffix_ctx_after.max().item())
        # prefix pass: one wave of CTAs (KV heads x query tiles x splits) for the
        # kernel the library picks for B x G rows per KV head: 256 rows and one
        # CTA per SM (tcgen05, two tiles), else 128 rows and two per SM (tcgen05,
        # one tile)
        if prefix_splits is None:
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            rows = B * w.group
            rows_per_cta, per_sm = (256, 1) if rows > 128 else (128, 2)
            units = w.num_kv_heads * max(1, -(-rows // rows_per_cta))
            prefix_splits = max(1, min(self.P // w.block_size, -(-per_sm * sms // units)))
        if suffix_splits is None:
            suffix_splits = kf.kf_choose_num_splits(B, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                                    self.max_suffix,
                                                    inp.suffix_ctx_after.cpu().numpy().astype(np.int32))
        self.Sp, self.Ss = int(prefix_splits), int(suffix_splits)
        self.q_start = torch.tensor([0, B], dtype=torch.int32, device=dev)
        self.prefix_len = torch.tensor([self.P], dtype=torch.int32, device=dev)
        self.concurrent = bool(concurrent) and bool(fused_suffix)
        # slots: the prefix pass's Sp, then the suffix splits (four calls) or
        # the suffix step's one merged slot (concurrent)
        S = self.Sp + (1 if self.concurrent else self.Ss)
        self.out_partial = torch.empty((S, B, Hq, w.head_dim), dtype=torch.float32, device=dev)
        self.lse_partial = torch.empty((S, B, Hq), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, Hq, w.head_dim), dtype=out_dtype, device=dev)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        self.fused = False
        self.with_append = True
        # fused_suffix: append + suffix attention + merge with the prefix partials
        # in one kf_decode_step_merge_partials launch (two launches per step);
        # otherwise four calls (append, prefix, suffix, merge)
        self.fused_suffix = bool(fused_suffix)
        self.workspace = kf.make_workspace(B, Hq, w.num_kv_heads, w.head_dim, self.Ss, dev) if fused_suffix else None
        # the fused suffix step merges one pre-merged prefix partial instead of
        # the prefix pass's Sp slots: one small kf_merge_partials launch (Sp
        # rows in, one out) costs less than the Sp-slot merge in the suffix
        # step's tail (measured on the cascade workload: 4.5 us vs 8.8 us)
        self.prefix_o = torch.empty((1, B, Hq, w.head_dim), dtype=torch.float32, device=dev)
        self.prefix_lse = torch.empty((1, B, Hq), dtype=torch.float32, device=dev)
        self.side = torch.cuda.Stream(device=dev) if self.concurrent else None

    def append(self, stream=None) -> None:
        i = self.inp
        kf.kf_append_kv(i.k_new, i.v_new, i.k_cache, i.v_cache, i.suffix_tables, i.suffix_ctx_before, stream)

    def prefix(self, stream=None) -> None:
        """The shared prefix, attended once by every request's query."""
        i, w, Sp = self.inp, self.w, self.Sp
        kf.kf_paged_multiquery_attention(i.q, self.q_start, i.k_cache, i.v_cache, i.prefix_table, self.prefix_len,
                                         False, self.P, w.batch, w.scale, Sp, self.out_partial[:Sp],
                                         self.lse_partial[:Sp], stream)

    def suffix(self, stream=None) -> None:
        """Each request's own blocks after the prefix."""
        i, w, Sp = self.inp, self.w, self.Sp
        kf.kf_paged_decode_attention(i.q, i.k_cache, i.v_cache, i.suffix_tables, i.suffix_ctx_after,
                                     self.max_suffix, w.scale, self.Ss, self.out_partial[Sp:],
                                     self.lse_partial[Sp:], stream)

    def attention(self, stream=None) -> None:
        self.prefix(stream)
        self.suffix(stream)

    def merge(self, stream=None) -> None:
        kf.kf_merge_partials(self.out_partial, self.lse_partial, self.out, lse_out=self.lse, stream=stream)

    def prefix_merge(self, stream=None) -> None:
        """The prefix pass's Sp partial slots merged into one (o, lse) slot."""
        Sp = self.Sp
        kf.kf_merge_partials(self.out_partial[:Sp], self.lse_partial[:Sp], self.prefix_o[0],
                             lse_out=self.prefix_lse[0], stream=stream)

    def suffix_step(self, stream=None) -> None:
        """Append, suffix attention and the merge with the merged prefix partial, one launch."""
        i, w = self.inp, self.w
        kf.kf_decode_step_merge_partials(i.q, i.k_new, i.v_new, i.k_cache, i.v_cache, i.suffix_tables,
                                         i.suffix_ctx_before, self.max_suffix, w.scale, self.Ss,
                                         self.prefix_o, self.prefix_lse, self.workspace,
                                         out=self.out, lse_out=self.lse, stream=stream)

    def suffix_slot(self, stream=None) -> None:
        """Append, suffix attention and the merge of the suffix splits into the
        suffix slot (fp32 o and lse after the prefix pass's slots), one launch."""
        i, w, Sp = self.inp, self.w, self.Sp
        kf.kf_decode_step(i.q, i.k_new, i.v_new, i.k_cache, i.v_cache, i.suffix_tables, i.suffix_ctx_before,
                          self.max_suffix, w.scale, self.Ss, self.workspace, out=self.out_partial[Sp],
                          lse_out=self.lse_partial[Sp], stream=stream)

    def final_merge(self, stream=None) -> None:
        """The prefix pass's slots and the suffix slot merged into the output."""
        kf.kf_merge_partials(self.out_partial, self.lse_partial, self.out, lse_out=self.lse, stream=stream)

    def run(self, stream=None) -> None:
        if self.concurrent and (stream is None or isinstance(stream, torch.cuda.Stream)):
            # fork: the suffix step on the second stream, the prefix pass here;
            # join before the merge (both are captured as graph branches)
            main = stream if stream is not None else torch.cuda.current_stream()
            self.side.wait_stream(main)
            self.suffix_slot(self.side)
            self.prefix(main)
            main.wait_stream(self.side)
            self.final_merge(main)
            return
        if self.concurrent:
            self.prefix(stream)
            self.suffix_slot(stream)
            self.final_merge(stream)
            return
        if self.fused_suffix:
            self.prefix(stream)
            self.prefix_merge(stream)
            self.suffix_step(stream)
            return
        self.append(stream)
        self.attention(stream)
        self.merge(stream)

    @property
    def launches_per_step(self) -> int:
        return 3 if self.fused_suffix else 4

    @property
    def num_splits(self) -> int:
        return self.Sp + self.Ss

    @property
    def views(self):
        return [None, None]

    def prefix_flops(self) -> float:
        """Algorithmic FLOPs of the prefix pass: 4 D per (token, query row)."""
        w = self.w
        return 4.0 * w.head_dim * w.num_q_heads * w.batch * self.P

    def suffix_kv_bytes(self) -> int:
        return int(self.inp.suffix_ctx_after.to(torch.int64).sum().item()) * self.w.kv_bytes_per_token()

    def unique_kv_bytes(self) -> int:
        """KV bytes the cascade step must read: the prefix once, each suffix once."""
        w = self.w
        tok = self.P + int(self.inp.suffix_ctx_after.to(torch.int64).sum().item())
        return tok * w.kv_bytes_per_token()



class ChunkStep:
    """Chunked prefill of one attention layer: every request's newest `chunk`
    cached tokens are queries that attend to the request's paged history and
    causally to the chunk (query j of a chunk of C over L cached tokens attends
    to tokens [0, L - C + j]; "Mathematical Formulation of Chunked Attention",
    ultrainstinct.tech). One kf_paged_multiquery_attention call (the library
    picks the kernel by rows per KV head) and one kf_merge_partials; with one
    split and fp32 output the merge of a single partial is the identity (o and
    lse as they are), so the partial slot is the output and no merge runs."""

    def __init__(self, inp: DecodeInputs, num_splits: Optional[int] = None, out_dtype=torch.float32):
        w = inp.workload
        assert w.chunk and inp.q_chunk is not None
        self.inp, self.w = inp, w
        dev = inp.q_chunk.device
        self.C = int(w.chunk)
        self.N = w.batch * self.C
        self.max_ctx = int(inp.ctx_after.max().item())
        if num_splits is None:
            # about one wave of CTAs: KV heads x requests x 256-row query groups x splits
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            units = w.num_kv_heads * w.batch * max(1, -(-self.C * w.group // 256))
            num_splits = max(1, min(self.max_ctx // w.block_size, sms // units if units < sms else 1))
        self.S = int(num_splits)
        Hq, D = w.num_q_heads, w.head_dim
        self.out_partial = torch.empty((self.S, self.N, Hq, D), dtype=torch.float32, device=dev)
        self.lse_partial = torch.empty((self.S, self.N, Hq), dtype=torch.float32, device=dev)
        if self.S == 1 and out_dtype == torch.float32:
            self.out, self.lse = self.out_partial[0], self.lse_partial[0]
        else:
            self.out = torch.empty((self.N, Hq, D), dtype=out_dtype, device=dev)
            self.lse = torch.empty((self.N, Hq), dtype=torch.float32, device=dev)
        self.fused = False
        self.with_append = False

    def attention(self, stream=None) -> None:
        i, w = self.inp, self.w
        kf.kf_paged_multiquery_attention(i.q_chunk, i.q_start, i.k_cache, i.v_cache, i.block_tables, i.ctx_after,
                                         True, self.max_ctx, self.C, w.scale, self.S, self.out_partial,
                                         self.lse_partial, stream)

    @property
    def merges(self) -> bool:
        """False when the output is the single partial slot itself."""
        return not (self.out.data_ptr() == self.out_partial[0].data_ptr() and
                    self.lse.data_ptr() == self.lse_partial[0].data_ptr())

    def merge(self, stream=None) -> None:
        if self.merges:
            kf.kf_merge_partials(self.out_partial, self.lse_partial, self.out, lse_out=self.lse, stream=stream)

    def run(self, stream=None) -> None:
        self.attention(stream)
        self.merge(stream)

    @property
    def launches_per_step(self) -> int:
        return 2 if self.merges else 1

    @property
    def num_splits(self) -> int:
        return self.S

    @property
    def views(self):
        return [None]

    def flops(self) -> float:
        """Algorithmic FLOPs: 4 D per (attended token, query row); query j of a
        chunk of C over L tokens attends to L - C + j + 1 tokens."""
        w, C = self.w, self.C
        L = self.inp.ctx_after.to(torch.int64).cpu()
        tokens = int((C * (L - C) + C * (C + 1) // 2).sum())
        return 4.0 * w.head_dim * w.num_q_heads * tokens
