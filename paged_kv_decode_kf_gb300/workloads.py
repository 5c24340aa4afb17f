"""Seeded synthetic inputs for one paged-KV decode step.

This module is the one piece shared by the CUDA path and the CPU oracle. It
holds no attention arithmetic: only shapes, random draws and the layout of
the paged cache and its block tables.

Layout (the paged block layout of "Disaggregated Inference Architecture:
Paged KV-Cache Tiering, Chunked Prefill, and Asynchronous Overlap",
ultrainstinct.tech, section "Physical Memory Block Layout": a block holds
block_size tokens x H_kv x D elements, and a block table maps a sequence's
logical block i to a physical frame):

    k_cache, v_cache : bf16 [num_blocks, block_size, num_kv_heads, head_dim]
    block_tables     : int32 [batch, max_blocks]; entry (b, i) is the physical
                       block holding tokens [i*bs, (i+1)*bs) of request b;
                       unused entries are -1
    q                : bf16 [batch, num_q_heads, head_dim]
    k_new, v_new     : bf16 [batch, num_kv_heads, head_dim]
    ctx_before       : int32 [batch], tokens already cached (pre-append)
    ctx_after        : ctx_before + 1, the range attention covers after the
                       step's append (KernelFlume, academ.us/article/2606.29207,
                       section 3.2: the tail node appends K_new/V_new, then
                       attends over the updated range)

Recipe (every draw seeded, in this order): context lengths and the physical
block permutation from numpy PCG64(seed); then q, k_cache, v_cache, k_new,
v_new from a torch generator seeded with the same seed, as N(0,1) rounded to
bf16. Every pool slot, used or not, is filled. Physical ids are a random
permutation of [0, num_blocks) assigned to (request, logical block) in order.

A "shards" workload also carries, per shard, a block table holding a
contiguous slice of each request's logical blocks, the shard-local context
lengths, and a tail table (the shard holding each request's newest token),
mirroring KernelFlume's token-range partitions over attention nodes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch


# ----------------------------------------------------------------------------
# Context-length distributions (pre-append lengths)
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Fixed:
    values: tuple

    def draw(self, rng: np.random.Generator, batch: int, block_size: int) -> np.ndarray:
        assert len(self.values) == batch
        return np.asarray(self.values, dtype=np.int64)


@dataclass(frozen=True)
class Uniform:
    lo: int
    hi: int  # inclusive

    def draw(self, rng, batch, block_size):
        return rng.integers(self.lo, self.hi + 1, size=batch, dtype=np.int64)


@dataclass(frozen=True)
class LogNormal:
    """round(exp(ln(median) + sigma*z)) clipped to [lo, hi]."""
    median: float
    sigma: float
    lo: int
    hi: int

    def draw(self, rng, batch, block_size):
        z = rng.standard_normal(batch)
        v = np.rint(np.exp(math.log(self.median) + self.sigma * z))
        return np.clip(v, self.lo, self.hi).astype(np.int64)


@dataclass(frozen=True)
class Mixture:
    """Exact request counts per uniform band, shuffled. The first
    `fresh_block_first` requests are rounded down to a multiple of the block
    size, so that the step's append opens a freshly allocated block."""
    bands: tuple  # ((count, lo, hi), ...)
    fresh_block_first: int = 0

    def draw(self, rng, batch, block_size):
        parts = [rng.integers(lo, hi + 1, size=n, dtype=np.int64) for (n, lo, hi) in self.bands]
        v = np.concatenate(parts)
        assert v.shape[0] == batch
        v = v[rng.permutation(batch)]
        k = self.fresh_block_first
        v[:k] = (v[:k] // block_size) * block_size
        v[:k] = np.maximum(v[:k], block_size)
        return v


# ----------------------------------------------------------------------------
# Workload specs
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    lengths: object
    seed: int
    spare_blocks: int = 0          # physical blocks beyond those the tables use
    num_splits: tuple = (0,)       # 0 = library's choice
    shards: int = 0                # >0: KV spread over this many token-range shards
    description: str = ""
    kv_dtype: str = "bf16"         # "bf16" or "fp8" (E4M3 codes with per-KV-head scales)
    shared_prefix: int = 0         # >0: every request starts with these many shared tokens
                                   # (whole blocks); `lengths` then draws the private suffixes
    chunk: int = 0                 # >0: the last `chunk` cached tokens of each request are a
                                   # prefill chunk whose queries attend causally (multi-query)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token over all KV heads."""
        return 2 * self.num_kv_heads * self.head_dim * (1 if self.kv_dtype == "fp8" else 2)


CONFIGS = {
    "tiny": Workload(
        name="tiny", batch=2, num_q_heads=2, num_kv_heads=1, head_dim=64, block_size=16,
        lengths=Fixed((37, 100)), seed=1000, spare_blocks=6, num_splits=(1, 3),
        description="batch 2, 2 q heads / 1 kv head, D 64, bs 16, ctx {37,100} before the "
                    "append, 16 physical blocks, splits 1 and 3"),
    "llama8b": Workload(
        name="llama8b", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        lengths=Uniform(3584, 4096), seed=1001,
        description="Llama-3.1-8B-shaped decode layer: batch 64, 32/8 heads, D 128, bs 16, "
                    "ctx U[3584,4096]"),
    "longctx": Workload(
        name="longctx", batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        lengths=LogNormal(81920.0, 0.5, 8192, 262144), seed=1002,
        description="long-context agentic decode: batch 16, 32/8 heads, D 128, bs 16, ctx "
                    "log-normal median 80K (sigma 0.5) clipped to [8K,256K]"),
    "shard4": Workload(
        name="shard4", batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        lengths=Uniform(16384, 65536), seed=1003, shards=4,
        description="KV over 4 token-range shards: batch 32, 32/8 heads, D 128, bs 16, ctx "
                    "U[16K,64K], one partial per shard then a merge"),
    "ragged": Workload(
        name="ragged", batch=256, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
        lengths=Mixture(((179, 1024, 8192), (64, 8192, 65536), (13, 65536, 131072)),
                        fresh_block_first=8), seed=1004,
        description="ragged continuous batch with append: batch 256, 32/8 heads, D 128, bs 32, "
                    "179/64/13 requests from U[1K,8K]/U[8K,64K]/U[64K,128K]"),
}

# Shared-prefix batch for cascade attention (the pages' cascade example: many
# requests behind one long common prompt), not one of the five configs.
CONFIGS["cascade"] = Workload(
    name="cascade", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
    lengths=Uniform(64, 2048), seed=1005, shared_prefix=16384,
    description="shared-prefix batch: 64 requests behind one 16K-token prefix, private suffixes "
                "U[64,2048], 32/8 heads, D 128, bs 16")

# Chunked prefill (multi-query, causal): each request's newest `chunk` tokens are
# in the cache and their queries attend to the paged history and causally to
# the chunk, not one of the five configs.
CONFIGS["specverify"] = Workload(
    name="specverify", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
    lengths=Uniform(3584, 4096), seed=1007, chunk=4,
    description="speculative verify: the llama8b batch (64 requests, U[3.5K,4K] cached tokens, "
                "32/8 heads, D 128, bs 16) checking 4 draft tokens each, causally")

CONFIGS["chunk"] = Workload(
    name="chunk", batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
    lengths=Uniform(4096, 12288), seed=1006, chunk=1024,
    description="chunked prefill: 4 requests, each a causal 1024-token chunk at the end of "
                "U[4K,12K] cached tokens, 32/8 heads, D 128, bs 16")

CONFIG_ORDER = ("tiny", "llama8b", "longctx", "shard4", "ragged")


def scaled(w: Workload, *, batch: Optional[int] = None, lengths=None, name=None,
           seed: Optional[int] = None, spare_blocks: Optional[int] = None,
           kv_dtype: Optional[str] = None, description: Optional[str] = None) -> Workload:
    """The same heads/dims/block size as `w` with another batch or length mix
    (used for oracle-sized parity cases)."""
    return Workload(
        name=name or (w.name + "-small"), batch=batch if batch is not None else w.batch,
        num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        block_size=w.block_size, lengths=lengths if lengths is not None else w.lengths,
        seed=seed if seed is not None else w.seed + 7919,
        spare_blocks=w.spare_blocks if spare_blocks is None else spare_blocks,
        num_splits=w.num_splits, shards=w.shards,
        description=w.description if description is None else description,
        kv_dtype=kv_dtype or w.kv_dtype, shared_prefix=w.shared_prefix, chunk=w.chunk)


def with_kv_dtype(w: Workload, kv_dtype: str) -> Workload:
    """`w` with another cache element type (same lengths, tables and seed)."""
    return Workload(name=w.name, batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                    head_dim=w.head_dim, block_size=w.block_size, lengths=w.lengths, seed=w.seed,
                    spare_blocks=w.spare_blocks, num_splits=w.num_splits, shards=w.shards,
                    description=w.description + ("" if kv_dtype == "bf16" else ", FP8 E4M3 KV cache"),
                    kv_dtype=kv_dtype, shared_prefix=w.shared_prefix, chunk=w.chunk)


def fp8_scales(num_kv_heads: int):
    """Per-KV-head K and V scales of the FP8 workloads: powers of two 2^-(4..6),
    so N(0,1) data sits well inside E4M3's +-448 after division."""
    k = np.array([2.0 ** -(4 + h % 3) for h in range(num_kv_heads)], dtype=np.float32)
    v = np.array([2.0 ** -(4 + (h + 1) % 3) for h in range(num_kv_heads)], dtype=np.float32)
    return k, v


# ----------------------------------------------------------------------------
# Materialised inputs
# ----------------------------------------------------------------------------

@dataclass
class ShardView:
    block_tables: torch.Tensor   # int32 [B, max_shard_blocks]
    ctx_after: torch.Tensor      # int32 [B], shard-local tokens after the append
    first_block: np.ndarray      # int64 [B], first logical block of the shard


@dataclass
class DecodeInputs:
    workload: Workload
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    block_tables: torch.Tensor
    # ... FP8 caches: k_cache/v_cache are uint8 E4M3 codes, with these scales
    k_scale: Optional[torch.Tensor] = field(default=None, kw_only=True)
    v_scale: Optional[torch.Tensor] = field(default=None, kw_only=True)
    # ... shared-prefix batches: the prefix's table and each request's suffix
    prefix_table: Optional[torch.Tensor] = field(default=None, kw_only=True)
    suffix_tables: Optional[torch.Tensor] = field(default=None, kw_only=True)
    suffix_ctx_before: Optional[torch.Tensor] = field(default=None, kw_only=True)
    suffix_ctx_after: Optional[torch.Tensor] = field(default=None, kw_only=True)
    # ... chunked prefill: the chunk queries [B * chunk, Hq, D] and their row starts [B + 1]
    q_chunk: Optional[torch.Tensor] = field(default=None, kw_only=True)
    q_start: Optional[torch.Tensor] = field(default=None, kw_only=True)
    ctx_before: torch.Tensor
    ctx_after: torch.Tensor
    num_blocks: int
    shards: list = field(default_factory=list)
    tail_tables: Optional[torch.Tensor] = None      # shard table holding each request's tail
    tail_ctx_before: Optional[torch.Tensor] = None  # tail-local pre-append length

    @property
    def scale(self) -> float:
        return self.workload.scale

    @property
    def max_ctx_after(self) -> int:
        return int(self.ctx_after.max().item()) if self.ctx_after.numel() else 0

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one attention pass reads: sum_b L_b * 2*Hkv*D*2."""
        return int(self.ctx_after.to(torch.int64).sum().item()) * self.workload.kv_bytes_per_token()

    def to(self, device) -> "DecodeInputs":
        mv = lambda t: None if t is None else t.to(device)
        return DecodeInputs(
            workload=self.workload, q=mv(self.q), k_cache=mv(self.k_cache), v_cache=mv(self.v_cache),
            k_new=mv(self.k_new), v_new=mv(self.v_new), block_tables=mv(self.block_tables),
            ctx_before=mv(self.ctx_before), ctx_after=mv(self.ctx_after), num_blocks=self.num_blocks,
            shards=[ShardView(mv(s.block_tables), mv(s.ctx_after), s.first_block) for s in self.shards],
            tail_tables=mv(self.tail_tables), tail_ctx_before=mv(self.tail_ctx_before),
            k_scale=mv(self.k_scale), v_scale=mv(self.v_scale), prefix_table=mv(self.prefix_table),
            suffix_tables=mv(self.suffix_tables), suffix_ctx_before=mv(self.suffix_ctx_before),
            suffix_ctx_after=mv(self.suffix_ctx_after))


def _bf16_normal(shape, gen: torch.Generator, device) -> torch.Tensor:
    if torch.device(device).type == "cpu":
        return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.bfloat16)


@dataclass
class Layout:
    """Host-side plan of one workload: lengths, tables and shard slices."""
    ctx_before: np.ndarray        # int64 [B]
    ctx_after: np.ndarray         # int64 [B]
    n_blocks: np.ndarray          # int64 [B], blocks each table holds (post-append)
    block_tables: np.ndarray      # int32 [B, max_blocks]
    num_blocks: int               # physical pool size
    shard_tables: list = field(default_factory=list)   # int32 [B, cap] per shard
    shard_ctx_after: list = field(default_factory=list)  # int32 [B] per shard
    shard_first_block: list = field(default_factory=list)  # int64 [B] per shard
    tail_tables: Optional[np.ndarray] = None
    tail_ctx_before: Optional[np.ndarray] = None
    prefix_table: Optional[np.ndarray] = None       # int32 [1, prefix blocks]
    suffix_tables: Optional[np.ndarray] = None      # int32 [B, max suffix blocks]
    suffix_ctx_before: Optional[np.ndarray] = None  # int64 [B]


def plan_layout(w: Workload, lengths: Optional[Sequence[int]] = None) -> Layout:
    """Draw the context lengths and the physical block permutation of `w`
    (the first draws of its seed) and build the block tables."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    B, bs = w.batch, w.block_size
    if lengths is None:
        L0 = w.lengths.draw(rng, B, bs)
    else:
        L0 = np.asarray(lengths, dtype=np.int64)
        assert L0.shape == (B,)
    if w.shared_prefix:
        return _plan_shared_prefix(w, L0, rng)
    L1 = L0 + 1
    n_blocks = (L1 + bs - 1) // bs
    max_blocks = int(n_blocks.max()) if B else 1
    NB = int(n_blocks.sum()) + w.spare_blocks
    perm = rng.permutation(NB)
    bt = np.full((B, max(max_blocks, 1)), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        nb = int(n_blocks[b])
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    lay = Layout(ctx_before=L0, ctx_after=L1, n_blocks=n_blocks, block_tables=bt, num_blocks=NB)
    if w.shards > 0:
        _plan_shards(lay, w.shards, bs)
    return lay


def _plan_shared_prefix(w: Workload, suffix0: np.ndarray, rng) -> Layout:
    """Every request's table starts with the same prefix blocks (the first
    physical ids drawn), followed by its own suffix blocks."""
    B, bs, P = w.batch, w.block_size, w.shared_prefix
    assert P % bs == 0, "the shared prefix must be whole blocks"
    NP = P // bs
    L0 = suffix0 + P
    L1 = L0 + 1
    n_suffix = (suffix0 + 1 + bs - 1) // bs
    NB = NP + int(n_suffix.sum()) + w.spare_blocks
    perm = rng.permutation(NB)
    prefix = perm[:NP].astype(np.int32)
    n_blocks = NP + n_suffix
    bt = np.full((B, int(n_blocks.max())), -1, dtype=np.int32)
    st = np.full((B, max(int(n_suffix.max()), 1)), -1, dtype=np.int32)
    pos = NP
    for b in range(B):
        ns = int(n_suffix[b])
        bt[b, :NP] = prefix
        bt[b, NP:NP + ns] = perm[pos:pos + ns]
        st[b, :ns] = perm[pos:pos + ns]
        pos += ns
    return Layout(ctx_before=L0, ctx_after=L1, n_blocks=n_blocks, block_tables=bt, num_blocks=NB,
                  prefix_table=prefix[None, :].copy(), suffix_tables=st, suffix_ctx_before=suffix0)


def _plan_shards(lay: Layout, n_shards: int, bs: int) -> None:
    """Cut each request's logical blocks into `n_shards` contiguous slices of
    ceil(n_b / n_shards) blocks (trailing slices may be short or empty). The
    slice holding position ctx_before[b] (the new token) is the tail."""
    bt, L0, L1, n_blocks = lay.block_tables, lay.ctx_before, lay.ctx_after, lay.n_blocks
    B = bt.shape[0]
    per = (n_blocks + n_shards - 1) // n_shards
    cap = max(int(per.max()) if B else 1, 1)
    tail_tab = np.full((B, cap), -1, dtype=np.int32)
    tail_before = np.zeros(B, dtype=np.int32)
    for s in range(n_shards):
        tab = np.full((B, cap), -1, dtype=np.int32)
        first = np.minimum(s * per, n_blocks)
        last = np.minimum((s + 1) * per, n_blocks)
        ctx = np.zeros(B, dtype=np.int32)
        for b in range(B):
            nb = int(last[b] - first[b])
            if nb > 0:
                tab[b, :nb] = bt[b, first[b]:last[b]]
            lo_tok = int(first[b]) * bs
            ctx[b] = int(np.clip(L1[b] - lo_tok, 0, nb * bs))
            if nb > 0 and lo_tok <= L0[b] < lo_tok + nb * bs:
                tail_tab[b, :] = tab[b, :]
                tail_before[b] = L0[b] - lo_tok
        lay.shard_tables.append(tab)
        lay.shard_ctx_after.append(ctx)
        lay.shard_first_block.append(first.astype(np.int64))
    lay.tail_tables = tail_tab
    lay.tail_ctx_before = tail_before


def make_inputs(w: Workload, device="cpu", lengths: Optional[Sequence[int]] = None) -> DecodeInputs:
    """Materialise the seeded inputs of workload `w` on `device`.

    `lengths` overrides the drawn pre-append context lengths (tests)."""
    lay = plan_layout(w, lengths)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    B, H, Hkv, D, bs, NB = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, lay.num_blocks
    q = _bf16_normal((B, H, D), gen, dev)
    k_cache = _bf16_normal((NB, bs, Hkv, D), gen, dev)
    v_cache = _bf16_normal((NB, bs, Hkv, D), gen, dev)
    k_new = _bf16_normal((B, Hkv, D), gen, dev)
    v_new = _bf16_normal((B, Hkv, D), gen, dev)
    k_scale = v_scale = None
    if w.kv_dtype == "fp8":
        # E4M3 codes of the same N(0,1) draws divided by the per-head scales,
        # converted by torch's float8_e4m3fn cast
        ks, vs = fp8_scales(Hkv)
        k_scale = torch.from_numpy(ks).to(dev)
        v_scale = torch.from_numpy(vs).to(dev)
        k_cache = (k_cache.float() / k_scale.view(1, 1, Hkv, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
        v_cache = (v_cache.float() / v_scale.view(1, 1, Hkv, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    inp = DecodeInputs(
        workload=w, q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        block_tables=i32(lay.block_tables), ctx_before=i32(lay.ctx_before),
        ctx_after=i32(lay.ctx_after), num_blocks=NB, k_scale=k_scale, v_scale=v_scale)
    for tab, ctx, first in zip(lay.shard_tables, lay.shard_ctx_after, lay.shard_first_block):
        inp.shards.append(ShardView(i32(tab), i32(ctx), first))
    if lay.tail_tables is not None:
        inp.tail_tables = i32(lay.tail_tables)
        inp.tail_ctx_before = i32(lay.tail_ctx_before)
    if lay.prefix_table is not None:
        inp.prefix_table = i32(lay.prefix_table)
        inp.suffix_tables = i32(lay.suffix_tables)
        inp.suffix_ctx_before = i32(lay.suffix_ctx_before)
        inp.suffix_ctx_after = i32(lay.suffix_ctx_before + 1)
    if w.chunk:
        # drawn after everything else, so the other inputs do not depend on it;
        # the chunk is the last `chunk` of each request's ctx_after tokens
        assert int(lay.ctx_after.min()) >= w.chunk, "every context must hold the chunk"
        inp.q_chunk = _bf16_normal((B * w.chunk, H, D), gen, dev)
        inp.q_start = i32(np.arange(B + 1) * w.chunk)
    return inp


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The bf16 tensor's bit patterns as a host uint16 array (no rounding)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
