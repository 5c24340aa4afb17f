"""Host-side input recipe: lengths, tables, shard slices (CPU only)."""
import numpy as np
import pytest
import torch

from paged_kv_decode_kf_gb300 import workloads as wl


@pytest.mark.parametrize("name", wl.CONFIG_ORDER)
def test_layout_invariants(name):
    w = wl.CONFIGS[name]
    lay = wl.plan_layout(w)
    B, bs = w.batch, w.block_size
    assert np.array_equal(lay.ctx_after, lay.ctx_before + 1)
    assert np.array_equal(lay.n_blocks, -(-lay.ctx_after // bs))
    used = np.concatenate([lay.block_tables[b, :lay.n_blocks[b]] for b in range(B)])
    assert len(np.unique(used)) == used.size == int(lay.n_blocks.sum())     # each frame once
    assert used.min() >= 0 and used.max() < lay.num_blocks
    assert lay.num_blocks == used.size + w.spare_blocks
    for b in range(B):
        assert np.all(lay.block_tables[b, lay.n_blocks[b]:] == -1)


def test_tiny_config_matches_spec():
    w = wl.CONFIGS["tiny"]
    lay = wl.plan_layout(w)
    assert list(lay.ctx_before) == [37, 100] and lay.num_blocks == 16
    assert list(lay.n_blocks) == [3, 7]                   # 38 and 101 tokens after the append


def test_length_distributions():
    lay = wl.plan_layout(wl.CONFIGS["llama8b"])
    assert lay.ctx_before.min() >= 3584 and lay.ctx_before.max() <= 4096
    lay = wl.plan_layout(wl.CONFIGS["longctx"])
    assert lay.ctx_before.min() >= 8192 and lay.ctx_before.max() <= 262144
    lay = wl.plan_layout(wl.CONFIGS["shard4"])
    assert lay.ctx_before.min() >= 16384 and lay.ctx_before.max() <= 65536
    w = wl.CONFIGS["ragged"]
    lay = wl.plan_layout(w)
    L = lay.ctx_before
    assert np.all(L[:8] % 32 == 0)                          # append opens a fresh block
    assert np.all(L[8:] >= 1024) and L.max() <= 131072
    assert (L >= 65536).sum() >= 13 - 0 and (L <= 8192).sum() >= 179 - 8


def test_seeded_reproducible():
    a = wl.plan_layout(wl.CONFIGS["longctx"])
    b = wl.plan_layout(wl.CONFIGS["longctx"])
    assert np.array_equal(a.block_tables, b.block_tables) and np.array_equal(a.ctx_before, b.ctx_before)
    w = wl.scaled(wl.CONFIGS["llama8b"], batch=2, lengths=wl.Fixed((40, 70)))
    x, y = wl.make_inputs(w), wl.make_inputs(w)
    assert all(np.array_equal(wl.bf16_bits(getattr(x, f)), wl.bf16_bits(getattr(y, f)))
               for f in ("q", "k_cache", "v_cache", "k_new", "v_new"))


@pytest.mark.parametrize("lengths", [(16383, 20000, 65536, 3, 0, 15, 16, 17)])
def test_shard_slices(lengths):
    w = wl.scaled(wl.CONFIGS["shard4"], batch=len(lengths), lengths=wl.Fixed(lengths))
    lay = wl.plan_layout(w)
    bs = w.block_size
    for b in range(w.batch):
        pieces, total = [], 0
        for s in range(w.shards):
            tab, ctx = lay.shard_tables[s][b], int(lay.shard_ctx_after[s][b])
            nb = -(-ctx // bs)
            pieces.append(tab[:nb])
            total += ctx
            assert np.all(tab[nb:] == -1)
        assert total == lay.ctx_after[b]
        assert np.array_equal(np.concatenate(pieces), lay.block_tables[b, :lay.n_blocks[b]])
        # the tail table holds the block of position ctx_before[b] at tail-local position
        p = int(lay.tail_ctx_before[b])
        g = int(lay.ctx_before[b])
        assert lay.tail_tables[b, p // bs] == lay.block_tables[b, g // bs] and p % bs == g % bs


def test_chunk_inputs():
    """Chunked prefill: B * chunk query rows drawn after every other input (the
    cache, q and new rows are those of the same workload without a chunk), row
    starts at multiples of the chunk, every context at least one chunk long."""
    w = wl.scaled(wl.CONFIGS["chunk"], batch=3, lengths=wl.Fixed((1100, 2047, 5000)))
    i = wl.make_inputs(w, "cpu")
    assert tuple(i.q_chunk.shape) == (3 * w.chunk, w.num_q_heads, w.head_dim)
    assert i.q_start.tolist() == [0, w.chunk, 2 * w.chunk, 3 * w.chunk]
    assert int(i.ctx_after.min()) >= w.chunk
    import dataclasses
    plain = wl.make_inputs(dataclasses.replace(w, chunk=0), "cpu")
    assert plain.q_chunk is None
    assert torch.equal(plain.k_cache, i.k_cache) and torch.equal(plain.q, i.q)
    lay = wl.plan_layout(wl.CONFIGS["chunk"])
    assert int(lay.ctx_after.min()) >= wl.CONFIGS["chunk"].chunk


def test_specverify_inputs():
    """Speculative verify: the llama8b batch (same heads, dims, block size and
    length range) with 4 causal draft queries per request, row starts at
    multiples of 4."""
    w = wl.CONFIGS["specverify"]
    base = wl.CONFIGS["llama8b"]
    assert (w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size) == \
        (base.batch, base.num_q_heads, base.num_kv_heads, base.head_dim, base.block_size)
    assert w.chunk == 4 and (w.lengths.lo, w.lengths.hi) == (base.lengths.lo, base.lengths.hi)
    small = wl.scaled(w, batch=3, lengths=wl.Fixed((10, 3000, 4)))
    i = wl.make_inputs(small, "cpu")
    assert tuple(i.q_chunk.shape) == (3 * 4, w.num_q_heads, w.head_dim)
    assert i.q_start.tolist() == [0, 4, 8, 12]
    assert int(i.ctx_after.min()) >= w.chunk
