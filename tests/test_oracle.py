"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, lib):
    pin(lib)


def test_rows_subset_matches_full(lib):
    import numpy as np
    from oracle_pins import _small, _arrays
    w, inp = _small(batch=3, hq=4, hkv=2, d=16, bs=4, lengths=(5, 30, 12))
    q, k, v, bt, ctx = _arrays(inp)
    o, lse = oracle.decode_partials(q, k, v, bt, ctx, w.scale, 3, max_context_len=40, threads=3)
    rows = [(2, 1), (0, 3), (1, 0)]
    o2, lse2 = oracle.decode_partials(q, k, v, bt, ctx, w.scale, 3, max_context_len=40, rows=rows)
    for b, h in rows:
        assert np.array_equal(o[:, b, h], o2[:, b, h]) and np.array_equal(lse[:, b, h], lse2[:, b, h])
    mo, ml = oracle.merge_partials(o, lse)
    mo2, ml2 = oracle.merge_partials(o2, lse2, rows=rows)
    for b, h in rows:
        assert np.array_equal(mo[b, h], mo2[b, h]) and ml[b, h] == ml2[b, h]


def test_rejects_bad_inputs(lib):
    import numpy as np
    from oracle_pins import _small, _arrays
    w, inp = _small(lengths=(5, 9, 16))
    q, k, v, bt, ctx = _arrays(inp)
    with pytest.raises(ValueError):       # context above max_context_len
        oracle.decode_partials(q, k, v, bt, ctx, w.scale, 2, max_context_len=int(ctx.max()) - 1)
    bad = bt.copy()
    bad[1, 0] = k.shape[0]                 # block id past the pool
    with pytest.raises(ValueError):
        oracle.decode_partials(q, k, v, bad, ctx, w.scale, 1)
