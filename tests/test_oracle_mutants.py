"""Planted mistakes: each mutation of the oracle's source must fail a pin.

The mutation is applied to a copy of the C file, compiled to a temporary
library and loaded beside the real one; the committed oracle is untouched.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "kf_oracle.c")

MUTANTS = {
    "interleaved_head_map": ("h / G, t0, t1, j->scale", "h % j->hkv, t0, t1, j->scale"),
    "dropped_log_l": ("*lse = m + log(l);", "*lse = m;"),
    "dropped_max_in_lse": ("*lse = m + log(l);", "*lse = log(l);"),
    "missing_normalisation": ("        o[d] /= l;", "        o[d] /= 1.0;"),
    "dropped_scale": ("s[i] = scale * dot;", "s[i] = dot;"),
    "v_slot_off_by_one": ("const uint16_t *v = v_cache + cache_row(blk, t % block_size,",
                          "const uint16_t *v = v_cache + cache_row(blk, (t + 1) % block_size,"),
    "logical_block_for_k": ("const uint16_t *k = k_cache + cache_row(blk,",
                            "const uint16_t *k = k_cache + cache_row(t / block_size,"),
    "k_v_swapped": ("const uint16_t *v = v_cache + cache_row(", "const uint16_t *v = k_cache + cache_row("),
    "merge_weight_sign": ("double w = exp(li - M);", "double w = exp(M - li);"),
    "merge_unnormalised": ("        o[d] /= wsum;", "        o[d] /= 1.0;"),
    "split_short_by_one": ("int64_t hi = lo + chunk * block_size;", "int64_t hi = lo + chunk * block_size - 1;"),
    "split_per_request_chunk": ("int64_t n_max = (max_context_len + block_size - 1) / block_size;",
                                "int64_t n_max = (ctx_len + block_size - 1) / block_size;"),
    "append_slot_off_by_one": ("int64_t dst = cache_row(blk, p % block_size,",
                               "int64_t dst = cache_row(blk, (p + 1) % block_size,"),
    "bf16_widen_wrong_half": ("uint32_t u = ((uint32_t)bits) << 16;", "uint32_t u = ((uint32_t)bits) << 15;"),
    "score_sign": ("s[i] = scale * dot;", "s[i] = -scale * dot;"),
    "lse_base2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "e4m3_bias_off_by_one": ("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    "e4m3_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) == 1.0))", "if (frac >= 0.5)"),
    "e4m3_overflow_to_nan": ("    if (a >= 448.0)\n        return sign | 0x7E;", "    if (a >= 448.0)\n        return sign | 0x7F;"),
    "fp8_v_scale_dropped": ("o[d] += p * (kfo_e4m3_to_double(v[d]) * v_scale);", "o[d] += p * kfo_e4m3_to_double(v[d]);"),
    "fp8_k_scale_is_v_scale": ("(double)k_scale[kvh],", "(double)v_scale[kvh],"),
    "chunk_causal_off_by_one": ("int64_t limit = causal ? L - C + j + 1 : L;", "int64_t limit = causal ? L - C + j : L;"),
    "chunk_causal_reversed": ("int64_t limit = causal ? L - C + j + 1 : L;", "int64_t limit = causal ? L - j : L;"),
    "chunk_split_not_clipped": ("                    if (t1 > limit)\n                        t1 = limit;",
                                "                    (void)limit;"),
    "chunk_kv_head_interleaved": ("num_kv_heads, head_dim, h / G, t0, t1, scale,",
                                  "num_kv_heads, head_dim, h % num_kv_heads, t0, t1, scale,"),
    "chunk_ignores_q_start": ("int64_t n = q_start[b] + j;", "int64_t n = j;"),
    "chunk_limit_from_max_context": ("int64_t limit = causal ? L - C + j + 1 : L;",
                                     "int64_t limit = causal ? max_context_len - C + j + 1 : L;"),
    "merge_max_is_first": ("        if (li > M)\n            M = li;", "        if (i == 0)\n            M = li;"),
    "split_chunk_floor": ("int64_t chunk = (n_max + num_splits - 1) / num_splits;",
                          "int64_t chunk = n_max / num_splits;"),
    "e4m3_subnormal_scale": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3_nan_code_ignored": ("    if (e == 15 && m == 7)\n        return NAN;", "    if (e == 15 && m == 7 && sign)\n        return NAN;"),
    "fp8_append_multiplies": ("float kq = (float)kfo_bf16_to_double(k_new[src + d]) / k_scale[h];",
                              "float kq = (float)kfo_bf16_to_double(k_new[src + d]) * k_scale[h];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    old = old.replace("\\n", "\n")
    new = new.replace("\\n", "\n")
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    mutated = src.replace(old, new)
    path = str(tmp_path / ("m_%s.c" % name))
    with open(path, "w") as f:
        f.write(mutated)
    so = oracle.build(force=True, src=path, out=str(tmp_path / ("libm_%s.so" % name)))
    lib = oracle.load(so)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, "no pin caught mutation " + name
