"""fp64 CPU oracle for split-KV paged decode attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The arithmetic lives in ``kf_oracle.c`` (plain
C, fp64), which shares nothing with the CUDA library; this module only
compiles it with gcc and marshals numpy arrays across ctypes.

bf16 tensors cross the boundary as their uint16 bit patterns and are widened
exactly inside the C code. See ``kf_oracle.c`` for what each function
computes and which passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kf_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libkf_oracle.so")
_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc into a shared library (in-tree)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _declare(lib) -> None:
    lib.kfo_bf16_to_double.restype = ctypes.c_double
    lib.kfo_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.kfo_split_range.restype = None
    lib.kfo_split_range.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_int64)]
    lib.kfo_partial.restype = ctypes.c_int
    lib.kfo_partial.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                ctypes.c_int64, ctypes.c_double, _f64p,
                                ctypes.POINTER(ctypes.c_double)]
    lib.kfo_merge.restype = None
    lib.kfo_merge.argtypes = [_f64p, ctypes.c_int64, _f64p, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_int, _f64p, ctypes.POINTER(ctypes.c_double)]
    lib.kfo_decode_partials.restype = ctypes.c_int
    lib.kfo_decode_partials.argtypes = [
        _u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64, _f64p, _f64p, ctypes.c_int]
    lib.kfo_merge_partials.restype = None
    lib.kfo_merge_partials.argtypes = [_f64p, _f64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, _f64p, _f64p]
    _u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
    _f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
    lib.kfo_e4m3_to_double.restype = ctypes.c_double
    lib.kfo_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.kfo_e4m3_from_float.restype = ctypes.c_uint8
    lib.kfo_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.kfo_decode_partials_fp8.restype = ctypes.c_int
    lib.kfo_decode_partials_fp8.argtypes = [
        _u16p, _u8p, _u8p, _f32p, _f32p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, _f64p, _f64p]
    lib.kfo_append_fp8.restype = ctypes.c_int
    lib.kfo_append_fp8.argtypes = [_u8p, _u8p, _u16p, _u16p, _f32p, _f32p, _i32p, ctypes.c_int, _i32p,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
    lib.kfo_multiquery_partials.restype = ctypes.c_int
    lib.kfo_multiquery_partials.argtypes = [
        _u16p, _i32p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
        ctypes.c_int64, _f64p, _f64p]
    lib.kfo_append.restype = ctypes.c_int
    lib.kfo_append.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64]


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; `path` loads another
    build of it (used by the planted-mistake tests)."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


# ----------------------------------------------------------------------------
# Thin wrappers
# ----------------------------------------------------------------------------

def bf16_to_f64(bits: int, lib=None) -> float:
    return (lib or load()).kfo_bf16_to_double(int(bits))


def split_range(ctx_len: int, block_size: int, num_splits: int, max_context_len: int,
                split: int, lib=None) -> Tuple[int, int]:
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    (lib or load()).kfo_split_range(ctx_len, block_size, num_splits, max_context_len, split,
                                    ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def partial(q_row, k_cache, v_cache, bt_row, block_size: int, kv_head: int,
            t_begin: int, t_end: int, scale: float, lib=None) -> Tuple[np.ndarray, float]:
    """(o [D], lse) of one query row over tokens [t_begin, t_end)."""
    k_cache, v_cache = _u16(k_cache), _u16(v_cache)
    nb, bs, hkv, d = k_cache.shape
    assert bs == block_size
    o = np.zeros(d, dtype=np.float64)
    lse = ctypes.c_double()
    rc = (lib or load()).kfo_partial(_u16(q_row), k_cache, v_cache, _i32(bt_row), nb, bs, hkv, d,
                                     kv_head, t_begin, t_end, scale, o, ctypes.byref(lse))
    if rc != 0:
        raise ValueError("oracle partial failed (rc=%d)" % rc)
    return o, lse.value


def merge(o_parts, lse_parts, lib=None) -> Tuple[np.ndarray, float]:
    """Merge partials o_parts [S, D], lse_parts [S]."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, D = o_parts.shape
    o = np.zeros(D, dtype=np.float64)
    lse = ctypes.c_double()
    (lib or load()).kfo_merge(o_parts, D, lse_parts, 1, S, D, o, ctypes.byref(lse))
    return o, lse.value


def decode_partials(q, k_cache, v_cache, block_tables, ctx_lens, scale: float, num_splits: int,
                    max_context_len: Optional[int] = None, rows: Optional[Sequence] = None,
                    threads: Optional[int] = None, lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Partials of every split: o [S, B, Hq, D], lse [S, B, Hq] (fp64).

    With `rows` (a list of (b, h) pairs) only those rows are computed; the
    others are left as NaN."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, ctx = _i32(block_tables), _i32(ctx_lens)
    B, Hq, D = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d2 == D and bt.shape[0] == B and ctx.shape == (B,)
    if max_context_len is None:
        max_context_len = int(ctx.max()) if B else 0
    o = np.full((num_splits, B, Hq, D), np.nan, dtype=np.float64)
    lse = np.full((num_splits, B, Hq), np.nan, dtype=np.float64)
    rows_arr = None
    n_rows = 0
    if rows is not None:
        rows_arr = _i32(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n_rows = rows_arr.shape[0]
    rc = (lib or load()).kfo_decode_partials(
        q, k_cache, v_cache, bt, bt.shape[1], ctx, B, Hq, hkv, D, bs, nb, scale, num_splits,
        max_context_len, None if rows_arr is None else rows_arr.ctypes.data, n_rows, o, lse,
        threads or default_threads())
    if rc != 0:
        raise ValueError("oracle decode_partials failed (rc=%d)" % rc)
    return o, lse


def merge_partials(o_part, lse_part, rows: Optional[Sequence] = None,
                   lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Merge [S, B, Hq, D] / [S, B, Hq] partials into out [B, Hq, D], lse [B, Hq]."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    S, B, Hq, D = o_part.shape
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    lse = np.full((B, Hq), np.nan, dtype=np.float64)
    rows_arr = None
    n_rows = 0
    if rows is not None:
        rows_arr = _i32(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n_rows = rows_arr.shape[0]
    (lib or load()).kfo_merge_partials(o_part, lse_part, S, B, Hq, D,
                                       None if rows_arr is None else rows_arr.ctypes.data,
                                       n_rows, out, lse)
    return out, lse


def attention(q, k_cache, v_cache, block_tables, ctx_lens, scale: float,
              rows: Optional[Sequence] = None, threads: Optional[int] = None,
              lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Unsplit decode attention: out [B, Hq, D], lse [B, Hq] (one split over the
    whole context)."""
    o, lse = decode_partials(q, k_cache, v_cache, block_tables, ctx_lens, scale, 1,
                             rows=rows, threads=threads, lib=lib)
    return o[0], lse[0]


def append(k_cache, v_cache, k_new, v_new, block_tables, ctx_before,
           lib=None) -> Tuple[np.ndarray, np.ndarray, int]:
    """Copies of the caches with each request's new K/V row written at its
    position ctx_before[b]; also returns how many requests were skipped."""
    k2, v2 = _u16(k_cache).copy(), _u16(v_cache).copy()
    nb, bs, hkv, d = k2.shape
    bt, ctx = _i32(block_tables), _i32(ctx_before)
    skipped = (lib or load()).kfo_append(k2, v2, _u16(k_new), _u16(v_new), bt, bt.shape[1], ctx,
                                         bt.shape[0], hkv, d, bs, nb)
    return k2, v2, skipped


# ----------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# ----------------------------------------------------------------------------

def e4m3_to_f64(code: int, lib=None) -> float:
    return (lib or load()).kfo_e4m3_to_double(int(code))


def e4m3_from_f32(x: float, lib=None) -> int:
    return int((lib or load()).kfo_e4m3_from_float(float(x)))


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8, a.dtype
    return a


def decode_partials_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, ctx_lens, scale: float,
                        num_splits: int, max_context_len: Optional[int] = None,
                        rows: Optional[Sequence] = None, lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Partials over an E4M3 cache (uint8 codes) with per-KV-head fp32 scales."""
    q, k_cache, v_cache = _u16(q), _u8(k_cache), _u8(v_cache)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt, ctx = _i32(block_tables), _i32(ctx_lens)
    B, Hq, D = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if max_context_len is None:
        max_context_len = int(ctx.max()) if B else 0
    o = np.full((num_splits, B, Hq, D), np.nan, dtype=np.float64)
    lse = np.full((num_splits, B, Hq), np.nan, dtype=np.float64)
    rows_arr, n_rows = None, 0
    if rows is not None:
        rows_arr = _i32(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n_rows = rows_arr.shape[0]
    rc = (lib or load()).kfo_decode_partials_fp8(
        q, k_cache, v_cache, ks, vs, bt, bt.shape[1], ctx, B, Hq, hkv, D, bs, nb, scale, num_splits,
        max_context_len, None if rows_arr is None else rows_arr.ctypes.data, n_rows, o, lse)
    if rc != 0:
        raise ValueError("oracle decode_partials_fp8 failed (rc=%d)" % rc)
    return o, lse


def attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, ctx_lens, scale: float,
                  rows: Optional[Sequence] = None, lib=None) -> Tuple[np.ndarray, np.ndarray]:
    o, lse = decode_partials_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, ctx_lens, scale, 1,
                                 rows=rows, lib=lib)
    return o[0], lse[0]


def append_fp8(k_cache, v_cache, k_new, v_new, k_scale, v_scale, block_tables, ctx_before,
               lib=None) -> Tuple[np.ndarray, np.ndarray, int]:
    """Copies of E4M3 caches with each request's new rows quantised in."""
    k2, v2 = _u8(k_cache).copy(), _u8(v_cache).copy()
    nb, bs, hkv, d = k2.shape
    bt, ctx = _i32(block_tables), _i32(ctx_before)
    skipped = (lib or load()).kfo_append_fp8(
        k2, v2, _u16(k_new), _u16(v_new), np.ascontiguousarray(k_scale, dtype=np.float32),
        np.ascontiguousarray(v_scale, dtype=np.float32), bt, bt.shape[1], ctx, bt.shape[0], hkv, d, bs, nb)
    return k2, v2, skipped


# ----------------------------------------------------------------------------
# Multi-query (chunked prefill / shared prefix) attention
# ----------------------------------------------------------------------------

def multiquery_partials(q, q_start, k_cache, v_cache, block_tables, ctx_lens, scale: float, causal: bool,
                        num_splits: int = 1, max_context_len: Optional[int] = None,
                        lib=None) -> Tuple[np.ndarray, np.ndarray]:
    """Partials o [S, Nq, Hq, D], lse [S, Nq, Hq] of query tokens grouped by
    request (q_start [B+1]) over each request's paged context."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    qs, bt, ctx = _i32(q_start), _i32(block_tables), _i32(ctx_lens)
    Nq, Hq, D = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    B = ctx.shape[0]
    if max_context_len is None:
        max_context_len = int(ctx.max()) if B else 0
    o = np.full((num_splits, Nq, Hq, D), np.nan, dtype=np.float64)
    lse = np.full((num_splits, Nq, Hq), np.nan, dtype=np.float64)
    rc = (lib or load()).kfo_multiquery_partials(q, qs, k_cache, v_cache, bt, bt.shape[1], ctx, int(bool(causal)),
                                                 B, Nq, Hq, hkv, D, bs, nb, scale, num_splits, max_context_len,
                                                 o, lse)
    if rc != 0:
        raise ValueError("oracle multiquery_partials failed (rc=%d)" % rc)
    return o, lse

