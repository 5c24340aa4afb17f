"""Thin ctypes binding of the C-ABI library (include/kf.h), same names.

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels. Tensors must be CUDA tensors in the layouts kf.h
states; the current torch stream is used unless one is given. Importing this
module loads ``_lib/libkf.so`` and fails loudly if it has not been built
(``__graft_entry__.build()``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libkf.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("the kf CUDA library is not built (%s missing); run "
                      "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

KF_OK, KF_ERR_INVALID, KF_ERR_UNSUPPORTED, KF_ERR_CUDA, KF_ERR_DEVICE = range(5)
KF_BF16, KF_F32 = 0, 1
KF_SPLITS_BALANCED = 0  # num_splits of the step calls: balanced one-wave schedule
KF_DEVERR_BLOCK_ID = 0x01
KF_DEVERR_CONTEXT_LEN = 0x02
KF_DEVERR_MAX_CONTEXT = 0x04
KF_DEVERR_APPEND_POS = 0x08
KF_DEVERR_TIMEOUT = 0x10

_vp, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float

_lib.kf_append_kv.restype = _i32
_lib.kf_append_kv.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i64, _vp]
_lib.kf_paged_decode_attention.restype = _i32
_lib.kf_paged_decode_attention.argtypes = [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                           _i32, _i32, _i64, _f32, _i32, _vp, _vp, _vp]
_lib.kf_choose_num_splits.restype = _i32
_lib.kf_choose_num_splits.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _vp, _i32]
_lib.kf_choose_num_splits_for.restype = _i32
_lib.kf_choose_num_splits_for.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _vp, _i32]
_lib.kf_choose_num_splits_fp8.restype = _i32
_lib.kf_choose_num_splits_fp8.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _vp, _i32]
_lib.kf_paged_multiquery_attention.restype = _i32
_lib.kf_paged_multiquery_attention.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                               _i32, _i32, _i32, _i32, _i64, _f32, _i32, _vp, _vp, _vp]
_lib.kf_merge_partials.restype = _i32
_lib.kf_merge_partials.argtypes = [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.kf_decode_step_workspace_size.restype = ctypes.c_size_t
_lib.kf_decode_step_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.kf_decode_step.restype = _i32
_lib.kf_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                _i32, _i64, _f32, _i32, _vp, ctypes.c_size_t, _vp, _i32, _vp, _vp]
_lib.kf_decode_step_static.restype = _i32
_lib.kf_decode_step_merge_partials.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                                _i32, _i32, _i64, _f32, _i32, _vp, _vp, _i32, _vp,
                                                ctypes.c_size_t, _vp, _i32, _vp, _vp]
_lib.kf_decode_step_merge_partials.restype = _i32
_lib.kf_decode_step_static.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                       _i32, _i32, _i64, _f32, _i32, _vp, _i32, _vp, _vp]
KF_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024
_lib.kf_append_kv_fp8.restype = _i32
_lib.kf_append_kv_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i64, _vp]
_lib.kf_paged_decode_attention_fp8.restype = _i32
_lib.kf_paged_decode_attention_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                               _i32, _i32, _i32, _i64, _f32, _i32, _vp, _vp, _vp]
_lib.kf_decode_step_fp8.restype = _i32
_lib.kf_decode_step_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                    _i32, _i32, _i32, _i64, _f32, _i32, _vp, ctypes.c_size_t, _vp, _i32, _vp,
                                    _vp]
_lib.kf_get_device_error.restype = _i32
_lib.kf_check_bounded_wait.restype = _i32
_lib.kf_check_bounded_wait.argtypes = [_vp]
_lib.kf_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), _vp]
_lib.kf_status_string.restype = ctypes.c_char_p
_lib.kf_status_string.argtypes = [_i32]
_lib.kf_version.restype = _i32
_lib.kf_version.argtypes = []


class KfError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, _lib.kf_status_string(status).decode(), status))


def raw():
    """The loaded ctypes library (for callers that pass raw pointers)."""
    return _lib


def _check(status: int, what: str) -> None:
    if status != KF_OK:
        raise KfError(status, what)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _io(t: torch.Tensor, dtype, name: str) -> int:
    """A per-step input or output of the kf_decode_step calls: a CUDA tensor, or
    a pinned host tensor the GPU reads or writes in place (zero-copy)."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("%s must be a CUDA tensor or pinned host memory" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def kf_version() -> int:
    return _lib.kf_version()


def kf_append_kv(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, block_tables: torch.Tensor,
                 context_lens_before: torch.Tensor, stream=None) -> None:
    """Write each request's new K/V row at position context_lens_before[b]."""
    nb, bs, hkv, d = k_cache.shape
    B = block_tables.shape[0]
    _check(_lib.kf_append_kv(
        _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
        _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _dev(context_lens_before, torch.int32, "context_lens_before"), B, hkv, d, bs, nb,
        _stream(stream)), "kf_append_kv")


def kf_choose_num_splits(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                         block_size: int, max_context_len: int, context_lens_host=None,
                         device: Optional[int] = None, num_sms: Optional[int] = None,
                         kv_dtype: str = "bf16") -> int:
    """The library's split count for this batch (host-side plan)."""
    arr = None
    ptr = None
    if context_lens_host is not None:
        arr = torch.as_tensor(context_lens_host, dtype=torch.int32).cpu().contiguous()
        ptr = arr.data_ptr()
    if kv_dtype == "fp8":
        if num_sms is None:
            dev = torch.cuda.current_device() if device is None else device
            num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        n = _lib.kf_choose_num_splits_fp8(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                          max_context_len, ptr, num_sms)
    elif num_sms is not None:
        n = _lib.kf_choose_num_splits_for(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                          max_context_len, ptr, num_sms)
    else:
        dev = torch.cuda.current_device() if device is None else device
        n = _lib.kf_choose_num_splits(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                      max_context_len, ptr, dev)
    if n < 1:
        raise KfError(KF_ERR_INVALID, "kf_choose_num_splits")
    return n


def kf_paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_tables: torch.Tensor, context_lens: torch.Tensor,
                              max_context_len: int, scale: float, num_splits: int,
                              out_partial: Optional[torch.Tensor] = None,
                              lse_partial: Optional[torch.Tensor] = None,
                              stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split-KV decode attention; returns (out_partial [S,B,Hq,D], lse_partial [S,B,Hq])."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if out_partial is None:
        out_partial = torch.empty((num_splits, B, hq, d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((num_splits, B, hq), dtype=torch.float32, device=q.device)
    _check(_lib.kf_paged_decode_attention(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        block_tables.shape[1], _dev(context_lens, torch.int32, "context_lens"), int(max_context_len),
        B, hq, hkv, d, bs, nb, float(scale), int(num_splits),
        _dev(out_partial, torch.float32, "out_partial"), _dev(lse_partial, torch.float32, "lse_partial"),
        _stream(stream)), "kf_paged_decode_attention")
    return out_partial, lse_partial


def kf_paged_multiquery_attention(q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                                  v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  causal: bool, max_context_len: int, max_query_len: int, scale: float,
                                  num_splits: int, out_partial: Optional[torch.Tensor] = None,
                                  lse_partial: Optional[torch.Tensor] = None,
                                  stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Multi-query paged attention (chunked prefill / shared prefix); returns
    (out_partial [S, Nq, Hq, D], lse_partial [S, Nq, Hq])."""
    Nq, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    B = block_tables.shape[0]
    if out_partial is None:
        out_partial = torch.empty((num_splits, Nq, hq, d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((num_splits, Nq, hq), dtype=torch.float32, device=q.device)
    _check(_lib.kf_paged_multiquery_attention(
        _dev(q, torch.bfloat16, "q"), _dev(q_start, torch.int32, "q_start"),
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
        _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), int(bool(causal)), int(max_context_len),
        int(max_query_len), B, Nq, hq, hkv, d, bs, nb, float(scale), int(num_splits),
        _dev(out_partial, torch.float32, "out_partial"), _dev(lse_partial, torch.float32, "lse_partial"),
        _stream(stream)), "kf_paged_multiquery_attention")
    return out_partial, lse_partial


def kf_merge_partials(out_partial: torch.Tensor, lse_partial: torch.Tensor,
                      out: Optional[torch.Tensor] = None, out_dtype=torch.float32,
                      lse_out: Optional[torch.Tensor] = None, want_lse: bool = True,
                      stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """LSE merge of [S,B,Hq,D]/[S,B,Hq] partials; returns (out [B,Hq,D], lse [B,Hq] or None)."""
    S, B, hq, d = out_partial.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=out_partial.device)
    code = {torch.float32: KF_F32, torch.bfloat16: KF_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, hq), dtype=torch.float32, device=out_partial.device)
    _check(_lib.kf_merge_partials(
        _dev(out_partial, torch.float32, "out_partial"), _dev(lse_partial, torch.float32, "lse_partial"),
        S, B, hq, d, _dev(out, out.dtype, "out"), code,
        None if lse_out is None else _dev(lse_out, torch.float32, "lse_out"), _stream(stream)),
        "kf_merge_partials")
    return out, lse_out


def kf_decode_step_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                  num_splits: int) -> int:
    return int(_lib.kf_decode_step_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, num_splits))


def make_workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, num_splits: int,
                   device=None) -> torch.Tensor:
    """A zero-filled workspace for kf_decode_step (the zero fill is required once)."""
    n = kf_decode_step_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, num_splits)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def kf_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens_before: torch.Tensor,
                   max_context_len: int, scale: float, num_splits: int,
                   workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   out_dtype=torch.float32, lse_out: Optional[torch.Tensor] = None, want_lse: bool = True,
                   stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Append + split attention + merge in one launch; returns (out, lse).
    q, k_new, v_new, block_tables, context_lens_before, out and lse_out may be
    pinned host tensors (read and written by the kernel in place)."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=k_cache.device)
    code = {torch.float32: KF_F32, torch.bfloat16: KF_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, hq), dtype=torch.float32, device=k_cache.device)
    if workspace is None and num_splits != 1:
        raise ValueError("num_splits > 1 and the balanced schedule need a workspace (make_workspace)")
    ws_ptr = None if workspace is None else _dev(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(_lib.kf_decode_step(
        _io(q, torch.bfloat16, "q"), _io(k_new, torch.bfloat16, "k_new"), _io(v_new, torch.bfloat16, "v_new"),
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
        _io(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _io(context_lens_before, torch.int32, "context_lens_before"), int(max_context_len), B, hq, hkv, d,
        bs, nb, float(scale), int(num_splits), ws_ptr, ws_bytes, _io(out, out.dtype, "out"), code,
        None if lse_out is None else _io(lse_out, torch.float32, "lse_out"), _stream(stream)),
        "kf_decode_step")
    return out, lse_out


def kf_decode_step_merge_partials(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                  k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                                  context_lens_before: torch.Tensor, max_context_len: int, scale: float,
                                  num_splits: int, extra_out_partial: torch.Tensor,
                                  extra_lse_partial: torch.Tensor, workspace: torch.Tensor,
                                  out: Optional[torch.Tensor] = None, out_dtype=torch.float32,
                                  lse_out: Optional[torch.Tensor] = None, want_lse: bool = True,
                                  stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """kf_decode_step whose merge also takes the extra partials
    ([n, B, Hq, D] and [n, B, Hq]); returns (out, lse)."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    n_ex = int(extra_lse_partial.shape[0])
    if tuple(extra_out_partial.shape) != (n_ex, B, hq, d) or tuple(extra_lse_partial.shape) != (n_ex, B, hq):
        raise ValueError("extra partials must be [n, B, Hq, D] and [n, B, Hq]")
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=k_cache.device)
    code = {torch.float32: KF_F32, torch.bfloat16: KF_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, hq), dtype=torch.float32, device=k_cache.device)
    _check(_lib.kf_decode_step_merge_partials(
        _io(q, torch.bfloat16, "q"), _io(k_new, torch.bfloat16, "k_new"), _io(v_new, torch.bfloat16, "v_new"),
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
        _io(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _io(context_lens_before, torch.int32, "context_lens_before"), int(max_context_len), B, hq, hkv, d,
        bs, nb, float(scale), int(num_splits), _dev(extra_out_partial, torch.float32, "extra_out_partial"),
        _dev(extra_lse_partial, torch.float32, "extra_lse_partial"), n_ex,
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _io(out, out.dtype, "out"), code,
        None if lse_out is None else _io(lse_out, torch.float32, "lse_out"), _stream(stream)),
        "kf_decode_step_merge_partials")
    return out, lse_out


def kf_decode_step_static(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                          k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                          context_lens_before: torch.Tensor, max_context_len: int, scale: float,
                          num_splits: int, out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """kf_decode_step with the library's own fixed scratch instead of a workspace,
    for callers that may not allocate device memory; `out` (and `lse_out`) must
    be given. Calls on one device must not overlap on the GPU."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    code = {torch.float32: KF_F32, torch.bfloat16: KF_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    _check(_lib.kf_decode_step_static(
        _io(q, torch.bfloat16, "q"), _io(k_new, torch.bfloat16, "k_new"), _io(v_new, torch.bfloat16, "v_new"),
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
        _io(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _io(context_lens_before, torch.int32, "context_lens_before"), int(max_context_len), B, hq, hkv, d,
        bs, nb, float(scale), int(num_splits), _io(out, out.dtype, "out"), code,
        None if lse_out is None else _io(lse_out, torch.float32, "lse_out"), _stream(stream)),
        "kf_decode_step_static")


def _dev8(t: torch.Tensor, name: str) -> int:
    """An FP8 E4M3 cache: uint8 codes or torch.float8_e4m3fn."""
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError("%s must be uint8 E4M3 codes or float8_e4m3fn, got %s" % (name, t.dtype))
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    return t.data_ptr()


def kf_append_kv_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
                     context_lens_before, stream=None) -> None:
    """Quantise and write each request's new K/V row into E4M3 caches."""
    nb, bs, hkv, d = k_cache.shape
    B = block_tables.shape[0]
    _check(_lib.kf_append_kv_fp8(
        _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev8(k_cache, "k_cache"), _dev8(v_cache, "v_cache"), _dev(k_scale, torch.float32, "k_scale"),
        _dev(v_scale, torch.float32, "v_scale"), _dev(block_tables, torch.int32, "block_tables"),
        block_tables.shape[1], _dev(context_lens_before, torch.int32, "context_lens_before"), B, hkv, d,
        bs, nb, _stream(stream)), "kf_append_kv_fp8")


def kf_paged_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                  max_context_len: int, scale: float, num_splits: int,
                                  out_partial=None, lse_partial=None, stream=None):
    """Split-KV decode attention over E4M3 caches; returns (out_partial, lse_partial)."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if out_partial is None:
        out_partial = torch.empty((num_splits, B, hq, d), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        lse_partial = torch.empty((num_splits, B, hq), dtype=torch.float32, device=q.device)
    _check(_lib.kf_paged_decode_attention_fp8(
        _dev(q, torch.bfloat16, "q"), _dev8(k_cache, "k_cache"), _dev8(v_cache, "v_cache"),
        _dev(k_scale, torch.float32, "k_scale"), _dev(v_scale, torch.float32, "v_scale"),
        _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), int(max_context_len), B, hq, hkv, d, bs, nb,
        float(scale), int(num_splits), _dev(out_partial, torch.float32, "out_partial"),
        _dev(lse_partial, torch.float32, "lse_partial"), _stream(stream)), "kf_paged_decode_attention_fp8")
    return out_partial, lse_partial


def kf_decode_step_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
                       context_lens_before, max_context_len: int, scale: float, num_splits: int,
                       workspace=None, out=None, out_dtype=torch.float32, lse_out=None, want_lse=True,
                       stream=None):
    """Single-launch decode step over E4M3 caches; returns (out, lse). The
    per-step tensors may be pinned host memory, as for kf_decode_step."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=k_cache.device)
    code = {torch.float32: KF_F32, torch.bfloat16: KF_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, hq), dtype=torch.float32, device=k_cache.device)
    if workspace is None and num_splits != 1:
        raise ValueError("num_splits > 1 and the balanced schedule need a workspace (make_workspace)")
    _check(_lib.kf_decode_step_fp8(
        _io(q, torch.bfloat16, "q"), _io(k_new, torch.bfloat16, "k_new"), _io(v_new, torch.bfloat16, "v_new"),
        _dev8(k_cache, "k_cache"), _dev8(v_cache, "v_cache"), _dev(k_scale, torch.float32, "k_scale"),
        _dev(v_scale, torch.float32, "v_scale"), _io(block_tables, torch.int32, "block_tables"),
        block_tables.shape[1], _io(context_lens_before, torch.int32, "context_lens_before"),
        int(max_context_len), B, hq, hkv, d, bs, nb, float(scale), int(num_splits),
        None if workspace is None else _dev(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _io(out, out.dtype, "out"), code,
        None if lse_out is None else _io(lse_out, torch.float32, "lse_out"), _stream(stream)),
        "kf_decode_step_fp8")
    return out, lse_out


def kf_check_bounded_wait(stream=None) -> None:
    """Launch one bounded wait that nothing completes (sets KF_DEVERR_TIMEOUT)."""
    _check(_lib.kf_check_bounded_wait(_stream(stream)), "kf_check_bounded_wait")


def kf_get_device_error(stream=None) -> int:
    """Synchronise the stream, return and clear the device error word (0 = none)."""
    flags = ctypes.c_uint(0)
    st = _lib.kf_get_device_error(ctypes.byref(flags), _stream(stream))
    if st not in (KF_OK, KF_ERR_DEVICE):
        raise KfError(st, "kf_get_device_error")
    return flags.value
