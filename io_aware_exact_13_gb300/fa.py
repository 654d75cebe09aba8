"""Python binding of the C ABI in ``include/fa.h`` (argument marshalling only).

Every function here forwards device pointers, sizes and the current CUDA
stream to ``libfa.so``; all arithmetic runs in the library's CUDA kernels.
There is no CPU fallback: importing this module fails loudly when the library
has not been built, and every call raises if the library returns an error.

Names follow the C ABI: ``fa_fwd`` (bf16), ``fa_fwd_fp16``, ``fa_fwd_fp32``,
``fa_fwd_masked`` / ``fa_fwd_masked_fp16`` (a shared mask packed in a workspace),
``fa_fwd_dropout`` / ``fa_fwd_dropout_fp16`` (dropout on the probabilities),
``fa_fwd_splitkv`` / ``fa_fwd_splitkv_fp16`` (decoding), ``fa_bwd`` /
``fa_bwd_fp16`` (backward by recomputation), ``fa_fwd_varlen`` /
``fa_fwd_varlen_fp16`` (packed variable-length batches), their sizing helpers,
``fa_status_string``, ``fa_get_device_status``, ``fa_num_sms``. ``attention``,
``attention_decode``, ``attention_varlen`` and ``attention_backward`` are convenience wrappers that allocate outputs (and
the split-KV workspace) with torch and pick the entry point from the dtype.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with `python -m io_aware_exact_13_gb300.build` "
        "(there is no fallback implementation)")
lib = ctypes.CDLL(_LIB_PATH)

FA_OK = 0
FA_ERR_NULL = -1
FA_ERR_ALIGN = -2
FA_ERR_SHAPE = -3
FA_ERR_UNSUPPORTED = -4
FA_ERR_LAUNCH = -5
FA_ERR_TIMEOUT = -6
FA_ERR_WORKSPACE = -7
FA_ERR_SEQLENS = -8
FA_ERR_ARG = -9

# Every symbol the header declares, with its ctypes signature.
_vp = ctypes.c_void_p
_FWD_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
             ctypes.c_float, ctypes.c_int, _vp]
SIGNATURES = {
    "fa_fwd": (ctypes.c_int, _FWD_ARGS),
    "fa_fwd_fp16": (ctypes.c_int, _FWD_ARGS),
    "fa_fwd_fp32": (ctypes.c_int, _FWD_ARGS),
    "fa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_get_device_status": (ctypes.c_int, [_vp]),
    "fa_num_sms": (ctypes.c_int, []),
    "fa_fwd_bias": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, _vp]),
    "fa_fwd_bias_fp16": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, _vp]),
    "fa_fwd_gqa": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, _vp]),
    "fa_fwd_masked_workspace_bytes": (ctypes.c_longlong, [ctypes.c_int] * 2),
    "fa_fwd_dropout": (ctypes.c_int, [_vp] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, ctypes.c_float,
                                                                       ctypes.c_ulonglong, ctypes.c_ulonglong, _vp]),
    "fa_fwd_dropout_fp16": (ctypes.c_int, [_vp] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int,
                                                                            ctypes.c_float, ctypes.c_ulonglong,
                                                                            ctypes.c_ulonglong, _vp]),
    "fa_fwd_masked": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, _vp,
                                                                        ctypes.c_ulonglong, _vp]),
    "fa_fwd_masked_fp16": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, _vp,
                                                                             ctypes.c_ulonglong, _vp]),
    "fa_fwd_gqa_fp16": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, _vp]),
    "fa_splitkv_num_splits": (ctypes.c_int, [ctypes.c_int] * 5),
    "fa_splitkv_workspace_bytes": (ctypes.c_longlong, [ctypes.c_int] * 5),
    "fa_fwd_splitkv": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp] + [ctypes.c_int] * 5 +
                       [ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_ulonglong, _vp]),
    "fa_fwd_splitkv_fp16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp] + [ctypes.c_int] * 5 +
                            [ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_ulonglong, _vp]),
    "fa_fwd_splitkv_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp] + [ctypes.c_int] * 5 +
                               [ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp]),
    "fa_fwd_varlen": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, _vp]),
    "fa_fwd_varlen_fp16": (ctypes.c_int, [_vp] * 6 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, _vp]),
    "fa_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_ulonglong, _vp]),
    "fa_fwd_host": (ctypes.c_int, [_vp] * 10 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp]),
    "fa_fwd_host_fp16": (ctypes.c_int, [_vp] * 10 + [ctypes.c_int] * 4 +
                         [ctypes.c_float, ctypes.c_int, ctypes.c_int, _vp]),
    "fa_bwd_workspace_bytes": (ctypes.c_longlong, [ctypes.c_int] * 4),
    "fa_bwd": (ctypes.c_int, [_vp] * 9 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, _vp,
                                                                 ctypes.c_ulonglong, _vp]),
    "fa_bwd_fp16": (ctypes.c_int, [_vp] * 9 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, _vp,
                                                                      ctypes.c_ulonglong, _vp]),
}
for _name, (_res, _args) in SIGNATURES.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})")
        self.status = status


def fa_status_string(status: int) -> str:
    return lib.fa_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _raw_fwd(fn_name, q, k, v, mask, out, lse, B, H, N, d, scale, causal, stream):
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse), int(B), int(H), int(N),
                               int(d), float(scale), int(bool(causal)), ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def _check(q, k, v, mask, out, lse, dtype):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape or out.shape != q.shape:
        raise ValueError("q, k, v, out must all be [B, H, N, d]")
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous CUDA float32 [B, H, N] tensor")
    if mask is not None and (mask.dtype != torch.float32 or not mask.is_cuda or not mask.is_contiguous()
                             or mask.shape != (B, N, N)):
        raise ValueError("mask must be a contiguous CUDA float32 [B, N, N] tensor")
    return B, H, N, d


def fa_fwd(q, k, v, mask_or_null, out, lse, scale, causal, stream=None):
    """bf16 forward into caller-provided ``out`` [B,H,N,d] and ``lse`` [B,H,N]."""
    B, H, N, d = _check(q, k, v, mask_or_null, out, lse, torch.bfloat16)
    _raw_fwd("fa_fwd", q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream)


def fa_fwd_fp16(q, k, v, mask_or_null, out, lse, scale, causal, stream=None):
    """fp16 forward into caller-provided ``out`` and ``lse``."""
    B, H, N, d = _check(q, k, v, mask_or_null, out, lse, torch.float16)
    _raw_fwd("fa_fwd_fp16", q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream)


def fa_fwd_fp32(q, k, v, mask_or_null, out, lse, scale, causal, stream=None):
    """fp32 forward (fp32 arithmetic on the CUDA cores) into caller-provided ``out`` and ``lse``."""
    B, H, N, d = _check(q, k, v, mask_or_null, out, lse, torch.float32)
    _raw_fwd("fa_fwd_fp32", q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream)


_BY_DTYPE = {torch.bfloat16: fa_fwd, torch.float16: fa_fwd_fp16, torch.float32: fa_fwd_fp32}


def attention(q, k, v, mask=None, scale=None, causal=False, out=None, lse=None, stream=None):
    """O, lse = softmax(scale * q k^T + mask) v for [B,H,N,d] CUDA tensors. A bf16 / fp16
    forward with a mask goes through ``fa_fwd_masked`` with a workspace from torch."""
    if q.dtype not in _BY_DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if mask is not None and q.dtype in _MASKED:
        ws = torch.empty(fa_fwd_masked_workspace_bytes(B, N), dtype=torch.uint8, device=q.device)
        _MASKED[q.dtype](q, k, v, mask, out, lse, scale, causal, ws, stream)
    else:
        _BY_DTYPE[q.dtype](q, k, v, mask, out, lse, scale, causal, stream)
    return out, lse


# ---------------------------------------------------------------- additive mask, packed
def fa_fwd_masked_workspace_bytes(B, N) -> int:
    n = int(lib.fa_fwd_masked_workspace_bytes(int(B), int(N)))
    if n < 0:
        raise FAError(n, "fa_fwd_masked_workspace_bytes")
    return n


def _fwd_masked(fn_name, dtype, q, k, v, mask, out, lse, scale, causal, workspace, stream):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape or out.shape != q.shape or H % Hkv:
        raise ValueError("q, out: [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous CUDA float32 [B, H, N] tensor")
    if (mask is None or mask.dtype != torch.float32 or mask.shape != (B, N, N) or not mask.is_contiguous()
            or not mask.is_cuda):
        raise ValueError("mask must be a contiguous CUDA float32 [B, N, N] tensor")
    if workspace is None or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                               float(scale), int(bool(causal)), _ptr(workspace), nbytes,
                               ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_fwd_masked(q, k, v, mask, out, lse, scale, causal, workspace, stream=None):
    """bf16 forward with a shared [B, N, N] fp32 mask, packed to one bit per entry in ``workspace``
    (at least ``fa_fwd_masked_workspace_bytes(B, N)`` bytes) when its entries are all 0 or -inf;
    k, v may hold fewer heads (grouped-query)."""
    _fwd_masked("fa_fwd_masked", torch.bfloat16, q, k, v, mask, out, lse, scale, causal, workspace, stream)


def fa_fwd_masked_fp16(q, k, v, mask, out, lse, scale, causal, workspace, stream=None):
    """fp16 forward with a shared mask and a workspace (see ``fa_fwd_masked``)."""
    _fwd_masked("fa_fwd_masked_fp16", torch.float16, q, k, v, mask, out, lse, scale, causal, workspace, stream)


_MASKED = {torch.bfloat16: fa_fwd_masked, torch.float16: fa_fwd_masked_fp16}


# ---------------------------------------------------------------- dropout
def _fwd_dropout(fn_name, dtype, q, k, v, out, lse, scale, causal, p_drop, seed, offset, stream):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape or out.shape != q.shape or H % Hkv:
        raise ValueError("q, out: [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous CUDA float32 [B, H, N] tensor")
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d, float(scale),
                               int(bool(causal)), float(p_drop), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                               ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_fwd_dropout(q, k, v, out, lse, scale, causal, p_drop, seed, offset=0, stream=None):
    """bf16 forward with dropout: keep decisions from Philox4x64-10 keyed by ``seed``, counter
    {query row, key / 32, b*H + h, ``offset``}; k, v may hold fewer heads (grouped-query)."""
    _fwd_dropout("fa_fwd_dropout", torch.bfloat16, q, k, v, out, lse, scale, causal, p_drop, seed, offset, stream)


def fa_fwd_dropout_fp16(q, k, v, out, lse, scale, causal, p_drop, seed, offset=0, stream=None):
    """fp16 forward with dropout (see ``fa_fwd_dropout``)."""
    _fwd_dropout("fa_fwd_dropout_fp16", torch.float16, q, k, v, out, lse, scale, causal, p_drop, seed, offset, stream)


def attention_dropout(q, k, v, p_drop, seed, offset=0, scale=None, causal=False, stream=None):
    """Forward with dropout; allocates O and lse."""
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fn = {torch.bfloat16: fa_fwd_dropout, torch.float16: fa_fwd_dropout_fp16}[q.dtype]
    fn(q, k, v, out, lse, scale, causal, p_drop, seed, offset, stream)
    return out, lse


# ---------------------------------------------------------------- forward from host memory
def fa_fwd_host(q_host, k_host, v_host, out_host, lse_host, q_dev, k_dev, v_dev, out_dev, lse_dev, scale, causal,
                n_chunks=4, stream=None):
    """Forward with inputs and outputs in (pinned) host tensors; the device tensors
    are caller-owned staging buffers. Copies and compute are pipelined over head
    chunks; synchronise the stream before reading out_host / lse_host."""
    dtype = q_host.dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("bf16 or fp16 inputs")
    for name, t in (("q_host", q_host), ("k_host", k_host), ("v_host", v_host), ("out_host", out_host)):
        if t.dtype != dtype or t.is_cuda or not t.is_contiguous() or t.shape != q_host.shape:
            raise ValueError(f"{name} must be a contiguous host {dtype} tensor shaped like q_host")
    for name, t in (("q_dev", q_dev), ("k_dev", k_dev), ("v_dev", v_dev), ("out_dev", out_dev)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous() or t.shape != q_host.shape:
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor shaped like q_host")
    B, H, N, d = q_host.shape
    for name, t, cuda in (("lse_host", lse_host, False), ("lse_dev", lse_dev, True)):
        if t.dtype != torch.float32 or t.is_cuda != cuda or not t.is_contiguous() or t.shape != (B, H, N):
            raise ValueError(f"{name} must be a contiguous float32 [B, H, N] tensor")
    fn = lib.fa_fwd_host if dtype == torch.bfloat16 else lib.fa_fwd_host_fp16
    rc = fn(*[_ptr(t) for t in (q_host, k_host, v_host, out_host, lse_host, q_dev, k_dev, v_dev, out_dev, lse_dev)],
            B, H, N, d, float(scale), int(bool(causal)), int(n_chunks), ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_host")


# ---------------------------------------------------------------- grouped-query attention
def _fwd_gqa(fn_name, dtype, q, k, v, mask_or_null, out, lse, scale, causal, stream):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape or out.shape != q.shape or H % Hkv:
        raise ValueError("q, out: [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous CUDA float32 [B, H, N] tensor")
    if mask_or_null is not None and (mask_or_null.dtype != torch.float32 or mask_or_null.shape != (B, N, N)
                                     or not mask_or_null.is_contiguous() or not mask_or_null.is_cuda):
        raise ValueError("mask must be a contiguous CUDA float32 [B, N, N] tensor")
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(mask_or_null), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                               float(scale), int(bool(causal)), ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_fwd_gqa(q, k, v, mask_or_null, out, lse, scale, causal, stream=None):
    """bf16 grouped-query forward: k, v are [B, Hkv, N, d], shared by H / Hkv query heads each."""
    _fwd_gqa("fa_fwd_gqa", torch.bfloat16, q, k, v, mask_or_null, out, lse, scale, causal, stream)


def fa_fwd_gqa_fp16(q, k, v, mask_or_null, out, lse, scale, causal, stream=None):
    """fp16 grouped-query forward."""
    _fwd_gqa("fa_fwd_gqa_fp16", torch.float16, q, k, v, mask_or_null, out, lse, scale, causal, stream)


# ---------------------------------------------------------------- per-head additive bias
def _fwd_bias(fn_name, dtype, q, k, v, bias, out, lse, scale, causal, stream):
    B, H, N, d = _check(q, k, v, None, out, lse, dtype)
    if (bias is None or bias.dtype != torch.float32 or bias.shape != (B, H, N, N) or not bias.is_contiguous()
            or not bias.is_cuda):
        raise ValueError("bias must be a contiguous CUDA float32 [B, H, N, N] tensor")
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                               int(bool(causal)), ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_fwd_bias(q, k, v, bias, out, lse, scale, causal, stream=None):
    """bf16 forward with a per-head additive bias [B, H, N, N] (fp32)."""
    _fwd_bias("fa_fwd_bias", torch.bfloat16, q, k, v, bias, out, lse, scale, causal, stream)


def fa_fwd_bias_fp16(q, k, v, bias, out, lse, scale, causal, stream=None):
    """fp16 forward with a per-head additive bias [B, H, N, N] (fp32)."""
    _fwd_bias("fa_fwd_bias_fp16", torch.float16, q, k, v, bias, out, lse, scale, causal, stream)


def attention_bias(q, k, v, bias, scale=None, causal=False, stream=None):
    """Forward with a per-head additive bias; allocates O and lse."""
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fn = {torch.bfloat16: fa_fwd_bias, torch.float16: fa_fwd_bias_fp16}[q.dtype]
    fn(q, k, v, bias, out, lse, scale, causal, stream)
    return out, lse


# ---------------------------------------------------------------- split-KV decoding
def fa_splitkv_num_splits(B, H, Nq, Nk, d) -> int:
    n = int(lib.fa_splitkv_num_splits(int(B), int(H), int(Nq), int(Nk), int(d)))
    if n < 0:
        raise FAError(n, "fa_splitkv_num_splits")
    return n


def fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits) -> int:
    n = int(lib.fa_splitkv_workspace_bytes(int(B), int(H), int(Nq), int(d), int(n_splits)))
    if n < 0:
        raise FAError(n, "fa_splitkv_workspace_bytes")
    return n


def _check_splitkv(q, k, v, out, lse, dtype):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("q, out must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("k, v must be [B, H, Nk, d] with q's B, H, d")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, Nq):
        raise ValueError("lse must be a contiguous CUDA float32 [B, H, Nq] tensor")
    return B, H, Nq, k.shape[2], d


def _raw_splitkv(fn_name, q, k, v, out, lse, scale, causal, n_splits, workspace, stream, dtype):
    B, H, Nq, Nk, d = _check_splitkv(q, k, v, out, lse, dtype)
    if workspace is None or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, float(scale),
                               int(bool(causal)), int(n_splits), _ptr(workspace), nbytes,
                               ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_fwd_splitkv(q, k, v, out, lse, scale, causal, n_splits, workspace, stream=None):
    """bf16 split-KV forward (Nq <= 16 query rows, Nk keys) into ``out`` and ``lse``."""
    _raw_splitkv("fa_fwd_splitkv", q, k, v, out, lse, scale, causal, n_splits, workspace, stream, torch.bfloat16)


def fa_fwd_splitkv_fp16(q, k, v, out, lse, scale, causal, n_splits, workspace, stream=None):
    """fp16 split-KV forward into ``out`` and ``lse``."""
    _raw_splitkv("fa_fwd_splitkv_fp16", q, k, v, out, lse, scale, causal, n_splits, workspace, stream,
                 torch.float16)


def fa_fwd_splitkv_noalloc(q, k, v, out, lse, scale, causal, n_splits, stream=None):
    """bf16 split-KV forward with no workspace: for callers that cannot allocate
    device memory at the call site (a framework owning all device memory, a
    serving loop that must not pay cudaMalloc's device-wide synchronisation, a
    fixed-budget embedded host). The library's fixed 16 MiB scratch array is
    used instead; calls that overlap on the GPU race on it."""
    B, H, Nq, Nk, d = _check_splitkv(q, k, v, out, lse, torch.bfloat16)
    rc = lib.fa_fwd_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, float(scale),
                                    int(bool(causal)), int(n_splits), ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_splitkv_noalloc")


def attention_decode(q, k, v, scale=None, causal=False, n_splits=None, stream=None):
    """Split-KV forward for few query rows; the workspace is a torch allocation."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    n_splits = fa_splitkv_num_splits(B, H, Nq, Nk, d) if n_splits is None else n_splits
    ws = torch.empty(fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fn = {torch.bfloat16: fa_fwd_splitkv, torch.float16: fa_fwd_splitkv_fp16}[q.dtype]
    fn(q, k, v, out, lse, scale, causal, n_splits, ws, stream)
    return out, lse


# ---------------------------------------------------------------- packed variable-length batch
def _raw_varlen(fn_name, dtype, q, k, v, out, lse, cu_seqlens, max_seqlen, scale, causal, stream):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor [total, heads, d]")
    total, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (total, Hkv, d) or v.shape != k.shape or out.shape != q.shape or H % Hkv:
        raise ValueError("q, out: [total, H, d]; k, v: [total, Hkv, d] with Hkv dividing H")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (H, total):
        raise ValueError("lse must be a contiguous CUDA float32 [H, total] tensor")
    if (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or not cu_seqlens.is_contiguous()
            or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2):
        raise ValueError("cu_seqlens must be a contiguous CUDA int32 [nseq + 1] tensor")
    nseq = cu_seqlens.numel() - 1
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens), nseq, total,
                               int(max_seqlen), H, Hkv, d, float(scale), int(bool(causal)),
                               ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_fwd_varlen(q, k, v, out, lse, cu_seqlens, max_seqlen, scale, causal, stream=None):
    """bf16 forward over packed sequences: q, out [total, H, d], k, v [total, Hkv, d], lse [H, total]."""
    _raw_varlen("fa_fwd_varlen", torch.bfloat16, q, k, v, out, lse, cu_seqlens, max_seqlen, scale, causal, stream)


def fa_fwd_varlen_fp16(q, k, v, out, lse, cu_seqlens, max_seqlen, scale, causal, stream=None):
    """fp16 forward over packed sequences."""
    _raw_varlen("fa_fwd_varlen_fp16", torch.float16, q, k, v, out, lse, cu_seqlens, max_seqlen, scale, causal,
                stream)


def attention_varlen(q, k, v, cu_seqlens, max_seqlen, scale=None, causal=False, stream=None):
    """O [total, H, d] and lse [H, total] for packed sequences; allocates the outputs with torch."""
    total, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    fn = {torch.bfloat16: fa_fwd_varlen, torch.float16: fa_fwd_varlen_fp16}[q.dtype]
    fn(q, k, v, out, lse, cu_seqlens, max_seqlen, scale, causal, stream)
    return out, lse


# ---------------------------------------------------------------- backward (recomputation)
def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    n = int(lib.fa_bwd_workspace_bytes(int(B), int(H), int(N), int(d)))
    if n < 0:
        raise FAError(n, "fa_bwd_workspace_bytes")
    return n


def _raw_bwd(fn_name, dtype, q, k, v, out, dout, lse, dq, dk, dv, scale, causal, workspace, stream):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout), ("dq", dq), ("dk", dk),
                    ("dv", dv)):
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError(f"{name} must be [B, H, N, d] like q")
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be a contiguous CUDA float32 [B, H, N] tensor")
    if workspace is None or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    rc = getattr(lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, H, N, d, float(scale), int(bool(causal)), _ptr(workspace), nbytes,
                               ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, fn_name)


def fa_bwd(q, k, v, out, dout, lse, dq, dk, dv, scale, causal, workspace, stream=None):
    """bf16 backward into caller-provided ``dq``, ``dk``, ``dv`` [B,H,N,d]."""
    _raw_bwd("fa_bwd", torch.bfloat16, q, k, v, out, dout, lse, dq, dk, dv, scale, causal, workspace, stream)


def fa_bwd_fp16(q, k, v, out, dout, lse, dq, dk, dv, scale, causal, workspace, stream=None):
    """fp16 backward into caller-provided ``dq``, ``dk``, ``dv``."""
    _raw_bwd("fa_bwd_fp16", torch.float16, q, k, v, out, dout, lse, dq, dk, dv, scale, causal, workspace, stream)


def attention_backward(q, k, v, out, dout, lse, scale=None, causal=False, workspace=None, stream=None):
    """(dq, dk, dv) of sum(dout * out) for out, lse from ``attention``; allocates
    the outputs and, unless given, the workspace with torch."""
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = {torch.bfloat16: fa_bwd, torch.float16: fa_bwd_fp16}[q.dtype]
    fn(q, k, v, out, dout, lse, dq, dk, dv, scale, causal, workspace, stream)
    return dq, dk, dv


def fa_get_device_status(stream=None) -> int:
    return int(lib.fa_get_device_status(ctypes.c_void_p(_stream_handle(stream))))


def fa_selftest_wait_timeout(timeout_ns, stream=None):
    """Enqueue the bounded-wait self-test (a wait nothing completes); afterwards
    fa_get_device_status() must report FA_ERR_TIMEOUT."""
    rc = lib.fa_selftest_wait_timeout(int(timeout_ns), ctypes.c_void_p(_stream_handle(stream)))
    if rc != FA_OK:
        raise FAError(rc, "fa_selftest_wait_timeout")


def fa_num_sms() -> int:
    return int(lib.fa_num_sms())
