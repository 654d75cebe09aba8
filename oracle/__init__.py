"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package. The product path (the
CUDA library and its Python binding) never imports, loads or calls it, and the
two share no code.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc and marshals numpy arrays through ctypes.

Pins (what ties each routine to the pages rather than to itself) are in
``tests/test_oracle_pins.py``. Sources, by page title and section:

* "FlashAttention: Exact Attention as an IO-Aware Streaming Computation",
  sections "Problem setting" and "Mathematical structure": the definition and
  the running (m, l, a) statistics.
* "FlashAttention" (glossary), sections "Move less data" (additive mask M),
  "Why a tile can be discarded", "One row, checked two ways" and "Practice":
  block summaries, their merge and the two worked examples.
* "IO-aware exact attention", sections "Tile order and on-chip capacity"
  (causal: keys at or before the query), "Backward recomputation" and "Why
  implementations form a family" (bias and dropout as variants).
* Dropout's keep decisions: the counter-based generator Philox4x64-10 of Salmon,
  Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, OpenMP, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "attn_oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # The mutation tests (tests/test_oracle_mutants.py) point this at a copy of the
    # oracle built with one planted mistake, to show that the pins catch it.
    override = os.environ.get("ORACLE_MUTANT_LIB")
    if override:
        lib = ctypes.CDLL(override)
    else:
        build()
        lib = ctypes.CDLL(_LIB)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    ip = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_attn_f64.argtypes = [dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int]
    lib.oracle_attn_rows_f64.argtypes = lib.oracle_attn_f64.argtypes + [ip, i64]
    lib.oracle_attn_blockwise_f64.argtypes = lib.oracle_attn_f64.argtypes + [i64]
    lib.oracle_attn_bwd_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int]
    lib.oracle_block_summary_f64.argtypes = [dp, dp, i64, i64, dp, dp, dp]
    lib.oracle_block_summary_f64.restype = None
    lib.oracle_merge_f64.argtypes = [ctypes.c_double, ctypes.c_double, dp, ctypes.c_double, ctypes.c_double, dp, i64, dp, dp, dp]
    lib.oracle_merge_f64.restype = None
    u64 = ctypes.c_uint64
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.oracle_philox4x64_10.argtypes = [u64p, u64p, u64p]
    lib.oracle_philox4x64_10.restype = None
    lib.oracle_dropout_keep.argtypes = [ctypes.POINTER(ctypes.c_uint8), i64, i64, i64, i64, ctypes.c_int, u64, u64]
    lib.oracle_attn_dropout_f64.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, ctypes.c_double,
                                            ctypes.c_int, ctypes.c_int, u64, u64]
    for f in (lib.oracle_attn_f64, lib.oracle_attn_rows_f64, lib.oracle_attn_blockwise_f64, lib.oracle_attn_bwd_f64,
              lib.oracle_num_threads, lib.oracle_dropout_keep, lib.oracle_attn_dropout_f64):
        f.restype = ctypes.c_int
    _lib = lib
    return lib


def _f64(a) -> np.ndarray:
    """Exact conversion to a C-contiguous fp64 array (bf16/fp16/fp32 all embed in fp64)."""
    if hasattr(a, "detach"):  # a torch tensor: widen on the CPU, which is exact
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q, k, v, mask):
    B, H, Nq, d = q.shape
    Bk, Hk, Nk, dk = k.shape
    if (Bk, Hk, dk) != (B, H, d) or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    if mask is not None and mask.shape != (B, Nq, Nk):
        raise ValueError(f"mask must be [B, Nq, Nk] = {(B, Nq, Nk)}, got {mask.shape}")
    return B, H, Nq, Nk, d


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attention(q, k, v, mask=None, scale=None, causal=False):
    """Materialised fp64 attention. Returns (out [B,H,Nq,d], lse [B,H,Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    mask = None if mask is None else _f64(mask)
    B, H, Nq, Nk, d = _shapes(q, k, v, mask)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    rc = _load().oracle_attn_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse),
                                 B, H, Nq, Nk, d, scale, int(bool(causal)))
    if rc != 0:
        raise RuntimeError("oracle_attn_f64 failed")
    return out, lse


def attention_bias(q, k, v, bias, scale=None, causal=False):
    """Attention with a per-head additive bias [B, H, Nq, Nk]: head h of every batch
    index is the shared-mask definition above run on that head alone with mask
    bias[:, h] ("IO-aware exact attention", section "Why implementations form a
    family", names bias as a variant; the glossary's additive M, per head).
    Returns (out [B,H,Nq,d], lse [B,H,Nq])."""
    q, k, v, bias = _f64(q), _f64(k), _f64(v), _f64(bias)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if bias.shape != (B, H, Nq, Nk):
        raise ValueError(f"bias must be [B, H, Nq, Nk] = {(B, H, Nq, Nk)}, got {bias.shape}")
    out = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    for h in range(H):
        o, l = attention(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], mask=bias[:, h], scale=scale, causal=causal)
        out[:, h] = o[:, 0]
        lse[:, h] = l[:, 0]
    return out, lse


def attention_rows(q, k, v, rows, mask=None, scale=None, causal=False):
    """Materialised fp64 attention for flat row ids (b*H + h)*Nq + i.
    Returns (out [len(rows), d], lse [len(rows)])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    mask = None if mask is None else _f64(mask)
    B, H, Nq, Nk, d = _shapes(q, k, v, mask)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((rows.size, d))
    lse = np.zeros(rows.size)
    rc = _load().oracle_attn_rows_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse),
                                      B, H, Nq, Nk, d, scale, int(bool(causal)),
                                      rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.size)
    if rc != 0:
        raise RuntimeError("oracle_attn_rows_f64 failed")
    return out, lse


def attention_blockwise(q, k, v, block, mask=None, scale=None, causal=False):
    """Blockwise (summary + merge) fp64 attention; must equal ``attention``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    mask = None if mask is None else _f64(mask)
    B, H, Nq, Nk, d = _shapes(q, k, v, mask)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    rc = _load().oracle_attn_blockwise_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse),
                                           B, H, Nq, Nk, d, scale, int(bool(causal)), int(block))
    if rc != 0:
        raise RuntimeError("oracle_attn_blockwise_f64 failed")
    return out, lse


def block_summary(scores, values):
    """(m, l, u) of one row's block: scores [n], values [n] or [n, dv]."""
    s = _f64(scores).reshape(-1)
    vals = _f64(values)
    vals2 = vals.reshape(s.size, -1)
    dv = vals2.shape[1]
    m = ctypes.c_double()
    l = ctypes.c_double()
    u = np.zeros(dv)
    _load().oracle_block_summary_f64(_ptr(s), _ptr(np.ascontiguousarray(vals2)), s.size, dv,
                                     ctypes.byref(m), ctypes.byref(l), _ptr(u))
    return m.value, l.value, (u if vals.ndim > 1 else u[0])


def merge(a, b):
    """Merge two block summaries (m, l, u) onto their common maximum."""
    (mA, lA, uA), (mB, lB, uB) = a, b
    uA1 = np.atleast_1d(_f64(uA))
    uB1 = np.atleast_1d(_f64(uB))
    m = ctypes.c_double()
    l = ctypes.c_double()
    u = np.zeros(uA1.size)
    _load().oracle_merge_f64(float(mA), float(lA), _ptr(uA1), float(mB), float(lB), _ptr(uB1), uA1.size,
                             ctypes.byref(m), ctypes.byref(l), _ptr(u))
    scalar = np.ndim(uA) == 0
    return m.value, l.value, (u[0] if scalar else u)


def attention_bwd(q, k, v, dout, mask=None, scale=None, causal=False):
    """fp64 gradients (dq, dk, dv) of sum(dout * attention(q, k, v))."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    mask = None if mask is None else _f64(mask)
    B, H, Nq, Nk, d = _shapes(q, k, v, mask)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = _load().oracle_attn_bwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(dout), _ptr(dq), _ptr(dk),
                                     _ptr(dv), B, H, Nq, Nk, d, scale, int(bool(causal)))
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd_f64 failed")
    return dq, dk, dv


# ---------------------------------------------------------------- dropout
def dropout_threshold(p_drop: float) -> int:
    """Keep threshold of drop probability p: the keep probability (1 - p) rounded to a
    multiple of 1/256 (halves up), as a count of the 256 byte values that keep."""
    t = int(np.floor((1.0 - float(p_drop)) * 256.0 + 0.5)) if float(p_drop) >= 0.0 else 0
    if not 1 <= t <= 256:
        raise ValueError(f"drop probability {p_drop} keeps nothing (or is negative)")
    return t


def philox4x64_10(counter, key):
    """One Philox4x64-10 block (Salmon et al., SC 2011): four 64-bit words."""
    c = (ctypes.c_uint64 * 4)(*[int(x) & (2**64 - 1) for x in counter])
    k = (ctypes.c_uint64 * 2)(*[int(x) & (2**64 - 1) for x in key])
    o = (ctypes.c_uint64 * 4)()
    _load().oracle_philox4x64_10(c, k, o)
    return tuple(int(x) for x in o)


def dropout_keep(B, H, Nq, Nk, p_drop, seed, offset=0):
    """keep[B, H, Nq, Nk] (bool) of the dropout definition in attn_oracle.h."""
    keep = np.zeros((B, H, Nq, Nk), dtype=np.uint8)
    rc = _load().oracle_dropout_keep(keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), B, H, Nq, Nk,
                                     dropout_threshold(p_drop), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1))
    if rc != 0:
        raise RuntimeError("oracle_dropout_keep failed")
    return keep.astype(bool)


def attention_dropout(q, k, v, p_drop, seed, offset=0, scale=None, causal=False):
    """fp64 attention with dropout ("IO-aware exact attention", section "Why
    implementations form a family", names the variant; the reading and the keep
    stream are stated in attn_oracle.h). Returns (out [B,H,Nq,d], lse [B,H,Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, Nk, d = _shapes(q, k, v, None)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    rc = _load().oracle_attn_dropout_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, scale,
                                         int(bool(causal)), dropout_threshold(p_drop), int(seed) & (2**64 - 1),
                                         int(offset) & (2**64 - 1))
    if rc != 0:
        raise RuntimeError("oracle_attn_dropout_f64 failed")
    return out, lse
