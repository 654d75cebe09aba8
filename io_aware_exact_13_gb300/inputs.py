"""Seeded synthetic inputs for the attention forward.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic. Its tensors feed both the CUDA path and the fp64 oracle,
so both sides see identical bits.

Recipe (per workload): a CPU ``torch.Generator`` seeded with the workload's
seed draws, in this order, Q, K and V as fp32 standard normals of shape
[B, H, N, d]; then, where the workload asks for it, a per-key-row offset
U(-a, a) of shape [B, H, N, 1] added to K; then an additive fp32 mask of
shape [B, N, N] whose entries are -inf with probability ``mask_frac`` (0
otherwise) plus ``round(full_row_frac * N)`` query rows per batch index,
chosen without replacement, set entirely to -inf. Q, K, V are multiplied by
``mul`` and finally rounded to the storage dtype (round to nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str
    causal: bool
    scale: float
    seed: int
    mul: float = 1.0
    k_offset: float = 0.0
    mask_frac: float = 0.0
    full_row_frac: float = 0.0
    note: str = field(default="", compare=False)

    @property
    def has_mask(self) -> bool:
        return self.mask_frac > 0.0 or self.full_row_frac > 0.0

    @property
    def flops(self) -> float:
        """Attention flop count 4*B*H*N^2*d, halved for causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N, "d": self.d,
                "dtype": self.dtype, "causal": self.causal, "mask": self.has_mask, "scale": self.scale}


# The five workloads of the attention-forward benchmark suite, smallest first.
WORKLOADS = {
    "n256_d64_fp32": Workload("n256_d64_fp32", 1, 1, 256, 64, "fp32", False, 1 / 8, 1001,
                              note="fp32 inputs, no mask, non-causal"),
    "b4h8_n1024_d64_bf16_causal": Workload("b4h8_n1024_d64_bf16_causal", 4, 8, 1024, 64, "bf16", True, 1 / 8, 1002),
    "b2h16_n4096_d128_fp16_mask": Workload("b2h16_n4096_d128_fp16_mask", 2, 16, 4096, 128, "fp16", False,
                                           1 / math.sqrt(128), 1003, mul=1.5, mask_frac=0.10, full_row_frac=0.01,
                                           note="additive [B,N,N] mask, 10% -inf, ~1% rows fully masked"),
    "b1h32_n8192_d128_bf16_causal": Workload("b1h32_n8192_d128_bf16_causal", 1, 32, 8192, 128, "bf16", True,
                                             1 / math.sqrt(128), 1004),
    "b1h8_n32768_d128_bf16_causal_koff": Workload("b1h8_n32768_d128_bf16_causal_koff", 1, 8, 32768, 128, "bf16",
                                                  True, 1 / math.sqrt(128), 1005, k_offset=4.0,
                                                  note="K rows offset by U(-4,4) to stress max rescaling"),
}
HEADLINE = "b1h32_n8192_d128_bf16_causal"


@dataclass(frozen=True)
class DecodeWorkload:
    """Few query rows (Nq) against a long key/value sequence (Nk)."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def kv_bytes(self) -> int:
        """K and V bytes, each read once per call."""
        return 2 * self.B * self.H * self.Nk * self.d * (4 if self.dtype == "fp32" else 2)

    @property
    def flops(self) -> float:
        return 4.0 * self.B * self.H * self.Nq * self.Nk * self.d

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "Nq": self.Nq, "Nk": self.Nk, "d": self.d,
                "dtype": self.dtype, "causal": self.causal}


DECODE_WORKLOADS = {
    "decode_b8h32_nq1_nk32768_d128_bf16": DecodeWorkload("decode_b8h32_nq1_nk32768_d128_bf16", 8, 32, 1, 32768,
                                                         128, "bf16", False, 2001),
    "decode_b4h32_nq4_nk8192_d128_bf16_causal": DecodeWorkload("decode_b4h32_nq4_nk8192_d128_bf16_causal", 4, 32,
                                                               4, 8192, 128, "bf16", True, 2002),
}


def make_decode(w: DecodeWorkload):
    q, k, v, _ = make_qkv(w.B, w.H, w.Nq, w.d, w.dtype, w.seed, Nk=w.Nk)
    return q, k, v


def make_qkv(B, H, N, d, dtype="bf16", seed=0, mul=1.0, k_offset=0.0, mask_frac=0.0, full_row_frac=0.0,
             Nk: Optional[int] = None):
    """Draw (q, k, v, mask_or_None) on the CPU following the recipe above.

    ``Nk`` (default N) sets the key/value length; the mask, if any, is [B, N, Nk].
    """
    Nk = N if Nk is None else Nk
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    if k_offset:
        off = (torch.rand((B, H, Nk, 1), generator=g, dtype=torch.float32) * 2.0 - 1.0) * k_offset
        k = k + off
    mask = None
    if mask_frac > 0.0 or full_row_frac > 0.0:
        drop = torch.rand((B, N, Nk), generator=g, dtype=torch.float32) < mask_frac
        mask = torch.zeros((B, N, Nk), dtype=torch.float32)
        mask[drop] = float("-inf")
        nfull = int(round(full_row_frac * N))
        for b in range(B):
            rows = torch.randperm(N, generator=g)[:nfull]
            mask[b, rows, :] = float("-inf")
    if mul != 1.0:
        q, k, v = q * mul, k * mul, v * mul
    t = DTYPES[dtype]
    return q.to(t).contiguous(), k.to(t).contiguous(), v.to(t).contiguous(), mask


def make_workload(w: Workload):
    """(q, k, v, mask_or_None) on the CPU for a named workload."""
    return make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.mul, w.k_offset, w.mask_frac, w.full_row_frac)


def sample_rows(total_rows: int, n: int, seed: int = 0) -> torch.Tensor:
    """n distinct flat row ids in [0, total_rows), sorted, from a seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    n = min(n, total_rows)
    return torch.randperm(total_rows, generator=g)[:n].sort().values


# ---------------------------------------------------------------- backward workloads
# The backward measurement of "IO-aware exact attention" (section "Backward
# recomputation", its stored-state vs recomputed exercise): batch 2, 16 heads,
# head dimension 64, sequence lengths 512 to 4096, identical inputs and loss
# gradients for every path.
@dataclass(frozen=True)
class BwdWorkload:
    B: int
    H: int
    N: int
    d: int
    dtype: str = "bf16"
    causal: bool = False
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        """Matrix flops of the recomputing backward: five N x N x d products
        (S, dP, dV, dK, dQ), halved when causal."""
        f = 5 * 2.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def describe(self) -> dict:
        return {"B": self.B, "H": self.H, "N": self.N, "d": self.d, "dtype": self.dtype, "causal": self.causal}


BWD_WORKLOADS = {
    f"bwd_b2h16_n{n}_d64_bf16": BwdWorkload(2, 16, n, 64, "bf16", False, seed=400 + n)
    for n in (512, 1024, 2048, 4096)
}
BWD_WORKLOADS["bwd_b2h16_n4096_d64_bf16_causal"] = BwdWorkload(2, 16, 4096, 64, "bf16", True, seed=8300)
BWD_WORKLOADS["bwd_b1h32_n8192_d128_bf16_causal"] = BwdWorkload(1, 32, 8192, 128, "bf16", True, seed=8301)


def make_bwd(B, H, N, d, dtype="bf16", seed=0):
    """(q, k, v, dout) on the CPU: one CPU generator seeded with ``seed`` draws
    fp32 standard normals for Q, K, V and then the loss gradient dO, each
    [B, H, N, d], rounded to the storage dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    t = DTYPES[dtype]
    out = []
    for _ in range(4):
        out.append(torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(t).contiguous())
    return tuple(out)


# ---------------------------------------------------------------- packed variable-length batches
def varlen_lengths(total_tokens, lo, hi, seed):
    """Sequence lengths for a packed batch: a CPU generator seeded with ``seed``
    draws log-uniform lengths in [lo, hi] until their sum reaches total_tokens;
    the last length is cut so that the lengths sum to exactly total_tokens."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out, acc = [], 0
    while acc < total_tokens:
        u = float(torch.rand((), generator=g))
        L = int(round(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))))
        L = min(L, total_tokens - acc)
        out.append(L)
        acc += L
    return out


def make_varlen(lengths, H, Hkv, d, dtype="bf16", seed=0):
    """(q [total, H, d], k [total, Hkv, d], v [total, Hkv, d], cu_seqlens int32 [nseq + 1]) on the CPU:
    fp32 standard normals drawn in the order q, k, v by a generator seeded with ``seed``, rounded to dtype."""
    total = int(sum(lengths))
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    t = DTYPES[dtype]
    q = torch.randn((total, H, d), generator=g, dtype=torch.float32).to(t).contiguous()
    k = torch.randn((total, Hkv, d), generator=g, dtype=torch.float32).to(t).contiguous()
    v = torch.randn((total, Hkv, d), generator=g, dtype=torch.float32).to(t).contiguous()
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return q, k, v, cu


@dataclass(frozen=True)
class VarlenWorkload:
    total: int
    lo: int
    hi: int
    H: int
    d: int
    dtype: str = "bf16"
    causal: bool = True
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def lengths(self):
        return varlen_lengths(self.total, self.lo, self.hi, self.seed)

    def flops(self) -> float:
        f = sum(4.0 * L * L * self.d * self.H for L in self.lengths())
        return f / 2 if self.causal else f

    def describe(self) -> dict:
        L = self.lengths()
        return {"total_tokens": self.total, "nseq": len(L), "len_min": min(L), "len_max": max(L),
                "len_mix": f"log-uniform [{self.lo}, {self.hi}]", "H": self.H, "d": self.d, "dtype": self.dtype,
                "causal": self.causal}


VARLEN_WORKLOADS = {
    "varlen_t65536_h32_d128_bf16_causal": VarlenWorkload(65536, 256, 8192, 32, 128, "bf16", True, seed=7100),
}


# ---------------------------------------------------------------- grouped-query attention
@dataclass(frozen=True)
class GqaWorkload:
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    dtype: str = "bf16"
    causal: bool = True
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def describe(self) -> dict:
        return {"B": self.B, "H": self.H, "Hkv": self.Hkv, "N": self.N, "d": self.d, "dtype": self.dtype,
                "causal": self.causal}


GQA_WORKLOADS = {
    "gqa_b1h32kv8_n8192_d128_bf16_causal": GqaWorkload(1, 32, 8, 8192, 128, "bf16", True, seed=7200),
}


def make_gqa(w: GqaWorkload):
    """(q [B, H, N, d], k, v [B, Hkv, N, d]) on the CPU: q drawn by make_qkv with the workload's
    seed, then k and v by make_qkv with seed + 1 (fp32 normals rounded to the dtype)."""
    q, _, _, _ = make_qkv(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed)
    _, k, v, _ = make_qkv(w.B, w.Hkv, w.N, w.d, w.dtype, seed=w.seed + 1)
    return q, k, v
