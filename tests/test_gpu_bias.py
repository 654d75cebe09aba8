"""GPU parity of the per-head additive bias forward (fa_fwd_bias, fa_fwd_bias_fp16)
against the oracle's per-head definition, element by element.

Shapes span several tiles and a ragged tail; N % 4 != 0 takes the path in which
each thread reads its row's bias directly, N % 4 == 0 the staged copies. Bias
values are N(0, 1) with a fraction of -inf entries and some rows of some heads
fully masked (output 0, lse -inf)."""
import math

import pytest
import torch

import oracle
from io_aware_exact_13_gb300.inputs import make_qkv
from parity_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def make_bias(B, H, N, seed, minus_inf_frac=0.1, full_rows=2):
    g = torch.Generator().manual_seed(seed)
    bias = torch.randn((B, H, N, N), generator=g, dtype=torch.float32)
    bias[torch.rand((B, H, N, N), generator=g) < minus_inf_frac] = -math.inf
    for b in range(B):
        for h in range(H):
            rows = torch.randperm(N, generator=g)[:full_rows]
            bias[b, h, rows] = -math.inf
    return bias


CASES = [
    # B, H, N, d, dtype, causal
    (1, 2, 200, 128, "bf16", False),
    (2, 3, 333, 64, "fp16", True),
    (1, 2, 516, 128, "fp16", False),   # N % 4 == 0: staged copies, ragged last block
    (2, 2, 130, 64, "bf16", True),     # N % 4 != 0: direct loads
    (1, 4, 1024, 128, "bf16", True),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", CASES)
def test_bias_matches_oracle(fa, B, H, N, d, dtype, causal):
    q, k, v, _ = make_qkv(B, H, N, d, dtype, seed=N + 31 * H + d)
    bias = make_bias(B, H, N, seed=N + 7)
    dev = torch.device("cuda")
    scale = 1 / math.sqrt(d)
    out, lse = fa.attention_bias(q.to(dev), k.to(dev), v.to(dev), bias.to(dev), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention_bias(q, k, v, bias, scale=scale, causal=causal)
    compare(out, lse, ref_o, ref_l)


def test_bias_equal_on_every_head_is_the_shared_mask(fa):
    """A bias that repeats one [B, N, N] mask on every head gives the bits of the shared
    fp32-mask forward without a workspace (the same kernel; only the mask's head
    coordinate differs)."""
    B, H, N, d = 2, 3, 384, 128
    q, k, v, mask = make_qkv(B, H, N, d, "fp16", seed=5, mask_frac=0.1, full_row_frac=0.01)
    dev = torch.device("cuda")
    bias = mask[:, None].expand(B, H, N, N).contiguous()
    o1, l1 = fa.attention_bias(q.to(dev), k.to(dev), v.to(dev), bias.to(dev), scale=0.1, causal=False)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    fa.fa_fwd_fp16(q.to(dev), k.to(dev), v.to(dev), mask.to(dev), o2, l2, 0.1, False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bias_larger_workload_every_row(fa):
    """B=1, H=8, N=2048, d=128, fp16 (x1.5 inputs), 10 % -inf bias entries and fully
    masked rows in every head: every row against the oracle."""
    B, H, N, d = 1, 8, 2048, 128
    q, k, v, _ = make_qkv(B, H, N, d, "fp16", seed=2048, mul=1.5)
    bias = make_bias(B, H, N, seed=99, full_rows=20)
    dev = torch.device("cuda")
    out, lse = fa.attention_bias(q.to(dev), k.to(dev), v.to(dev), bias.to(dev), scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention_bias(q, k, v, bias, scale=1 / math.sqrt(d))
    compare(out, lse, ref_o, ref_l)


def test_bias_host_validation(fa):
    dev = torch.device("cuda")
    q = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((1, 2, 64), dtype=torch.float32, device=dev)
    with pytest.raises(ValueError):
        fa.fa_fwd_bias(q, q, q, torch.zeros((1, 64, 64), device=dev), out, lse, 0.1, False)  # shared-mask shape
    import ctypes

    rc = fa.lib.fa_fwd_bias(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                            ctypes.c_void_p(q.data_ptr()), None, ctypes.c_void_p(out.data_ptr()),
                            ctypes.c_void_p(lse.data_ptr()), 1, 2, 64, 64, ctypes.c_float(0.1), 0, None)
    assert rc == fa.FA_ERR_NULL
