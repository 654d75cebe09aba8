"""GPU parity of grouped-query attention: the oracle sees K/V repeated per query head."""
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


@pytest.mark.parametrize("B,H,Hkv,N,d,dtype,causal", [
    (1, 8, 2, 1000, 128, "bf16", True),
    (2, 6, 3, 513, 64, "fp16", False),
    (1, 4, 1, 777, 128, "bf16", False),  # one K/V head for all query heads
    (2, 4, 4, 300, 128, "bf16", True),   # Hkv = H is plain attention
])
def test_gqa_matches_repeated_heads(fa, B, H, Hkv, N, d, dtype, causal):
    q, _, _, _ = make_qkv(B, H, N, d, dtype, seed=N + H)
    _, k, v, _ = make_qkv(B, Hkv, N, d, dtype, seed=N + Hkv + 1)
    dev = torch.device("cuda")
    out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fn = fa.fa_fwd_gqa if dtype == "bf16" else fa.fa_fwd_gqa_fp16
    fn(q.to(dev), k.to(dev), v.to(dev), None, out, lse, 1 / math.sqrt(d), causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    g = H // Hkv
    ref_o, ref_l = oracle.attention(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1),
                                    scale=1 / math.sqrt(d), causal=causal)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("N,causal", [(300, False), (260, True), (517, False)])
def test_gqa_with_additive_mask(fa, N, causal):
    """Grouped-query attention with an additive [B,N,N] mask (shared by all heads of a batch index;
    N % 4 == 0 takes the TMA mask copies, 517 the direct loads)."""
    B, H, Hkv, d = 2, 6, 2, 128
    q, _, _, mask = make_qkv(B, H, N, d, "bf16", seed=N + 5, mask_frac=0.2, full_row_frac=0.02)
    _, k, v, _ = make_qkv(B, Hkv, N, d, "bf16", seed=N + 6)
    dev = torch.device("cuda")
    out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), mask.to(dev), out, lse, 1 / math.sqrt(d), causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    g = H // Hkv
    ref_o, ref_l = oracle.attention(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1), mask=mask,
                                    scale=1 / math.sqrt(d), causal=causal)
    compare(out, lse, ref_o, ref_l)


def test_gqa_workload_every_head(fa):
    """The benchmark's grouped-query workload in the benchmark's launch; every
    query head against the oracle with its K/V head repeated."""
    from io_aware_exact_13_gb300.inputs import GQA_WORKLOADS, make_gqa

    w = GQA_WORKLOADS["gqa_b1h32kv8_n8192_d128_bf16_causal"]
    q, k, v = make_gqa(w)
    dev = torch.device("cuda")
    out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    fa.fa_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), None, out, lse, w.scale, w.causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    g = w.H // w.Hkv
    ref_o, ref_l = oracle.attention(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1), scale=w.scale,
                                    causal=w.causal)
    compare(out, lse, ref_o, ref_l)
