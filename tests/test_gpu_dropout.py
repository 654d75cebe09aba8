"""GPU parity of the forward with dropout (``fa_fwd_dropout``) against the fp64
oracle, which draws the same keep decisions from its own Philox4x64-10 (the two
share no code: the kernel and the oracle each implement the published generator).

The keep pattern itself is checked exactly: with V the identity (N = d) every
output entry is its key's weight, which is 0 exactly when the key was dropped.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_13_gb300.inputs import make_qkv
from parity_util import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def run(fa, q, k, v, scale, causal, p_drop, seed, offset=0):
    B, H, N, d = q.shape
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fn = fa.fa_fwd_dropout if q.dtype == torch.bfloat16 else fa.fa_fwd_dropout_fp16
    fn(q.to(DEV), k.to(DEV), v.to(DEV), out, lse, scale, causal, p_drop, seed, offset)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return out, lse


CASES = [
    # B, H, Hkv, N, d, dtype, causal, p
    (1, 2, 2, 300, 128, "bf16", False, 0.1),
    (2, 2, 2, 257, 64, "fp16", True, 0.3),
    (1, 3, 3, 1000, 128, "bf16", True, 0.5),
    (2, 4, 2, 200, 128, "bf16", False, 0.2),  # grouped-query
    (1, 2, 2, 128, 64, "bf16", False, 0.9),
    (1, 1, 1, 1, 128, "fp16", False, 0.25),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,dtype,causal,p", CASES)
def test_dropout_matches_oracle(fa, B, H, Hkv, N, d, dtype, causal, p):
    q, _, _, _ = make_qkv(B, H, N, d, dtype, seed=N + H + 3)
    _, k, v, _ = make_qkv(B, Hkv, N, d, dtype, seed=N + Hkv + 4)
    seed, offset = 1234567 + N, 3
    scale = 1 / math.sqrt(d)
    out, lse = run(fa, q, k, v, scale, causal, p, seed, offset)
    g = H // Hkv
    ref_o, ref_l = oracle.attention_dropout(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1), p, seed,
                                            offset, scale=scale, causal=causal)
    # 1 / q up to 10 scales the probabilities; the tolerance grows with it
    qk = oracle.dropout_threshold(p) / 256
    compare(out, lse, ref_o, ref_l, o_max=2e-2 / qk, o_mean=2e-3 / qk)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_probability_is_plain_attention(fa, causal):
    q, k, v, _ = make_qkv(2, 3, 700, 128, "bf16", seed=8)
    o1, l1 = run(fa, q, k, v, 0.09, causal, 0.0, seed=99)
    o2, l2 = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), scale=0.09, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_is_undropped_and_calls_repeat(fa):
    q, k, v, _ = make_qkv(1, 2, 500, 64, "fp16", seed=9)
    o1, l1 = run(fa, q, k, v, 0.125, True, 0.4, seed=5, offset=10)
    o2, l2 = run(fa, q, k, v, 0.125, True, 0.4, seed=5, offset=10)
    o3, l3 = run(fa, q, k, v, 0.125, True, 0.4, seed=5, offset=11)
    _, l0 = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)   # same (seed, offset): same pattern
    assert not torch.equal(o1, o3) and torch.equal(l1, l3)
    assert torch.equal(l1, l0)


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "fp16")])
def test_keep_pattern_exactly(fa, d, dtype):
    """V = I with N = d: out[b, h, i, j] is key j's weight, zero exactly where the oracle's
    stream drops (b, h, i, j) (scores are kept small, so no kept weight underflows)."""
    B, H, N = 2, 2, d
    q, k, _, _ = make_qkv(B, H, N, d, dtype, seed=21)
    v = torch.eye(N, dtype=q.dtype).expand(B, H, N, N).contiguous()
    p, seed, offset = 0.3, 2**40 + 17, 2**33 + 5
    out, _ = run(fa, q, k, v, 0.05, False, p, seed, offset)
    keep = oracle.dropout_keep(B, H, N, N, p, seed, offset)
    got = out.float().cpu().numpy() != 0.0
    assert np.array_equal(got, keep), f"{int((got != keep).sum())} keep decisions differ"


def test_dropout_writes_stay_inside_their_buffers(fa):
    """Guard bands around O and lse stay untouched (ragged N against the 128-key blocks)."""
    B, H, N, d = 1, 3, 333, 128
    q, k, v, _ = make_qkv(B, H, N, d, "bf16", seed=21)
    pad = 4096
    obuf = torch.full((B * H * N * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    lbuf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    out = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd_dropout(q.to(DEV), k.to(DEV), v.to(DEV), out, lse, 0.1, True, 0.2, 77, 5)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert bool((obuf[:pad] == 7.0).all()) and bool((obuf[-pad:] == 7.0).all())
    assert bool((lbuf[:pad] == 7.0).all()) and bool((lbuf[-pad:] == 7.0).all())
    ref_o, ref_l = oracle.attention_dropout(q, k, v, 0.2, 77, 5, scale=0.1, causal=True)
    qk = oracle.dropout_threshold(0.2) / 256
    compare(out, lse, ref_o, ref_l, o_max=2e-2 / qk, o_mean=2e-3 / qk)
