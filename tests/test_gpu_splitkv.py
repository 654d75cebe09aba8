"""GPU parity of the split-KV decoding forward against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_13_gb300.inputs import DECODE_WORKLOADS, make_decode, make_qkv
from parity_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def run(fa, q, k, v, causal, n_splits=None, scale=None):
    dev = torch.device("cuda")
    out, lse = fa.attention_decode(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal, n_splits=n_splits)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # B, H, Nq, Nk, d, dtype, causal, n_splits
    (1, 1, 1, 1, 128, "bf16", False, 1),
    (1, 2, 1, 100, 64, "bf16", False, 3),
    (2, 3, 3, 1000, 128, "bf16", False, None),
    (2, 2, 16, 777, 128, "fp16", False, 7),
    (1, 4, 5, 4096, 64, "fp16", True, None),
    (2, 2, 16, 20, 128, "bf16", True, 20),   # many empty splits for the early rows
    (1, 2, 9, 5000, 128, "bf16", True, 13),
    (3, 1, 2, 300, 64, "bf16", False, 300),  # one key per split
    (1, 2, 12, 2000, 64, "bf16", True, None),  # 16-row variant at d = 64 (16 lanes per key row)
    (2, 2, 4, 8192, 128, "bf16", True, None),  # the four-row decode shape, 8-lane groups
]


@pytest.mark.parametrize("Nq,d", [(1, 128), (4, 128), (8, 64), (16, 128)])
def test_splitkv_growing_scores_rescale(fa, Nq, d):
    """Large scores whose running maximum keeps growing along the keys (Q and K
    scaled by 3, K rows offset by up to +-4) exercise the lazy rescaling; V stays
    unit-scale so that the absolute tolerance keeps its meaning."""
    q, k, _, _ = make_qkv(1, 2, Nq, d, "bf16", seed=50 + Nq, mul=3.0, k_offset=4.0, Nk=6000)
    _, _, v, _ = make_qkv(1, 2, Nq, d, "bf16", seed=60 + Nq, Nk=6000)
    out, lse = run(fa, q, k, v, False, 5)
    ref_o, ref_l = oracle.attention(q, k, v, scale=1 / math.sqrt(d), causal=False)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal,n_splits", CASES)
def test_splitkv_small(fa, B, H, Nq, Nk, d, dtype, causal, n_splits):
    q, k, v, _ = make_qkv(B, H, Nq, d, dtype, seed=Nk + 31 * Nq + d, Nk=Nk)
    out, lse = run(fa, q, k, v, causal, n_splits)
    ref_o, ref_l = oracle.attention(q, k, v, scale=1 / math.sqrt(d), causal=causal)
    compare(out, lse, ref_o, ref_l)


def test_split_count_does_not_change_the_result(fa):
    q, k, v, _ = make_qkv(2, 4, 4, 128, "bf16", seed=3, Nk=3000)
    outs = [run(fa, q, k, v, False, n) for n in (1, 2, 5, 64, 3000)]
    for o, l in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (l - outs[0][1]).abs().max().item() <= 1e-3


def test_fully_hidden_rows(fa):
    # causal with Nq > Nk: the first Nq - Nk rows see no key at all
    q, k, v, _ = make_qkv(1, 2, 8, 64, "bf16", seed=4, Nk=5)
    out, lse = run(fa, q, k, v, True, 2)
    ref_o, ref_l = oracle.attention(q, k, v, scale=1 / 8, causal=True)
    compare(out, lse, ref_o, ref_l)
    assert bool(torch.isneginf(lse[:, :, :3]).all())


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_workloads(fa, name):
    w = DECODE_WORKLOADS[name]
    q, k, v = make_decode(w)
    out, lse = run(fa, q, k, v, w.causal)
    ref_o, ref_l = oracle.attention(q, k, v, scale=w.scale, causal=w.causal)
    compare(out, lse, ref_o, ref_l)


def test_workspace_checks(fa):
    q, k, v, _ = make_qkv(1, 2, 2, 64, "bf16", seed=5, Nk=256)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((1, 2, 2), dtype=torch.float32, device=dev)
    need = fa.fa_splitkv_workspace_bytes(1, 2, 2, 64, 4)
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_splitkv(qd, kd, vd, out, lse, 0.125, False, 4, small)
    assert e.value.status == fa.FA_ERR_WORKSPACE
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    fa.fa_fwd_splitkv(qd, kd, vd, out, lse, 0.125, False, 4, ws)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(q, k, v, scale=0.125)
    compare(out, lse, ref_o, ref_l)
