"""GPU parity of the backward by recomputation against the fp64 oracle's gradients.

The oracle's backward is pinned to central finite differences of its forward
(test_oracle_pins). Here the CUDA backward gets the same q, k, v, dO and either
the oracle's O (rounded to the storage type) and lse, or the CUDA forward's,
and dQ, dK, dV are compared with the oracle's fp64 gradients.

Tolerance, from the arithmetic: P and dS are rounded once to the 16-bit input
type before their products (relative error 2^-9 for bf16, 2^-11 for fp16), the
products accumulate in fp32, and D = rowsum(dO o O) uses O as stored (16 bit).
Each gradient element is a sum of such rounded terms, so its error is a small
multiple of 2^-9 times the sum of the terms' magnitudes; over whole tensors we
bound the normwise relative error ||got - ref|| / ||ref|| by 1e-2 and the
largest element error by 2e-2 of the tensor's largest magnitude.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_13_gb300.inputs import BWD_WORKLOADS, DTYPES, make_bwd

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
REL_MAX = 2e-2


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def _cmp(name, got, ref):
    g = got.float().cpu().double().numpy()
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = np.abs(g - r)
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    mx = float(err.max() / max(np.abs(r).max(), 1e-30))
    stats = {"tensor": name, "rel_fro": fro, "rel_max": mx}
    assert fro <= REL_FRO, stats
    assert mx <= REL_MAX, stats
    return stats


def _run_bwd(fa, q, k, v, o, do, lse, scale, causal):
    dev = torch.device("cuda")
    args = [t.to(dev) for t in (q, k, v, o, do)]
    dq, dk, dv = fa.attention_backward(*args[:4], args[4], lse.to(dev), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return dq, dk, dv


SMALL = [
    (1, 2, 128, 64, "bf16", False),    # one key block, one query block
    (1, 2, 300, 128, "bf16", True),    # ragged tail, causal diagonal blocks
    (2, 3, 517, 64, "fp16", True),
    (1, 2, 1000, 128, "bf16", False),  # several blocks, ragged
    (2, 2, 256, 64, "bf16", True),     # exact multiple of the block
    (1, 1, 1, 128, "bf16", False),     # a single row and key
    (1, 1, 129, 64, "fp16", False),    # one row past a block
    (1, 2, 700, 128, "fp16", True),    # d = 128 in fp16: causal, ragged tail
    (2, 1, 640, 128, "fp16", False),   # d = 128 in fp16: five query blocks, the two-stage ring wraps
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", SMALL)
def test_bwd_matches_oracle_given_oracle_forward(fa, B, H, N, d, dtype, causal):
    q, k, v, do = make_bwd(B, H, N, d, dtype, seed=7 * N + d + H)
    scale = 1 / math.sqrt(d)
    ref_o, ref_l = oracle.attention(q, k, v, scale=scale, causal=causal)
    o = torch.from_numpy(ref_o).to(DTYPES[dtype])
    lse = torch.from_numpy(ref_l).float()
    dq, dk, dv = _run_bwd(fa, q, k, v, o, do, lse, scale, causal)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale=scale, causal=causal)
    _cmp("dq", dq, rq)
    _cmp("dk", dk, rk)
    _cmp("dv", dv, rv)


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [(1, 2, 777, 128, "bf16", True), (2, 2, 640, 64, "fp16", False)])
def test_forward_then_backward_matches_oracle(fa, B, H, N, d, dtype, causal):
    """The training path: CUDA forward (O, lse) feeds the CUDA backward."""
    q, k, v, do = make_bwd(B, H, N, d, dtype, seed=N + 11)
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    dq, dk, dv = _run_bwd(fa, q, k, v, o.cpu(), do, lse.cpu(), scale, causal)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale=scale, causal=causal)
    _cmp("dq", dq, rq)
    _cmp("dk", dk, rk)
    _cmp("dv", dv, rv)


def test_bwd_scale_zero_uniform_probabilities(fa):
    """scale = 0: P is uniform over the visible keys, so dQ = dK = 0 and
    dV_j = (1/N) sum_i dO_i for every key (non-causal)."""
    B, H, N, d = 1, 2, 384, 64
    q, k, v, do = make_bwd(B, H, N, d, "bf16", seed=5)
    ref_o, ref_l = oracle.attention(q, k, v, scale=0.0)
    dq, dk, dv = _run_bwd(fa, q, k, v, torch.from_numpy(ref_o).bfloat16(), do, torch.from_numpy(ref_l).float(),
                          0.0, False)
    assert torch.count_nonzero(dq) == 0 and torch.count_nonzero(dk) == 0
    mean_do = do.double().mean(dim=2, keepdim=True).expand(B, H, N, d).numpy()
    _cmp("dv", dv, mean_do)


def test_bwd_deterministic_dk_dv(fa):
    """dK and dV come from one CTA each with a fixed order: bitwise repeatable."""
    q, k, v, do = make_bwd(1, 2, 700, 128, "bf16", seed=3)
    dev = torch.device("cuda")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=True)
    a = fa.attention_backward(q.to(dev), k.to(dev), v.to(dev), o, do.to(dev), lse, causal=True)
    b = fa.attention_backward(q.to(dev), k.to(dev), v.to(dev), o, do.to(dev), lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("name", ["bwd_b2h16_n4096_d64_bf16", "bwd_b2h16_n4096_d64_bf16_causal"])
def test_bwd_full_size_every_head(fa, name):
    """Full benchmark size in the benchmark's launch; dQ, dK, dV of every head
    against the oracle's gradients."""
    w = BWD_WORKLOADS[name]
    q, k, v, do = make_bwd(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed)
    dev = torch.device("cuda")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), scale=w.scale, causal=w.causal)
    dq, dk, dv = fa.attention_backward(q.to(dev), k.to(dev), v.to(dev), o, do.to(dev), lse, scale=w.scale,
                                       causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale=w.scale, causal=w.causal)
    _cmp("dq", dq, rq)
    _cmp("dk", dk, rk)
    _cmp("dv", dv, rv)


def test_bwd_full_size_d128_every_head(fa):
    """The d = 128 backward at its benchmark size (B1 H32 N8192 causal), in the
    benchmark's launch; dQ, dK, dV of all 32 heads against the oracle's
    gradients (the fp64 backward over all heads takes about a minute of host
    time)."""
    w = BWD_WORKLOADS["bwd_b1h32_n8192_d128_bf16_causal"]
    q, k, v, do = make_bwd(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed)
    dev = torch.device("cuda")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), scale=w.scale, causal=w.causal)
    dq, dk, dv = fa.attention_backward(q.to(dev), k.to(dev), v.to(dev), o, do.to(dev), lse, scale=w.scale,
                                       causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale=w.scale, causal=w.causal)
    _cmp("dq", dq, rq)
    _cmp("dk", dk, rk)
    _cmp("dv", dv, rv)


def test_bwd_host_validation(fa):
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 64), dtype=torch.float32, device=dev)
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_bwd(q, q, q, q, q, lse, q.clone(), q.clone(), q.clone(), 0.125, False, small)
    assert e.value.status == fa.FA_ERR_WORKSPACE
    q96 = torch.zeros((1, 1, 64, 96), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fa_bwd(q96, q96, q96, q96, q96, lse, q96.clone(), q96.clone(), q96.clone(), 0.1, False, ws)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "fp16")])
def test_bwd_writes_stay_inside_their_buffers(fa, d, dtype):
    """Guard bands around dQ, dK, dV and the workspace stay untouched (N = 333 is ragged against the
    128-row blocks, causal), and the gradients still match the oracle."""
    B, H, N = 2, 2, 333
    q, k, v, do = make_bwd(B, H, N, d, dtype, seed=333 + d)
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda")
    ref_o, ref_l = oracle.attention(q, k, v, scale=scale, causal=True)
    t = DTYPES[dtype]
    o, lse = torch.from_numpy(ref_o).to(t), torch.from_numpy(ref_l).float()
    pad = 4096
    n = B * H * N * d
    bufs = [torch.full((n + 2 * pad,), 7.0, dtype=t, device=dev) for _ in range(3)]
    dq, dk, dv = (b[pad:pad + n].view(B, H, N, d) for b in bufs)
    nws = fa.fa_bwd_workspace_bytes(B, H, N, d)
    wbuf = torch.full((nws + 2 * pad,), 0x5A, dtype=torch.uint8, device=dev)
    ws = wbuf[pad:pad + nws]
    fn = fa.fa_bwd if t == torch.bfloat16 else fa.fa_bwd_fp16
    fn(q.to(dev), k.to(dev), v.to(dev), o.to(dev), do.to(dev), lse.to(dev), dq, dk, dv, scale, True, ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for b in bufs:
        assert bool((b[:pad] == 7.0).all()) and bool((b[-pad:] == 7.0).all())
    assert bool((wbuf[:pad] == 0x5A).all()) and bool((wbuf[-pad:] == 0x5A).all())
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale=scale, causal=True)
    _cmp("dq", dq, rq)
    _cmp("dk", dk, rk)
    _cmp("dv", dv, rv)
