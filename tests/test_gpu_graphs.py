"""CUDA graph capture of the library's launches.

A serving loop captures its attention calls once and replays them. The
forward, the masked forward with its packing pass (whose fp32-mask kernel is a
programmatic dependent of the 128-key kernel), the forward with dropout, the
split-KV decode (whose merge kernel is a programmatic dependent of the split
kernel) and the backward (three kernels chained by programmatic dependent
launch) are captured here, fed new inputs in the same buffers and
replayed; the results must equal those of eager calls on the same inputs (bit
for bit where the kernels are deterministic, and up to the order of the fp32 dQ
reductions for dQ).
"""
import math

import pytest
import torch

from io_aware_exact_13_gb300.inputs import make_bwd, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # first call outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _refill(dst, seed, shape, dtype="bf16"):
    src = make_qkv(*shape, dtype, seed=seed)[:3]
    for d, s in zip(dst, src):
        d.copy_(s)


def test_forward_graph_replay(fa):
    dev = torch.device("cuda")
    shape = (1, 4, 1000, 128)
    qd, kd, vd = (t.to(dev) for t in make_qkv(*shape, "bf16", seed=31)[:3])
    out = torch.empty_like(qd)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    g = _capture(lambda: fa.attention(qd, kd, vd, causal=True, out=out, lse=lse))
    _refill((qd, kd, vd), 32, shape)
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = fa.attention(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_splitkv_graph_replay(fa):
    dev = torch.device("cuda")
    B, H, Nq, Nk, d = 2, 8, 4, 3000, 128
    q, k, v, _ = make_qkv(B, H, Nq, d, "bf16", seed=41, Nk=Nk)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    n_splits = fa.fa_splitkv_num_splits(B, H, Nq, Nk, d)
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits), dtype=torch.uint8, device=dev)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    scale = 1 / math.sqrt(d)
    g = _capture(lambda: fa.fa_fwd_splitkv(qd, kd, vd, out, lse, scale, True, n_splits, ws))
    q2, k2, v2, _ = make_qkv(B, H, Nq, d, "bf16", seed=42, Nk=Nk)
    qd.copy_(q2), kd.copy_(k2), vd.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = torch.empty_like(out), torch.empty_like(lse)
    ws2 = torch.empty_like(ws)
    fa.fa_fwd_splitkv(qd, kd, vd, ref_o, ref_l, scale, True, n_splits, ws2)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_graph_replay(fa, d):
    dev = torch.device("cuda")
    B, H, N = 1, 4, 700
    q, k, v, do = (t.to(dev) for t in make_bwd(B, H, N, d, "bf16", seed=51 + d))
    scale = 1 / math.sqrt(d)
    o, lse = fa.attention(q, k, v, scale=scale, causal=True)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    g = _capture(lambda: fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, True, ws))
    do.copy_(make_bwd(B, H, N, d, "bf16", seed=61 + d)[3])  # a new upstream gradient
    g.replay()
    torch.cuda.synchronize()
    rq, rk, rv = fa.attention_backward(q, k, v, o, do, lse, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(dk, rk) and torch.equal(dv, rv)
    err = (dq.float() - rq.float()).abs().max().item()
    assert err <= 1e-2 * rq.float().abs().max().item(), err


@pytest.mark.parametrize("other_values", [False, True])
def test_masked_forward_graph_replay(fa, other_values):
    """fa_fwd_masked: verdict reset, packing pass, the 128-key kernel and its programmatic dependent (the
    fp32-mask kernel) captured together; a new mask in the same buffer is packed by the replay. With
    other_values the replayed mask has a 0.5 in it, so the replay takes the fp32-mask kernel."""
    dev = torch.device("cuda")
    B, H, N, d = 2, 3, 520, 128
    q, k, v, m1 = (t.to(dev) for t in make_qkv(B, H, N, d, "fp16", seed=71, mask_frac=0.2, full_row_frac=0.02))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_fwd_masked_workspace_bytes(B, N), dtype=torch.uint8, device=dev)
    g = _capture(lambda: fa.fa_fwd_masked_fp16(q, k, v, m1, out, lse, 0.1, False, ws))
    m2 = make_qkv(B, H, N, d, "fp16", seed=72, mask_frac=0.3)[3].to(dev)
    if other_values:
        m2[1, 7, 11] = 0.5
    m1.copy_(m2)
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = torch.empty_like(out), torch.empty_like(lse)
    fa.fa_fwd_masked_fp16(q, k, v, m2, ref_o, ref_l, 0.1, False, torch.empty_like(ws))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_dropout_graph_replay(fa):
    dev = torch.device("cuda")
    shape = (1, 4, 900, 64)
    qd, kd, vd = (t.to(dev) for t in make_qkv(*shape, "bf16", seed=81)[:3])
    out = torch.empty_like(qd)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    g = _capture(lambda: fa.fa_fwd_dropout(qd, kd, vd, out, lse, 0.125, True, 0.2, 1234, 5))
    _refill((qd, kd, vd), 82, shape)
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = fa.attention_dropout(qd, kd, vd, 0.2, 1234, 5, scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
