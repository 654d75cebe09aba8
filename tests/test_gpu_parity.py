"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Element-by-element on small and ragged shapes (several tiles plus a tail), and on
sampled rows plus whole-tensor properties at the five full workload sizes, in
the launch configuration the benchmark times.
"""
import math

import pytest
import torch

import oracle
from io_aware_exact_13_gb300.inputs import WORKLOADS, make_qkv, make_workload
from parity_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def run(fa, q, k, v, mask, scale, causal, stream=None):
    dev = torch.device("cuda")
    out, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), mask=None if mask is None else mask.to(dev),
                            scale=scale, causal=causal, stream=stream)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return out, lse


SMALL = [
    # B, H, N, d, dtype, causal, masked
    (1, 1, 1, 128, "bf16", False, False),
    (1, 1, 3, 64, "bf16", True, False),
    (1, 2, 127, 128, "bf16", True, False),
    (1, 2, 128, 128, "bf16", False, False),
    (2, 1, 129, 64, "bf16", False, False),
    (1, 3, 200, 128, "bf16", True, False),
    (1, 1, 255, 128, "fp16", True, False),
    (2, 2, 256, 128, "bf16", True, False),
    (1, 2, 257, 64, "fp16", False, False),
    (2, 3, 384, 128, "bf16", True, False),
    (1, 2, 1000, 128, "bf16", True, False),
    (1, 2, 1000, 64, "bf16", False, False),
    (1, 63, 1024, 64, "bf16", False, False),  # 252 two-tile items: last wave too full to cut into single tiles
    (2, 2, 300, 128, "fp16", False, True),
    (1, 3, 513, 128, "bf16", True, True),
    (2, 2, 260, 64, "fp16", True, True),
    (1, 2, 20, 128, "bf16", False, True),   # mask by TMA: every box reaches past N (zero fill)
    (2, 1, 68, 64, "bf16", True, True),     # mask by TMA: second key block ragged, rows past N in the tile
    (1, 1, 256, 64, "fp32", False, False),
    (1, 2, 300, 64, "fp32", True, False),
    (1, 2, 200, 64, "fp32", False, True),
    (1, 2, 300, 128, "fp32", True, False),   # d = 128 on the fp32 path: causal, ragged tail
    (2, 1, 200, 128, "fp32", False, True),   # masked, rows fully masked
    (1, 2, 129, 128, "fp32", True, True),    # causal and masked together, one row past a block
    (1, 1, 1, 128, "fp32", False, False),    # a single row and key
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,masked", SMALL)
def test_small_shapes_elementwise(fa, B, H, N, d, dtype, causal, masked):
    q, k, v, mask = make_qkv(B, H, N, d, dtype, seed=17 * N + d + B, mask_frac=0.2 if masked else 0.0,
                             full_row_frac=0.02 if masked else 0.0)
    scale = 1.0 / math.sqrt(d)
    out, lse = run(fa, q, k, v, mask, scale, causal)
    ref_o, ref_l = oracle.attention(q, k, v, mask=mask, scale=scale, causal=causal)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_workloads_every_row(fa, name):
    """Full-size launch, every output row against the oracle (its fp64 run over all
    rows takes seconds to about half a minute of host time per workload), and
    whole-tensor properties on top."""
    w = WORKLOADS[name]
    q, k, v, mask = make_workload(w)
    out, lse = run(fa, q, k, v, mask, w.scale, w.causal)
    ref_o, ref_l = oracle.attention(q, k, v, mask=mask, scale=w.scale, causal=w.causal)
    compare(out, lse, ref_o, ref_l)
    # properties on every row: finite, and each O row is a convex combination of V rows
    of = out.float()
    assert not torch.isnan(of).any() and not torch.isinf(of).any()
    vmax = v.float().to(out.device).amax(dim=2, keepdim=True)
    vmin = v.float().to(out.device).amin(dim=2, keepdim=True)
    slack = 2e-2
    assert bool((of <= vmax + slack).all()) and bool((of >= vmin - slack).all())
    if mask is None:
        assert bool(torch.isfinite(lse).all())
    else:
        fully = torch.isneginf(mask.to(lse.device)).all(dim=-1)  # [B, N]
        assert torch.equal(torch.isneginf(lse), fully[:, None, :].expand_as(lse))


def test_deterministic_bits(fa):
    q, k, v, _ = make_qkv(1, 4, 1536, 128, "bf16", seed=5)
    o1, l1 = run(fa, q, k, v, None, 0.09, True)
    o2, l2 = run(fa, q, k, v, None, 0.09, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_mean_of_values(fa, causal):
    q, k, v, _ = make_qkv(1, 2, 333, 64, "bf16", seed=6)
    out, lse = run(fa, q, k, v, None, 0.0, causal)
    vf = v.double()
    if causal:
        ref = vf.cumsum(dim=2) / torch.arange(1, 334, dtype=torch.float64).view(1, 1, -1, 1)
        ref_l = torch.log(torch.arange(1, 334, dtype=torch.float64)).view(1, 1, -1).expand(1, 2, 333)
    else:
        ref = vf.mean(dim=2, keepdim=True).expand_as(vf)
        ref_l = torch.full((1, 2, 333), math.log(333.0), dtype=torch.float64)
    compare(out, lse, ref.numpy(), ref_l.numpy())


def test_negative_scale(fa):
    q, k, v, _ = make_qkv(1, 2, 300, 128, "bf16", seed=8)
    out, lse = run(fa, q, k, v, None, -0.1, False)
    ref_o, ref_l = oracle.attention(q, k, v, scale=-0.1)
    compare(out, lse, ref_o, ref_l)


def test_large_score_range_rescaling(fa):
    """Scores spread over a range far beyond the lazy-rescale threshold."""
    q, k, v, _ = make_qkv(1, 2, 1024, 128, "bf16", seed=9, k_offset=30.0)
    out, lse = run(fa, q, k, v, None, 0.25, True)
    ref_o, ref_l = oracle.attention(q, k, v, scale=0.25, causal=True)
    compare(out, lse, ref_o, ref_l)


def test_outputs_stay_inside_their_buffers(fa):
    """Guard bands around O and lse stay untouched (no out-of-bounds writes)."""
    B, H, N, d = 1, 3, 333, 128
    q, k, v, _ = make_qkv(B, H, N, d, "bf16", seed=10)
    dev = torch.device("cuda")
    pad = 4096
    obuf = torch.full((B * H * N * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device=dev)
    out = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), None, out, lse, 1 / math.sqrt(d), True)
    torch.cuda.synchronize()
    assert bool((obuf[:pad] == 7.0).all()) and bool((obuf[-pad:] == 7.0).all())
    assert bool((lbuf[:pad] == 7.0).all()) and bool((lbuf[-pad:] == 7.0).all())
    ref_o, ref_l = oracle.attention(q, k, v, scale=1 / math.sqrt(d), causal=True)
    compare(out, lse, ref_o, ref_l)


def test_side_stream_and_no_allocation(fa):
    q, k, v, _ = make_qkv(1, 2, 700, 128, "bf16", seed=11)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((1, 2, 700), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s):
        fa.fa_fwd(qd, kd, vd, None, out, lse, 0.1, False, stream=s)
    s.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 == free1, "the library must not allocate device memory"
    ref_o, ref_l = oracle.attention(q, k, v, scale=0.1)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("d", [64, 128])
def test_back_to_back_calls_that_read_each_others_outputs(fa, d):
    """The 128-key forward is launched as a programmatic dependent of the work ahead of it and may start
    before that work ends; it must read nothing in global memory until it has. Three forwards are queued
    with no synchronisation, each reading the one before's output (O as the next Q, then as K and V),
    into buffers first filled with a sentinel far from any attention output: a read that came early would
    see it. Each result is compared with the oracle on the GPU's own inputs."""
    B, H, N = 1, 4, 700
    q, k, v, _ = make_qkv(B, H, N, d, "bf16", seed=70 + d)
    dev = torch.device("cuda")
    scale = 1 / math.sqrt(d)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    outs = [torch.full((B, H, N, d), 300.0, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    lses = [torch.full((B, H, N), 300.0, dtype=torch.float32, device=dev) for _ in range(3)]
    fa.fa_fwd(qd, kd, vd, None, outs[0], lses[0], scale, True)
    fa.fa_fwd(outs[0], kd, vd, None, outs[1], lses[1], scale, True)
    fa.fa_fwd(outs[1], outs[0], outs[0], None, outs[2], lses[2], scale, False)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o0, o1 = outs[0].cpu(), outs[1].cpu()
    for (qi, ki, vi, causal), o, l in zip([(q, k, v, True), (o0, k, v, True), (o1, o0, o0, False)], outs, lses):
        ref_o, ref_l = oracle.attention(qi, ki, vi, scale=scale, causal=causal)
        compare(o, l, ref_o, ref_l)
