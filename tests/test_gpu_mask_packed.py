"""GPU tests of the masked forward with a workspace (``fa_fwd_masked``): a mask whose
entries are all 0 or -inf is packed to one bit per entry and applied by the
128-key kernel; any other mask is applied as given by the fp32-mask kernel.

Which kernel did the work is visible in the results, because the two kernels
sum in different orders. The packed path gives exactly what the 128-key
kernel gives without a mask (an all-zero mask), or with the same exclusions
expressed as `causal` (a top-left triangle of -inf). The other path gives
exactly what ``fa_fwd`` gives with the same fp32 mask. Both are also compared
with the fp64 oracle.
"""
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


DEV = torch.device("cuda")


def masked(fa, q, k, v, mask, scale, causal, ws_extra=0):
    """fa_fwd_masked with a fresh workspace (filled with garbage first: the call must not depend on it)."""
    B, H, N, d = q.shape
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    ws = torch.full((fa.fa_fwd_masked_workspace_bytes(B, N) + ws_extra,), 0xA5, dtype=torch.uint8, device=DEV)
    fn = fa.fa_fwd_masked if q.dtype == torch.bfloat16 else fa.fa_fwd_masked_fp16
    fn(q.to(DEV), k.to(DEV), v.to(DEV), mask.to(DEV), out, lse, scale, causal, ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return out, lse


def plain(fa, q, k, v, mask, scale, causal):
    """fa_fwd / fa_fwd_fp16 (no workspace: the fp32 mask as given, or no mask)."""
    B, H, N, d = q.shape
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fn = fa.fa_fwd if q.dtype == torch.bfloat16 else fa.fa_fwd_fp16
    fn(q.to(DEV), k.to(DEV), v.to(DEV), None if mask is None else mask.to(DEV), out, lse, scale, causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return out, lse


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [
    (1, 2, 1000, 128, "bf16", False),
    (1, 2, 1000, 128, "bf16", True),
    (2, 3, 517, 64, "fp16", False),   # N % 4 != 0: the mask rows are not 16-byte aligned
    (1, 1, 1, 128, "bf16", False),
])
def test_zero_mask_equals_no_mask_bitwise(fa, B, H, N, d, dtype, causal):
    q, k, v, _ = make_qkv(B, H, N, d, dtype, seed=N + 3 * H)
    mask = torch.zeros((B, N, N), dtype=torch.float32)
    mask[:, ::7, ::3] = -0.0  # negative zeros add nothing either
    o1, l1 = masked(fa, q, k, v, mask, 1 / math.sqrt(d), causal)
    o2, l2 = plain(fa, q, k, v, None, 1 / math.sqrt(d), causal)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("N,d,dtype", [(777, 128, "bf16"), (256, 64, "fp16"), (1300, 64, "bf16")])
def test_triangle_mask_equals_causal_bitwise(fa, N, d, dtype):
    """-inf above the diagonal, causal off == no mask, causal on: the excluded keys contribute
    exact zeros, whole blocks past the diagonal included."""
    B, H = 2, 2
    q, k, v, _ = make_qkv(B, H, N, d, dtype, seed=N + d)
    tri = torch.triu(torch.full((N, N), float("-inf")), diagonal=1)
    mask = tri.expand(B, N, N).contiguous()
    o1, l1 = masked(fa, q, k, v, mask, 0.11, False)
    o2, l2 = plain(fa, q, k, v, None, 0.11, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


PACKED = [
    # B, H, N, d, dtype, causal
    (2, 2, 300, 128, "fp16", False),
    (1, 3, 513, 128, "bf16", True),
    (2, 2, 260, 64, "fp16", True),
    (1, 2, 20, 128, "bf16", False),    # one ragged key block
    (2, 1, 68, 64, "bf16", True),
    (1, 2, 1024, 128, "bf16", False),  # several 128-key blocks, no tail
    (3, 2, 129, 64, "bf16", False),    # one key past a block
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", PACKED)
def test_packed_mask_matches_oracle(fa, B, H, N, d, dtype, causal):
    q, k, v, mask = make_qkv(B, H, N, d, dtype, seed=29 * N + d + B, mask_frac=0.2, full_row_frac=0.02)
    scale = 1.0 / math.sqrt(d)
    out, lse = masked(fa, q, k, v, mask, scale, causal)
    ref_o, ref_l = oracle.attention(q, k, v, mask=mask, scale=scale, causal=causal)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("B,H,N,d,dtype,causal", PACKED)
def test_fp32_mask_kernel_matches_oracle(fa, B, H, N, d, dtype, causal):
    """The same masks through fa_fwd (no workspace): the fp32-mask kernel applies them as given."""
    q, k, v, mask = make_qkv(B, H, N, d, dtype, seed=29 * N + d + B, mask_frac=0.2, full_row_frac=0.02)
    scale = 1.0 / math.sqrt(d)
    out, lse = plain(fa, q, k, v, mask, scale, causal)
    ref_o, ref_l = oracle.attention(q, k, v, mask=mask, scale=scale, causal=causal)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("N,causal", [(300, False), (260, True), (517, False)])
def test_packed_mask_grouped_query(fa, N, causal):
    B, H, Hkv, d = 2, 6, 2, 128
    q, _, _, mask = make_qkv(B, H, N, d, "bf16", seed=N + 15, mask_frac=0.2, full_row_frac=0.02)
    _, k, v, _ = make_qkv(B, Hkv, N, d, "bf16", seed=N + 16)
    out, lse = masked(fa, q, k, v, mask, 1 / math.sqrt(d), causal)
    g = H // Hkv
    ref_o, ref_l = oracle.attention(q, k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1), mask=mask,
                                    scale=1 / math.sqrt(d), causal=causal)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("N,d,dtype,causal", [(300, 128, "bf16", False), (517, 64, "fp16", True)])
def test_other_mask_values_take_the_fp32_mask(fa, N, d, dtype, causal):
    """A mask with finite nonzero entries: the result is fa_fwd's with the same mask, bit for bit."""
    B, H = 2, 2
    q, k, v, mask = make_qkv(B, H, N, d, dtype, seed=N + 41, mask_frac=0.2, full_row_frac=0.02)
    g = torch.Generator().manual_seed(N)
    finite = torch.isfinite(mask)
    mask[finite] = torch.randint(-4, 3, (int(finite.sum()),), generator=g).float() * 0.375
    o1, l1 = masked(fa, q, k, v, mask, 1 / math.sqrt(d), causal)
    o2, l2 = plain(fa, q, k, v, mask, 1 / math.sqrt(d), causal)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_l = oracle.attention(q, k, v, mask=mask, scale=1 / math.sqrt(d), causal=causal)
    compare(out=o1, lse=l1, ref_o=ref_o, ref_l=ref_l)


def test_one_other_value_anywhere_switches_paths(fa):
    """A single 0.5 in the last row of the last batch index: the whole call takes the fp32 mask."""
    B, H, N, d = 2, 2, 400, 128
    q, k, v, mask = make_qkv(B, H, N, d, "bf16", seed=77, mask_frac=0.1)
    mask[B - 1, N - 1, N - 2] = 0.5
    o1, l1 = masked(fa, q, k, v, mask, 0.1, False)
    o2, l2 = plain(fa, q, k, v, mask, 0.1, False)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workspace_reuse_across_masks(fa):
    """One workspace for two calls whose masks differ: each call packs its own mask."""
    B, H, N, d = 1, 2, 640, 64
    q, k, v, m1 = make_qkv(B, H, N, d, "bf16", seed=91, mask_frac=0.3)
    m2 = torch.zeros_like(m1)
    m2[:, :, : N // 2] = float("-inf")
    m2[:, :5] = 0.0
    ws = torch.empty(fa.fa_fwd_masked_workspace_bytes(B, N), dtype=torch.uint8, device=DEV)
    outs = []
    for m in (m1, m2, m1):
        out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
        fa.fa_fwd_masked(q.to(DEV), k.to(DEV), v.to(DEV), m.to(DEV), out, lse, 0.125, False, ws)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[2][0]) and torch.equal(outs[0][1], outs[2][1])
    for (o, l), m in zip(outs[:2], (m1, m2)):
        ref_o, ref_l = oracle.attention(q, k, v, mask=m, scale=0.125)
        compare(o, l, ref_o, ref_l)


def test_attention_wrapper_uses_the_packed_path(fa):
    """``attention(mask=...)`` for bf16 goes through fa_fwd_masked: an all-zero mask gives the
    unmasked result bit for bit."""
    q, k, v, _ = make_qkv(1, 2, 700, 128, "bf16", seed=5)
    mask = torch.zeros((1, 700, 700), dtype=torch.float32)
    o1, l1 = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), mask=mask.to(DEV), scale=0.1, causal=True)
    o2, l2 = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), scale=0.1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(ValueError):
        fa.fa_fwd_masked(q.to(DEV), k.to(DEV), v.to(DEV), None, o1, l1, 0.1, False,
                         torch.empty(16, dtype=torch.uint8, device=DEV))
    with pytest.raises(fa.FAError):
        fa.fa_fwd_masked(q.to(DEV), k.to(DEV), v.to(DEV), mask.to(DEV), o1, l1, 0.1, False,
                         torch.empty(16, dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("d,dtype,causal", [(64, "fp16", True), (128, "bf16", False)])
def test_masked_writes_stay_inside_their_buffers(fa, d, dtype, causal):
    """Guard bands around O, lse and the workspace stay untouched: N = 333 is ragged against the
    128-key blocks and N % 4 != 0 takes the packing pass's scalar loads."""
    B, H, N = 2, 3, 333
    q, k, v, mask = make_qkv(B, H, N, d, dtype, seed=N + d, mask_frac=0.2, full_row_frac=0.02)
    pad = 4096
    t = q.dtype
    obuf = torch.full((B * H * N * d + 2 * pad,), 7.0, dtype=t, device=DEV)
    lbuf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    nws = fa.fa_fwd_masked_workspace_bytes(B, N)
    wbuf = torch.full((nws + 2 * pad,), 0x5A, dtype=torch.uint8, device=DEV)
    out = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    ws = wbuf[pad:pad + nws]
    fn = fa.fa_fwd_masked if q.dtype == torch.bfloat16 else fa.fa_fwd_masked_fp16
    fn(q.to(DEV), k.to(DEV), v.to(DEV), mask.to(DEV), out, lse, 1 / math.sqrt(d), causal, ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert bool((obuf[:pad] == 7.0).all()) and bool((obuf[-pad:] == 7.0).all())
    assert bool((lbuf[:pad] == 7.0).all()) and bool((lbuf[-pad:] == 7.0).all())
    assert bool((wbuf[:pad] == 0x5A).all()) and bool((wbuf[-pad:] == 0x5A).all())
    ref_o, ref_l = oracle.attention(q, k, v, mask=mask, scale=1 / math.sqrt(d), causal=causal)
    compare(out, lse, ref_o, ref_l)
