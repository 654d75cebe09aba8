"""GPU parity of the packed variable-length forward: every sequence of the
batch against the oracle run on that sequence alone (attention never crosses
a sequence boundary)."""
import math

import pytest
import torch

import oracle
from io_aware_exact_13_gb300.inputs import VARLEN_WORKLOADS, make_varlen
from parity_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def _check_sequences(q, k, v, cu, out, lse, scale, causal, seqs=None):
    H, Hkv = q.shape[1], k.shape[1]
    g = H // Hkv
    cu = cu.tolist()
    seqs = range(len(cu) - 1) if seqs is None else seqs
    for s in seqs:
        a, b = cu[s], cu[s + 1]
        if b == a:
            continue
        qs = q[a:b].permute(1, 0, 2).unsqueeze(0)
        ks = k[a:b].permute(1, 0, 2).unsqueeze(0).repeat_interleave(g, dim=1)
        vs = v[a:b].permute(1, 0, 2).unsqueeze(0).repeat_interleave(g, dim=1)
        ro, rl = oracle.attention(qs, ks, vs, scale=scale, causal=causal)
        compare(out[a:b].permute(1, 0, 2).unsqueeze(0), lse[:, a:b].unsqueeze(0), ro, rl)


EDGE = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 0, 300]


@pytest.mark.parametrize("d,dtype,causal,H,Hkv", [(128, "bf16", True, 4, 4), (128, "bf16", False, 4, 2),
                                                  (64, "fp16", True, 3, 1), (64, "bf16", False, 2, 2)])
def test_varlen_edge_lengths(fa, d, dtype, causal, H, Hkv):
    q, k, v, cu = make_varlen(EDGE, H, Hkv, d, dtype, seed=d + H + int(causal))
    dev = torch.device("cuda")
    out, lse = fa.attention_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev), max(EDGE), causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    _check_sequences(q, k, v, cu, out.cpu(), lse.cpu(), 1 / math.sqrt(d), causal)


def test_varlen_single_sequence_equals_dense(fa):
    """One sequence of length N packed is the [1, H, N, d] forward, bit for bit: both
    run the same kernel, and every query row visits the same key blocks in the same
    order with the same arithmetic (only the work items' order and the tensor maps'
    coordinates differ)."""
    N, H, d = 1000, 4, 128
    q, k, v, cu = make_varlen([N], H, H, d, "bf16", seed=9)
    dev = torch.device("cuda")
    out, lse = fa.attention_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev), N, causal=True)
    o2, l2 = fa.attention(q.permute(1, 0, 2).unsqueeze(0).contiguous().to(dev),
                          k.permute(1, 0, 2).unsqueeze(0).contiguous().to(dev),
                          v.permute(1, 0, 2).unsqueeze(0).contiguous().to(dev), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out.permute(1, 0, 2), o2[0])
    assert torch.equal(lse, l2[0])
    _check_sequences(q, k, v, cu, out.cpu(), lse.cpu(), 1 / math.sqrt(d), True)


def test_varlen_larger_max_seqlen_and_tail_tokens_untouched(fa):
    """max_seqlen above every length is fine; tokens past cu_seqlens[nseq] are not written."""
    lengths = [200, 513, 77]
    q, k, v, cu = make_varlen(lengths + [50], 2, 2, 64, "bf16", seed=4)
    cu = cu[:-1].contiguous()  # the last 50 tokens belong to no sequence
    dev = torch.device("cuda")
    out = torch.full(q.shape, 7.0, dtype=q.dtype, device=dev)
    lse = torch.full((2, q.shape[0]), 7.0, dtype=torch.float32, device=dev)
    fa.fa_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), out, lse, cu.to(dev), 4096, 0.125, False)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.all(out[sum(lengths):] == 7.0) and torch.all(lse[:, sum(lengths):] == 7.0)
    _check_sequences(q, k, v, cu, out.cpu(), lse.cpu(), 0.125, False)


def test_varlen_bad_bounds_are_skipped_and_reported(fa):
    """A sequence longer than max_seqlen is skipped (rows untouched) and flagged;
    the other sequences are still computed."""
    lengths = [100, 600, 150]
    q, k, v, cu = make_varlen(lengths, 2, 2, 128, "bf16", seed=5)
    dev = torch.device("cuda")
    out = torch.full(q.shape, 3.0, dtype=q.dtype, device=dev)
    lse = torch.full((2, q.shape[0]), 3.0, dtype=torch.float32, device=dev)
    fa.fa_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), out, lse, cu.to(dev), 512, 1 / math.sqrt(128), True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_ERR_SEQLENS
    assert fa.fa_get_device_status() == fa.FA_OK  # reading clears it
    assert torch.all(out[100:700] == 3.0) and torch.all(lse[:, 100:700] == 3.0)
    _check_sequences(q, k, v, cu, out.cpu(), lse.cpu(), 1 / math.sqrt(128), True, seqs=[0, 2])


def test_varlen_workload_every_sequence(fa):
    """The benchmark's packed batch in the benchmark's launch; every sequence is
    checked against the oracle run on that sequence alone."""
    w = VARLEN_WORKLOADS["varlen_t65536_h32_d128_bf16_causal"]
    L = w.lengths()
    q, k, v, cu = make_varlen(L, w.H, w.H, w.d, w.dtype, seed=w.seed)
    dev = torch.device("cuda")
    out, lse = fa.attention_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev), max(L), scale=w.scale,
                                   causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    _check_sequences(q, k, v, cu, out.cpu(), lse.cpu(), w.scale, w.causal)


def test_varlen_many_sequences_and_levels(fa):
    """More sequences than a warp ballot covers (the item list scans them 32 at a
    time), zero lengths among them, lengths over several 256-row levels, and
    grouped K/V heads: every sequence against the oracle."""
    g = torch.Generator().manual_seed(21)
    lengths = [int(x) for x in torch.randint(0, 1500, (100,), generator=g)]
    lengths[5] = lengths[40] = lengths[99] = 0
    lengths[63] = 1500
    q, k, v, cu = make_varlen(lengths, 3, 1, 64, "bf16", seed=22)
    dev = torch.device("cuda")
    out, lse = fa.attention_varlen(q.to(dev), k.to(dev), v.to(dev), cu.to(dev), max(lengths), causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    _check_sequences(q, k, v, cu, out.cpu(), lse.cpu(), 1 / math.sqrt(64), True)


def test_varlen_all_sequences_empty(fa):
    """Every sequence has length 0: no work item, nothing written, no error."""
    q, k, v, _ = make_varlen([16], 2, 2, 128, "bf16", seed=23)
    cu = torch.zeros(5, dtype=torch.int32)
    dev = torch.device("cuda")
    out = torch.full(q.shape, 5.0, dtype=q.dtype, device=dev)
    lse = torch.full((2, q.shape[0]), 5.0, dtype=torch.float32, device=dev)
    fa.fa_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), out, lse, cu.to(dev), 16, 0.1, True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.all(out == 5.0) and torch.all(lse == 5.0)
