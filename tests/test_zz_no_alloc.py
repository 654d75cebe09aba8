"""The split-KV entry point that allocates nothing (fa_fwd_splitkv_noalloc).

It serves callers that cannot allocate device memory where they call
attention (a framework that owns all device memory, a serving loop that must
not pay cudaMalloc's device-wide synchronisation, a fixed-budget embedded
host): its scratch is a fixed array inside the library. Here it must give the
same bits as fa_fwd_splitkv with a caller-provided workspace (both run the
same two kernels on the same inputs), on two calls in a row (the second call
finds the first call's leftovers in the shared array), leave the device's free
memory unchanged across a call, and reject a problem whose scratch would not
fit. One case also goes through the Python wrapper, whose argument checks
must refuse a wrong element type.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes when run alone.
"""
import ctypes
import math

import pytest
import torch

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


def _reference(fa, qd, kd, vd, scale, causal, n_splits):
    B, H, Nq, d = qd.shape
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits), dtype=torch.uint8, device=qd.device)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=qd.device)
    fa.fa_fwd_splitkv(qd, kd, vd, out, lse, scale, causal, n_splits, ws)
    return out, lse


def _noalloc_via_c_abi(fa, qd, kd, vd, out, lse, scale, causal, n_splits):
    B, H, Nq, d = qd.shape
    Nk = kd.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fa.lib.fa_fwd_splitkv_noalloc(p(qd), p(kd), p(vd), p(out), p(lse), B, H, Nq, Nk, d, ctypes.c_float(scale),
                                         int(causal), n_splits, stream)


@pytest.mark.parametrize("shape", [(2, 4, 3, 5000, 128, True, 9), (1, 8, 1, 777, 64, False, 5)])
def test_noalloc_matches_workspace_entry_point_twice(fa, shape):
    B, H, Nq, Nk, d, causal, n_splits = shape
    dev = torch.device("cuda")
    scale = 1 / math.sqrt(d)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        q, k, v, _ = make_qkv(B, H, Nq, d, "bf16", seed=seed + Nk, Nk=Nk)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        ref_o, ref_l = _reference(fa, qd, kd, vd, scale, causal, n_splits)
        out = torch.full_like(qd, float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = _noalloc_via_c_abi(fa, qd, kd, vd, out, lse, scale, causal, n_splits)
        assert rc == fa.FA_OK, fa.fa_status_string(rc)
        torch.cuda.synchronize()
        if call == 1:  # the first call on a device may load the module; later calls allocate nothing
            assert torch.cuda.mem_get_info()[0] == free0, "a call changed the device's free memory"
        # the same kernels on the same inputs: the same bits
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
        compare(out, lse, ref_o.float().cpu().double().numpy(), ref_l.cpu().double().numpy())


def test_noalloc_python_wrapper(fa):
    """The binding's wrapper marshals the same call and checks its arguments."""
    dev = torch.device("cuda")
    B, H, Nq, Nk, d, n_splits = 1, 4, 2, 3000, 128, 7
    q, k, v, _ = make_qkv(B, H, Nq, d, "bf16", seed=21, Nk=Nk)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ref_o, ref_l = _reference(fa, qd, kd, vd, 0.1, True, n_splits)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    fa.fa_fwd_splitkv_noalloc(qd, kd, vd, out, lse, 0.1, True, n_splits)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    with pytest.raises(ValueError):
        fa.fa_fwd_splitkv_noalloc(qd.half(), kd.half(), vd.half(), out.half(), lse, 0.1, True, n_splits)


def test_noalloc_rejects_problems_beyond_its_scratch(fa):
    dev = torch.device("cuda")
    B, H, Nq, Nk, d, n_splits = 8, 64, 16, 1024, 128, 64  # needs ~134 MB of scratch
    assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits) > 16 << 20
    q = torch.zeros((B, H, Nq, d), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    rc = _noalloc_via_c_abi(fa, q, kv, kv, out, lse, 0.1, False, n_splits)
    assert rc == fa.FA_ERR_WORKSPACE
