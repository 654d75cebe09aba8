"""The host-memory forward (fa_fwd_host): copies and compute pipelined over head
chunks must give fa_fwd's results bit for bit, for any chunk count."""
import math

import pytest
import torch

from io_aware_exact_13_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


@pytest.mark.parametrize("B,H,N,d,dtype,causal,chunks", [
    (1, 8, 2048, 128, "bf16", True, 1),
    (1, 8, 2048, 128, "bf16", True, 3),
    (2, 4, 1000, 128, "bf16", False, 8),
    (2, 3, 517, 64, "fp16", True, 5),
    (1, 1, 1, 64, "bf16", False, 1),
])
def test_host_forward_equals_device_forward(fa, B, H, N, d, dtype, causal, chunks):
    q, k, v, _ = make_qkv(B, H, N, d, dtype, seed=N + chunks)
    dev = torch.device("cuda")
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    qd, kd, vd = torch.empty_like(q, device=dev), torch.empty_like(k, device=dev), torch.empty_like(v, device=dev)
    od = torch.empty_like(qd)
    ld = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    scale = 1 / math.sqrt(d)
    fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, scale, causal, chunks)
    torch.cuda.current_stream().synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = fa.attention(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref_o.cpu())
    assert torch.equal(lh, ref_l.cpu())
