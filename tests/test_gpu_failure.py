"""Failure detection on the GPU without a fault: a wait that nothing completes
must give up after its limit, report FA_ERR_TIMEOUT through the device status
word, and leave the context usable (a normal forward afterwards is correct)."""
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


def test_bounded_wait_reports_timeout_and_context_survives(fa):
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_selftest_wait_timeout(2_000_000)  # 2 ms
    assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_device_status() == fa.FA_OK  # reading clears the word
    q, k, v, _ = make_qkv(1, 2, 300, 128, "bf16", seed=77)
    dev = torch.device("cuda")
    out, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention(q, k, v, scale=1 / math.sqrt(128), causal=True)
    compare(out, lse, ref_o, ref_l)


def test_selftest_rejects_unbounded_limits(fa):
    with pytest.raises(fa.FAError):
        fa.fa_selftest_wait_timeout(0)
    with pytest.raises(fa.FAError):
        fa.fa_selftest_wait_timeout(5_000_000_000)
