"""The C-ABI library: it loads, exports every symbol include/fa.h declares, and
rejects bad arguments on the host before touching the GPU. CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    from io_aware_exact_13_gb300 import build

    build.build()
    from io_aware_exact_13_gb300 import fa as mod

    return mod


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_forward_family():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_fp16", "fa_fwd_fp32", "fa_status_string", "fa_get_device_status", "fa_num_sms",
              "fa_fwd_splitkv", "fa_fwd_splitkv_fp16", "fa_splitkv_workspace_bytes", "fa_splitkv_num_splits"):
        assert n in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa._LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"libfa.so does not export {name}"
        assert name in fa.SIGNATURES, f"binding has no signature for {name}"


def test_status_strings(fa):
    for code in range(0, -10, -1):
        s = fa.fa_status_string(code)
        assert s and s != "unknown status"
    assert fa.fa_status_string(12345) == "unknown status"


def _call(fa, name, q=0x10000, k=0x20000, v=0x30000, mask=None, out=0x40000, lse=0x50000, B=1, H=1, N=16, d=128,
          scale=0.1, causal=0):
    f = getattr(fa.lib, name)
    return f(ctypes.c_void_p(q) if q else None, ctypes.c_void_p(k) if k else None,
             ctypes.c_void_p(v) if v else None, ctypes.c_void_p(mask) if mask else None,
             ctypes.c_void_p(out) if out else None, ctypes.c_void_p(lse) if lse else None,
             B, H, N, d, ctypes.c_float(scale), causal, None)


@pytest.mark.parametrize("name", ["fa_fwd", "fa_fwd_fp16", "fa_fwd_fp32"])
def test_host_validation_rejects_before_launch(fa, name):
    assert _call(fa, name, q=0) == fa.FA_ERR_NULL
    assert _call(fa, name, lse=0) == fa.FA_ERR_NULL
    assert _call(fa, name, out=0) == fa.FA_ERR_NULL
    assert _call(fa, name, k=0x20008) == fa.FA_ERR_ALIGN
    assert _call(fa, name, mask=0x60004) == fa.FA_ERR_ALIGN
    assert _call(fa, name, lse=0x50002) == fa.FA_ERR_ALIGN
    assert _call(fa, name, N=0) == fa.FA_ERR_SHAPE
    assert _call(fa, name, B=-1) == fa.FA_ERR_SHAPE
    assert _call(fa, name, H=0) == fa.FA_ERR_SHAPE
    assert _call(fa, name, B=1 << 16, H=1 << 16) == fa.FA_ERR_SHAPE
    assert _call(fa, name, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _call(fa, name, d=256) == fa.FA_ERR_UNSUPPORTED


def test_fp32_grid_limit(fa):
    assert _call(fa, "fa_fwd_fp32", B=256, H=257) == fa.FA_ERR_SHAPE


def test_gqa_host_checks(fa):
    f = fa.lib.fa_fwd_gqa
    args = lambda H, Hkv: (ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000), None,
                           ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000), 1, H, Hkv, 64, 128,
                           ctypes.c_float(0.1), 0, None)
    assert f(*args(8, 3)) == fa.FA_ERR_SHAPE   # Hkv must divide H
    assert f(*args(8, 0)) == fa.FA_ERR_SHAPE
    assert fa.lib.fa_fwd_gqa_fp16(*args(4, 8)) == fa.FA_ERR_SHAPE


def test_splitkv_host_checks(fa):
    lib = fa.lib
    assert lib.fa_splitkv_workspace_bytes(1, 1, 1, 96, 4) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_splitkv_workspace_bytes(0, 1, 1, 64, 4) == fa.FA_ERR_SHAPE
    rows, d, n = 2 * 3 * 5, 128, 7
    expect = ((n * rows * d * 4 + 255) // 256) * 256 + ((n * rows * 4 + 255) // 256) * 256
    assert lib.fa_splitkv_workspace_bytes(2, 3, 5, d, n) == expect

    def call(name="fa_fwd_splitkv", q=0x10000, Nq=1, Nk=64, d=128, n_splits=2, ws=0x100000, ws_bytes=1 << 20):
        f = getattr(lib, name)
        return f(ctypes.c_void_p(q) if q else None, ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000),
                 ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000), 1, 2, Nq, Nk, d, ctypes.c_float(0.1), 0,
                 n_splits, ctypes.c_void_p(ws) if ws else None, ws_bytes, None)

    for name in ("fa_fwd_splitkv", "fa_fwd_splitkv_fp16"):
        assert call(name, q=0) == fa.FA_ERR_NULL
        assert call(name, q=0x10008) == fa.FA_ERR_ALIGN
        assert call(name, Nq=17) == fa.FA_ERR_SHAPE
        assert call(name, Nq=0) == fa.FA_ERR_SHAPE
        assert call(name, n_splits=0) == fa.FA_ERR_SHAPE
        assert call(name, n_splits=65) == fa.FA_ERR_SHAPE  # more splits than keys
        assert call(name, d=80) == fa.FA_ERR_UNSUPPORTED
        assert call(name, ws=0) == fa.FA_ERR_WORKSPACE
        assert call(name, ws=0x100010) == fa.FA_ERR_WORKSPACE  # not 256-byte aligned
        assert call(name, ws_bytes=16) == fa.FA_ERR_WORKSPACE


def test_binding_checks_shapes_without_a_gpu(fa):
    import torch

    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.attention(q, q, q)  # CPU tensors are refused by the binding


def test_product_path_does_not_import_the_oracle():
    """Nothing under the package or bench's GPU path may import oracle/."""
    pkg = os.path.join(ROOT, "io_aware_exact_13_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, re.M), f
                assert "attn_oracle" not in txt and "liboracle" not in txt, f


def _bwd(fa, name="fa_bwd", ptrs=None, B=1, H=1, N=16, d=64, ws=0x90000, ws_bytes=1 << 30):
    p = [0x10000 * (i + 1) for i in range(9)] if ptrs is None else ptrs
    f = getattr(fa.lib, name)
    return f(*[ctypes.c_void_p(x) if x else None for x in p], B, H, N, d, ctypes.c_float(0.125), 0,
             ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("name", ["fa_bwd", "fa_bwd_fp16"])
def test_bwd_host_validation_rejects_before_launch(fa, name):
    base = [0x10000 * (i + 1) for i in range(9)]
    for i in range(9):
        p = list(base)
        p[i] = 0
        assert _bwd(fa, name, p) == fa.FA_ERR_NULL
    p = list(base)
    p[1] += 8
    assert _bwd(fa, name, p) == fa.FA_ERR_ALIGN
    p = list(base)
    p[5] += 2  # lse needs 4 bytes
    assert _bwd(fa, name, p) == fa.FA_ERR_ALIGN
    assert _bwd(fa, name, N=0) == fa.FA_ERR_SHAPE
    assert _bwd(fa, name, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _bwd(fa, name, ws=0) == fa.FA_ERR_WORKSPACE
    assert _bwd(fa, name, ws=0x90010) == fa.FA_ERR_WORKSPACE  # not 256-byte aligned
    need = fa.fa_bwd_workspace_bytes(1, 1, 16, 64)
    assert _bwd(fa, name, ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE


def test_bwd_workspace_size(fa):
    # fp32 dQ accumulator (B*H*N*d) + two fp32 row arrays padded to 128 rows, each part 256-byte aligned
    assert fa.fa_bwd_workspace_bytes(2, 16, 4096, 64) == 2 * 16 * 4096 * 64 * 4 + 2 * (2 * 16 * 4096 * 4)
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 64) == 256 + 2 * 512
    with pytest.raises(fa.FAError):
        fa.fa_bwd_workspace_bytes(1, 1, 16, 80)


@pytest.mark.parametrize("name", ["fa_fwd_varlen", "fa_fwd_varlen_fp16"])
def test_varlen_host_validation(fa, name):
    f = getattr(fa.lib, name)

    def call(ptrs=(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000), nseq=2, total=100, maxlen=64, H=2, Hkv=2,
             d=64):
        return f(*[ctypes.c_void_p(x) if x else None for x in ptrs], nseq, total, maxlen, H, Hkv, d,
                 ctypes.c_float(0.125), 1, None)

    assert call(ptrs=(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0)) == fa.FA_ERR_NULL
    assert call(ptrs=(0x10008, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000)) == fa.FA_ERR_ALIGN
    assert call(ptrs=(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60002)) == fa.FA_ERR_ALIGN
    assert call(nseq=0) == fa.FA_ERR_SHAPE
    assert call(total=0) == fa.FA_ERR_SHAPE
    assert call(maxlen=0) == fa.FA_ERR_SHAPE
    assert call(H=3, Hkv=2) == fa.FA_ERR_SHAPE
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_status_string(fa.FA_ERR_SEQLENS) != "unknown status"


def test_fa_log_prints_the_dispatch_on_the_host(tmp_path):
    """FA_LOG=1 logs the kernel variant of each call that passes its argument
    checks (to stderr, before the device is touched: here, without a GPU, the
    call then fails with FA_ERR_LAUNCH); a call rejected by the checks logs nothing."""
    import subprocess
    import sys

    call = ("fa.lib.fa_fwd(ctypes.c_void_p(16), ctypes.c_void_p(32), ctypes.c_void_p(48), None, "
            "ctypes.c_void_p(64), ctypes.c_void_p(80), 2, 4, 300, {d}, ctypes.c_float(0.1), 1, None)")
    code = "import ctypes, io_aware_exact_13_gb300.fa as fa; print({a}); print({b})".format(
        a=call.format(d=96), b=call.format(d=128))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=dict(os.environ, FA_LOG="1"), capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == [str(-4), str(-5)]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[fa]")]
    assert len(lines) == 1 and "forward bf16 tcgen05 d=128 causal=1" in lines[0] and "N=300" in lines[0], r.stderr


@pytest.mark.parametrize("name", ["fa_fwd_host", "fa_fwd_host_fp16"])
def test_host_forward_validation(fa, name):
    f = getattr(fa.lib, name)

    def call(ptrs=None, B=1, H=2, N=16, d=64, chunks=2):
        p = [0x10000 * (i + 1) for i in range(10)] if ptrs is None else ptrs
        return f(*[ctypes.c_void_p(x) if x else None for x in p], B, H, N, d, ctypes.c_float(0.125), 0, chunks, None)

    base = [0x10000 * (i + 1) for i in range(10)]
    for i in range(10):
        p = list(base)
        p[i] = 0
        assert call(p) == fa.FA_ERR_NULL
    p = list(base)
    p[6] += 8  # k_dev misaligned
    assert call(p) == fa.FA_ERR_ALIGN
    assert call(chunks=0) == fa.FA_ERR_SHAPE
    assert call(chunks=3) == fa.FA_ERR_SHAPE  # more chunks than B*H = 2
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["fa_fwd_masked", "fa_fwd_masked_fp16"])
def test_masked_host_validation(fa, name):
    f = getattr(fa.lib, name)
    need = fa.fa_fwd_masked_workspace_bytes(2, 300)

    def call(mask=0x60000, H=4, Hkv=2, N=300, d=128, ws=0x100000, ws_bytes=None):
        return f(ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000),
                 ctypes.c_void_p(mask) if mask else None, ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000),
                 2, H, Hkv, N, d, ctypes.c_float(0.1), 0, ctypes.c_void_p(ws) if ws else None,
                 need if ws_bytes is None else ws_bytes, None)

    assert call(mask=0) == fa.FA_ERR_NULL       # the mask is required
    assert call(mask=0x60004) == fa.FA_ERR_ALIGN
    assert call(N=0) == fa.FA_ERR_SHAPE
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(ws=0) == fa.FA_ERR_WORKSPACE
    assert call(ws=0x100010) == fa.FA_ERR_WORKSPACE  # not 256-byte aligned
    assert call(ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    assert call(Hkv=3) == fa.FA_ERR_SHAPE            # Hkv must divide H


def test_masked_workspace_size(fa):
    # one bit per (row, key) in 16-byte units of 128 keys, then 256 bytes for the verdict word
    assert fa.fa_fwd_masked_workspace_bytes(2, 4096) == 2 * 4096 * 32 * 16 + 256
    assert fa.fa_fwd_masked_workspace_bytes(1, 1) == 16 + 256
    assert fa.fa_fwd_masked_workspace_bytes(3, 129) == 3 * 129 * 2 * 16 + 256
    with pytest.raises(fa.FAError):
        fa.fa_fwd_masked_workspace_bytes(0, 16)


@pytest.mark.parametrize("name", ["fa_fwd_dropout", "fa_fwd_dropout_fp16"])
def test_dropout_host_validation(fa, name):
    f = getattr(fa.lib, name)

    def call(q=0x10000, H=4, Hkv=2, N=300, d=128, p_drop=0.1):
        return f(ctypes.c_void_p(q) if q else None, ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000),
                 ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000), 2, H, Hkv, N, d, ctypes.c_float(0.1), 0,
                 ctypes.c_float(p_drop), 7, 0, None)

    assert call(q=0) == fa.FA_ERR_NULL
    assert call(q=0x10008) == fa.FA_ERR_ALIGN
    assert call(N=0) == fa.FA_ERR_SHAPE
    assert call(Hkv=3) == fa.FA_ERR_SHAPE
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(p_drop=0.999) == fa.FA_ERR_ARG       # keeps nothing
    assert call(p_drop=-0.001) == fa.FA_ERR_ARG
    assert call(p_drop=float("nan")) == fa.FA_ERR_ARG
