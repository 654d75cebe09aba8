"""Build ``libfa.so`` (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

A few translation units per element type plus the C ABI, compiled in parallel,
then linked as a shared library next to this file. Only the CUDA runtime and
the C++ standard library are linked; the driver entry point for tensor-map
encoding is looked up at run time.
"""
from __future__ import annotations

import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libfa.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["fa_api.cu", "fa_fwd_bf16.cu", "fa_fwd_fp16.cu", "fa_fwd_mask_bf16.cu", "fa_fwd_mask_fp16.cu",
           "fa_mask_pack.cu", "fa_fwd_drop_bf16.cu", "fa_fwd_drop_fp16.cu", "fa_fwd_fp32.cu", "fa_splitkv.cu", "fa_splitkv_noalloc.cu", "fa_bwd.cu",
           "fa_fwd_varlen_bf16.cu", "fa_fwd_varlen_fp16.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-Wno-deprecated-gpu-targets"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    inc = os.path.join(os.path.dirname(HERE), "include", "fa.h")
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [inc]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def check_ptxas_log(log: str) -> tuple[list[str], list[str]]:
    """(errors, warnings) from ptxas -v output. Error: a forward kernel that does
    not launch with 128 registers per thread (the warpgroup register split is
    sized for exactly that). Warning: register spills."""
    problems, warnings = [], []
    kernel = None
    for line in log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            kernel = m.group(1)
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and kernel and (int(m.group(1)) or int(m.group(2))):
            warnings.append(f"{kernel}: spills ({m.group(0)})")
        m = re.search(r"Used (\d+) registers", line)
        if m and kernel and re.search(r"fa_fwd_(bk128_)?kernel", kernel) and int(m.group(1)) != 128:
            problems.append(f"{kernel}: uses {m.group(1)} registers, expected 128")
    return problems, warnings


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link ``libfa.so``; returns its path."""
    deps = _deps()
    if not force and not _stale(LIB, deps):
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    log = "\n".join(r[1] for r in results)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write(log)
    problems, warnings = check_ptxas_log(log)
    with open(os.path.join(BUILD_DIR, "ptxas_warnings.txt"), "w") as f:
        f.write("\n".join(warnings) + "\n")
    if problems:
        raise RuntimeError("ptxas check failed:\n" + "\n".join(problems))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[r[0] for r in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(log, file=sys.stderr)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
