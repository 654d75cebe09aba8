"""The pins have teeth: each test here plants one plausible mistake in a copy of
the oracle's C source, builds it, and runs the pin suite (tests/test_oracle_pins.py)
against that copy in a subprocess. Every mutant must make at least one pin fail.
The real oracle is never modified; the copies live in a temporary directory."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

# (name, original text, mutated text): one mistake each, in every part of the oracle
MUTANTS = [
    ("causal_off_by_one", "return j <= i + (Nk - Nq);", "return j < i + (Nk - Nq);"),
    ("causal_alignment_top_left", "return j <= i + (Nk - Nq);", "return j <= i;"),
    ("scale_dropped", "double sij = scale * dot;", "double sij = dot;"),
    ("mask_sign", "if (mask) sij += mask[(b * Nq + i) * Nk + j];", "if (mask) sij -= mask[(b * Nq + i) * Nk + j];"),
    ("key_index_transposed", "for (int64_t t = 0; t < d; ++t) dot += qi[t] * kb[j * d + t];",
     "for (int64_t t = 0; t < d; ++t) dot += qi[t] * kb[t * Nk + j];"),
    ("head_index_swapped", "const double *kb = k + (b * H + h) * Nk * d;", "const double *kb = k + (h * H + b) * Nk * d;"),
    ("lse_without_log", "o[t] /= l;\n    *lse = m + log(l);", "o[t] /= l;\n    *lse = m + l;"),
    ("no_normalisation", "for (int64_t t = 0; t < d; ++t) o[t] /= l;", ";"),
    ("merge_without_rescale", "double fa = (mA == -INFINITY) ? 0.0 : exp(mA - mx);",
     "double fa = (mA == -INFINITY) ? 0.0 : 1.0;"),
    ("summary_wrong_max", "    *m = mx;\n    *l = 0.0;", "    *m = 0.0;\n    *l = 0.0;"),
    ("bwd_drops_D", "double dsij = pij * (dp[j] - rowdot);", "double dsij = pij * dp[j];"),
    ("bwd_dk_unscaled", "dkb[j * d + t] += scale * dsij * qi[t];", "dkb[j * d + t] += dsij * qi[t];"),
    ("bwd_dv_uses_dp", "dvb[j * d + t] += pij * doi[t];", "dvb[j * d + t] += dp[j] * doi[t];"),
    ("philox_nine_rounds", "for (int round = 0; round < 10; ++round) {", "for (int round = 0; round < 9; ++round) {"),
    ("philox_words_swapped", "        x0 = hi1 ^ x1 ^ k0;\n", "        x0 = hi0 ^ x1 ^ k0;\n"),
    ("dropout_counter_order", "const uint64_t ctr[4] = {(uint64_t)i, (uint64_t)g, (uint64_t)(b * H + h), offset};",
     "const uint64_t ctr[4] = {(uint64_t)g, (uint64_t)i, (uint64_t)(b * H + h), offset};"),
    ("dropout_byte_order", "const unsigned byte = (unsigned)((w[t / 8] >> (8 * (t % 8))) & 0xFFu);",
     "const unsigned byte = (unsigned)((w[t % 4] >> (8 * (t / 4))) & 0xFFu);"),
    ("dropout_renormalised", "        l += p;\n        if (keep[j])", "        if (keep[j]) l += p;\n        if (keep[j])"),
    ("dropout_unscaled", "o[t] = (o[t] / l) * inv_q;", "o[t] = o[t] / l;"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(source, tmp_path, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-I", os.path.join(ROOT, "oracle"),
                    "-o", str(lib), str(src), "-lm"], check=True)
    env = dict(os.environ, ORACLE_MUTANT_LIB=str(lib), OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"no pin caught mutant {name} (exit {r.returncode}):\n{r.stdout[-2000:]}"
    assert " failed" in r.stdout and " error" not in r.stdout, r.stdout[-2000:]


def test_unmutated_copy_passes(source, tmp_path):
    """Control: the same build and run with the source unchanged passes every pin,
    so the failures above come from the planted mistakes."""
    src = tmp_path / "copy.c"
    src.write_text(source)
    lib = tmp_path / "libcopy.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-I", os.path.join(ROOT, "oracle"),
                    "-o", str(lib), str(src), "-lm"], check=True)
    env = dict(os.environ, ORACLE_MUTANT_LIB=str(lib), OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
