"""Pins for the fp64 oracle: each test ties it to something other than itself.

* the pages' two worked examples (tests/golden/worked_examples.json, cited there);
* closed forms built so that every score is ln of a chosen integer, which makes the
  exact answer a ratio of integers evaluated here with ``fractions.Fraction``;
* special cases with textbook answers (scale 0 gives plain / prefix means, N = 1,
  constant values, the fully masked row convention);
* invariants (mask row shifts, joint key/value permutation, huge score offsets);
* the blockwise summary-and-merge routine against the materialised one;
* the backward routine against central differences of the forward routine.

Run on the CPU only (no GPU marker).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _fr(pair):
    return Fraction(pair[0], pair[1])


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return {e["name"]: e for e in json.load(f)["examples"]}


def _one_row(scores, values):
    """Put scores straight into a d = 1 problem: q = 1, k_j = s_j, scale = 1."""
    n = len(scores)
    q = np.ones((1, 1, 1, 1))
    k = np.asarray(scores, dtype=np.float64).reshape(1, 1, n, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, 1, n, 1)
    return q, k, v


# ---------------------------------------------------------------- worked examples

def test_worked_example_one_row_two_ways(oracle_lib, golden):
    ex = golden["one_row_checked_two_ways"]
    scores = [math.log(x) for x in ex["scores_ln"]]
    q, k, v = _one_row(scores, ex["values"])
    out, lse = oracle_lib.attention(q, k, v, scale=1.0)
    assert out[0, 0, 0, 0] == pytest.approx(float(_fr(ex["output"])), rel=1e-14)
    # weights (1, 2, 3)/6: the normaliser is 6, so lse = ln 6
    assert lse[0, 0, 0] == pytest.approx(math.log(6.0), rel=1e-14)

    s = ex["split_after"]
    A = oracle_lib.block_summary(scores[:s], ex["values"][:s])
    B = oracle_lib.block_summary(scores[s:], ex["values"][s:])
    assert A[0] == pytest.approx(math.log(ex["block_A"]["m_ln"]), rel=1e-15)
    assert A[1] == pytest.approx(float(_fr(ex["block_A"]["l"])), rel=1e-15)
    assert A[2] == pytest.approx(float(_fr(ex["block_A"]["u"])), rel=1e-15)
    assert B[0] == pytest.approx(math.log(ex["block_B"]["m_ln"]), rel=1e-15)
    assert B[1] == pytest.approx(float(_fr(ex["block_B"]["l"])), rel=1e-15)
    assert B[2] == pytest.approx(float(_fr(ex["block_B"]["u"])), rel=1e-15)
    # raising A's reference maximum to ln 3 multiplies its sums by 2/3
    assert math.exp(A[0] - B[0]) == pytest.approx(float(_fr(ex["rescale_A"])), rel=1e-14)
    m, l, u = oracle_lib.merge(A, B)
    assert m == pytest.approx(math.log(ex["merged"]["m_ln"]), rel=1e-15)
    assert l == pytest.approx(float(_fr(ex["merged"]["l"])), rel=1e-14)
    assert u == pytest.approx(float(_fr(ex["merged"]["u"])), rel=1e-14)
    assert u / l == pytest.approx(float(_fr(ex["output"])), rel=1e-14)
    # the unrescaled sums give the page's wrong answer, which the merge must not produce
    wrong = (A[2] + B[2]) / (A[1] + B[1])
    assert wrong == pytest.approx(float(_fr(ex["wrong_unrescaled_merge"])), rel=1e-14)
    assert abs(u / l - wrong) > 0.2


def test_worked_example_practice(oracle_lib, golden):
    ex = golden["practice_average_block_outputs"]
    scores = [math.log(x) for x in ex["scores_ln"]]
    q, k, v = _one_row(scores, ex["values"])
    out, lse = oracle_lib.attention(q, k, v, scale=1.0)
    assert out[0, 0, 0, 0] == pytest.approx(float(_fr(ex["output"])), rel=1e-14)
    assert lse[0, 0, 0] == pytest.approx(math.log(6.0), rel=1e-14)  # masses 1 + 3 + 2

    s = ex["split_after"]
    A = oracle_lib.block_summary(scores[:s], ex["values"][:s])
    B = oracle_lib.block_summary(scores[s:], ex["values"][s:])
    # separately normalised block outputs, and their unshifted masses l * e^m
    assert A[2] / A[1] == pytest.approx(ex["block_outputs"][0], rel=1e-14)
    assert B[2] / B[1] == pytest.approx(ex["block_outputs"][1], rel=1e-14)
    assert A[1] * math.exp(A[0]) == pytest.approx(ex["block_masses"][0], rel=1e-14)
    assert B[1] * math.exp(B[0]) == pytest.approx(ex["block_masses"][1], rel=1e-14)
    m, l, u = oracle_lib.merge(A, B)
    assert m == pytest.approx(math.log(ex["merged_at_common_max"]["m_ln"]), rel=1e-15)
    assert l == pytest.approx(float(_fr(ex["merged_at_common_max"]["l"])), rel=1e-14)
    assert u == pytest.approx(float(_fr(ex["merged_at_common_max"]["u"])), rel=1e-14)
    naive = sum(ex["block_outputs"]) / 2
    assert naive == pytest.approx(float(_fr(ex["wrong_simple_average"])))
    assert abs(u / l - naive) > 0.5
    # merge is symmetric in its arguments
    m2, l2, u2 = oracle_lib.merge(B, A)
    assert (m2, l2) == pytest.approx((m, l), rel=1e-15) and u2 == pytest.approx(u, rel=1e-15)


# ---------------------------------------------------------------- closed forms

def _exact(weights, values):
    """Exact softmax-weighted average: weights[i][j] >= 0 integers (0 = masked key),
    values[j][t] integers. Returns (out Fractions [Nq][dv], normaliser Fractions [Nq])."""
    outs, norms = [], []
    for wi in weights:
        z = sum(Fraction(w) for w in wi)
        norms.append(z)
        if z == 0:
            outs.append([Fraction(0)] * len(values[0]))
            continue
        outs.append([sum(Fraction(w) * Fraction(vj[t]) for w, vj in zip(wi, values)) / z
                     for t in range(len(values[0]))])
    return outs, norms


def _design(wk, uk, nq):
    """q_i = (1, i), k_j = (ln w_j, ln u_j): with scale 1, s_ij = ln(w_j * u_j**i)."""
    q = np.array([[1.0, float(i)] for i in range(nq)]).reshape(1, 1, nq, 2)
    k = np.array([[math.log(w), math.log(u)] for w, u in zip(wk, uk)]).reshape(1, 1, len(wk), 2)
    return q, k


def _check_exact(out, lse, W, vals, rel=1e-11):
    eo, ez = _exact(W, vals)
    for i in range(len(W)):
        for t in range(len(vals[0])):
            assert out[i, t] == pytest.approx(float(eo[i][t]), rel=rel, abs=1e-12), (i, t)
        if ez[i] == 0:
            assert lse[i] == -math.inf
        else:
            assert lse[i] == pytest.approx(math.log(ez[i]), rel=rel, abs=1e-12), i


def test_closed_form_two_dim_design(oracle_lib):
    wk, uk = [1, 2, 3, 5, 7], [1, 2, 1, 3, 2]
    vals = [[1, -2], [4, 0], [-3, 5], [2, 2], [0, 7]]
    nq = 4
    q, k = _design(wk, uk, nq)
    # values in a 2-wide head: d = 2 for q, k and v alike
    v = np.array(vals, dtype=np.float64).reshape(1, 1, len(wk), 2)
    out, lse = oracle_lib.attention(q, k, v, scale=1.0)
    W = [[w * u ** i for w, u in zip(wk, uk)] for i in range(nq)]
    _check_exact(out[0, 0], lse[0, 0], W, vals)


def test_closed_form_scale_is_applied(oracle_lib):
    # scale 1/2 on scores 2 ln w gives weights w: catches a dropped or squared scale
    wk, vals = [1, 4, 2], [[3, 1], [1, 1], [-1, 2]]
    q = np.array([[2.0, 0.0]]).reshape(1, 1, 1, 2)
    k = np.array([[math.log(w), 5.0] for w in wk]).reshape(1, 1, 3, 2)
    v = np.array(vals, dtype=np.float64).reshape(1, 1, 3, 2)
    out, lse = oracle_lib.attention(q, k, v, scale=0.5)
    _check_exact(out[0, 0], lse[0, 0], [wk], vals)


def test_closed_form_additive_mask(oracle_lib):
    wk, uk = [1, 2, 3, 4], [2, 1, 1, 3]
    vals = [[1, 0], [0, 1], [5, 5], [-1, 3]]
    C = [[1, 0, 2, 1], [0, 0, 0, 0], [3, 1, 0, 1]]  # 0 = -inf (masked), else ln C added
    nq = 3
    q, k = _design(wk, uk, nq)
    v = np.array(vals, dtype=np.float64).reshape(1, 1, 4, 2)
    mask = np.array([[math.log(c) if c else -math.inf for c in row] for row in C]).reshape(1, nq, 4)
    out, lse = oracle_lib.attention(q, k, v, mask=mask, scale=1.0)
    W = [[w * u ** i * c for w, u, c in zip(wk, uk, C[i])] for i in range(nq)]
    _check_exact(out[0, 0], lse[0, 0], W, vals)
    assert np.all(out[0, 0, 1] == 0.0) and lse[0, 0, 1] == -math.inf  # fully masked row


def test_closed_form_per_head_bias(oracle_lib):
    """Per-head bias [B, H, Nq, Nk]: every (b, h) gets its own integer bias matrix C
    (0 = -inf), so its weights are w_j u_j^i C[b][h][i][j]; a bias applied to the wrong
    head, batch index or row/key order breaks one of the closed forms."""
    B, H, nq = 2, 3, 3
    wk, uk = [1, 2, 3, 4], [2, 1, 1, 3]
    rng = np.random.default_rng(11)
    vals = [[[[int(x) for x in rng.integers(-5, 6, size=2)] for _ in range(4)] for _ in range(H)] for _ in range(B)]
    C = rng.integers(0, 4, size=(B, H, nq, 4))
    C[0, 1, 2] = 0  # one fully masked row
    qd, kd = _design(wk, uk, nq)
    q = np.broadcast_to(qd, (B, H, nq, 2)).copy()
    k = np.broadcast_to(kd, (B, H, 4, 2)).copy()
    v = np.array(vals, dtype=np.float64)
    bias = np.where(C > 0, np.log(np.maximum(C, 1)), -math.inf)
    out, lse = oracle_lib.attention_bias(q, k, v, bias, scale=1.0)
    for b in range(B):
        for h in range(H):
            W = [[w * u ** i * int(C[b, h, i, j]) for j, (w, u) in enumerate(zip(wk, uk))] for i in range(nq)]
            _check_exact(out[b, h], lse[b, h], W, vals[b][h])
    assert np.all(out[0, 1, 2] == 0.0) and lse[0, 1, 2] == -math.inf
    # a bias that is the same for every head is the shared mask
    shared = np.broadcast_to(bias[:, :1], bias.shape).copy()
    o2, l2 = oracle_lib.attention_bias(q, k, v, shared, scale=1.0)
    o3, l3 = oracle_lib.attention(q, k, v, mask=bias[:, 0], scale=1.0)
    np.testing.assert_array_equal(o2, o3)
    np.testing.assert_array_equal(l2, l3)


def test_closed_form_causal(oracle_lib):
    wk, uk = [1, 2, 3, 5], [3, 1, 2, 1]
    vals = [[2, 1], [-1, 4], [0, 0], [6, -6]]
    q, k = _design(wk, uk, 4)
    v = np.array(vals, dtype=np.float64).reshape(1, 1, 4, 2)
    out, lse = oracle_lib.attention(q, k, v, scale=1.0, causal=True)
    W = [[(w * u ** i if j <= i else 0) for j, (w, u) in enumerate(zip(wk, uk))] for i in range(4)]
    _check_exact(out[0, 0], lse[0, 0], W, vals)


def test_closed_form_causal_fewer_queries_than_keys(oracle_lib):
    # 2 queries against 4 keys: causal alignment puts the last query on the last key
    wk, uk = [1, 2, 3, 5], [3, 1, 2, 1]
    vals = [[2, 1], [-1, 4], [0, 0], [6, -6]]
    q, k = _design(wk, uk, 2)
    v = np.array(vals, dtype=np.float64).reshape(1, 1, 4, 2)
    out, lse = oracle_lib.attention(q, k, v, scale=1.0, causal=True)
    W = [[(w * u ** i if j <= i + 2 else 0) for j, (w, u) in enumerate(zip(wk, uk))] for i in range(2)]
    _check_exact(out[0, 0], lse[0, 0], W, vals)


def test_batch_and_head_indexing(oracle_lib):
    # every (b, h) gets its own closed-form problem; a mixed-up offset breaks one of them
    B, H, nq = 2, 3, 3
    rng = np.random.default_rng(7)
    q = np.zeros((B, H, nq, 2)); k = np.zeros((B, H, 4, 2)); v = np.zeros((B, H, 4, 2))
    mask = np.zeros((B, nq, 4))
    probs = {}
    for b in range(B):
        C = rng.integers(0, 3, size=(nq, 4)); C[:, 0] = 1 + b
        mask[b] = np.where(C > 0, np.log(np.maximum(C, 1)), -np.inf)
        for h in range(H):
            wk = list(rng.integers(1, 6, size=4)); uk = list(rng.integers(1, 4, size=4))
            vals = rng.integers(-5, 6, size=(4, 2)).tolist()
            qq, kk = _design(wk, uk, nq)
            q[b, h], k[b, h] = qq[0, 0], kk[0, 0]
            v[b, h] = np.array(vals, dtype=np.float64)
            probs[b, h] = ([[int(w) * int(u) ** i * int(C[i, j]) for j, (w, u) in enumerate(zip(wk, uk))]
                            for i in range(nq)], vals)
    out, lse = oracle_lib.attention(q, k, v, mask=mask, scale=1.0)
    for (b, h), (W, vals) in probs.items():
        _check_exact(out[b, h], lse[b, h], W, vals)
    # the row-subset routine must index the same rows
    rows = [(b * H + h) * nq + i for b in range(B) for h in range(H) for i in range(nq)][::-1]
    o_r, l_r = oracle_lib.attention_rows(q, k, v, rows, mask=mask, scale=1.0)
    np.testing.assert_array_equal(o_r, out.reshape(-1, 2)[rows])
    np.testing.assert_array_equal(l_r, lse.reshape(-1)[rows])


# ---------------------------------------------------------------- special cases

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_gives_means(oracle_lib, causal):
    B, H, N, d = 2, 2, 9, 5
    q, k, v = _rand((B, H, N, d), 1), _rand((B, H, N, d), 2), _rand((B, H, N, d), 3)
    out, lse = oracle_lib.attention(q, k, v, scale=0.0, causal=causal)
    for i in range(N):
        cnt = i + 1 if causal else N
        np.testing.assert_allclose(out[:, :, i], v[:, :, :cnt].mean(axis=2), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, i], math.log(cnt), rtol=1e-14)


def test_causal_first_row_and_single_key(oracle_lib):
    B, H, N, d = 1, 3, 7, 4
    q, k, v = _rand((B, H, N, d), 4), _rand((B, H, N, d), 5), _rand((B, H, N, d), 6)
    out, lse = oracle_lib.attention(q, k, v, scale=0.3, causal=True)
    np.testing.assert_allclose(out[:, :, 0], v[:, :, 0], rtol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), rtol=1e-13)
    out1, lse1 = oracle_lib.attention(q[:, :, :1], k[:, :, :1], v[:, :, :1], scale=0.3)
    np.testing.assert_allclose(out1, v[:, :, :1], rtol=1e-14)


def test_constant_values_and_unit_weights(oracle_lib):
    B, H, N, d = 1, 2, 33, 8
    q, k = _rand((B, H, N, d), 8) * 3, _rand((B, H, N, d), 9) * 3
    c = _rand((B, H, 1, d), 10)
    out, _ = oracle_lib.attention(q, k, np.repeat(c, N, axis=2), scale=0.7, causal=True)
    np.testing.assert_allclose(out, np.repeat(c, N, axis=2), rtol=1e-12, atol=1e-13)
    out1, _ = oracle_lib.attention(q, k, np.ones((B, H, N, d)), scale=0.7)
    np.testing.assert_allclose(out1, 1.0, rtol=1e-13)


def test_fully_masked_rows(oracle_lib):
    B, H, N, d = 2, 2, 6, 3
    q, k, v = _rand((B, H, N, d), 11), _rand((B, H, N, d), 12), _rand((B, H, N, d), 13)
    mask = np.zeros((B, N, N))
    mask[0, 2, :] = -np.inf
    mask[1, 5, :] = -np.inf
    out, lse = oracle_lib.attention(q, k, v, mask=mask, scale=0.5)
    assert np.all(out[0, :, 2] == 0.0) and np.all(lse[0, :, 2] == -np.inf)
    assert np.all(out[1, :, 5] == 0.0) and np.all(lse[1, :, 5] == -np.inf)
    assert np.all(np.isfinite(lse[0, :, [0, 1, 3, 4, 5]]))
    ob, lb = oracle_lib.attention_blockwise(q, k, v, block=2, mask=mask, scale=0.5)
    np.testing.assert_array_equal(ob[0, :, 2], 0.0)
    assert np.all(lb[1, :, 5] == -np.inf)


# ---------------------------------------------------------------- invariants

def test_mask_row_shift(oracle_lib):
    B, H, N, d = 2, 3, 17, 6
    q, k, v = _rand((B, H, N, d), 20), _rand((B, H, N, d), 21), _rand((B, H, N, d), 22)
    mask = np.where(np.random.default_rng(23).random((B, N, N)) < 0.2, -np.inf, 0.0)
    c = _rand((B, N, 1), 24) * 5
    o1, l1 = oracle_lib.attention(q, k, v, mask=mask, scale=0.4, causal=True)
    o2, l2 = oracle_lib.attention(q, k, v, mask=mask + c, scale=0.4, causal=True)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    fin = np.isfinite(l1)
    np.testing.assert_allclose(l2[fin], (l1 + c[:, None, :, 0])[fin], rtol=1e-12)
    assert np.array_equal(fin, np.isfinite(l2))


def test_key_value_permutation(oracle_lib):
    B, H, N, d = 1, 2, 40, 8
    q, k, v = _rand((B, H, N, d), 30), _rand((B, H, N, d), 31), _rand((B, H, N, d), 32)
    perm = np.random.default_rng(33).permutation(N)
    o1, l1 = oracle_lib.attention(q, k, v, scale=0.5)
    o2, l2 = oracle_lib.attention(q, k[:, :, perm], v[:, :, perm], scale=0.5)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-13)
    # a key-only permutation must change the result (catches a k/v index mix-up)
    o3, _ = oracle_lib.attention(q, k[:, :, perm], v, scale=0.5)
    assert np.abs(o3 - o1).max() > 1e-3


def test_large_scores_are_stable(oracle_lib):
    # the maximum is subtracted: adding 900 to every score of a row must not overflow
    wk, uk = [1, 2, 3], [1, 1, 1]
    q, k = _design(wk, uk, 1)
    v = np.array([[1, 0], [0, 1], [2, 2]], dtype=np.float64).reshape(1, 1, 3, 2)
    mask = np.full((1, 1, 3), 900.0)
    out, lse = oracle_lib.attention(q, k, v, mask=mask, scale=1.0)
    _check_exact(out[0, 0], lse[0, 0] - 900.0, [[1, 2, 3]], [[1, 0], [0, 1], [2, 2]], rel=1e-12)


# ---------------------------------------------------------------- blockwise = materialised

@pytest.mark.parametrize("block", [1, 2, 3, 64, 129])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_matches_materialised(oracle_lib, block, causal):
    B, H, N, d = 2, 2, 129, 16
    q, k, v = _rand((B, H, N, d), 40) * 2, _rand((B, H, N, d), 41), _rand((B, H, N, d), 42)
    mask = np.where(np.random.default_rng(43).random((B, N, N)) < 0.1, -np.inf, 0.0)
    mask[1, 7, :] = -np.inf
    o1, l1 = oracle_lib.attention(q, k, v, mask=mask, scale=0.25, causal=causal)
    o2, l2 = oracle_lib.attention_blockwise(q, k, v, block=block, mask=mask, scale=0.25, causal=causal)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isfinite(l1), np.isfinite(l2))
    fin = np.isfinite(l1)
    np.testing.assert_allclose(l2[fin], l1[fin], rtol=1e-12)


def test_merge_with_empty_blocks(oracle_lib):
    e = (-math.inf, 0.0, 0.0)
    a = (math.log(2.0), 1.5, 2.5)
    assert oracle_lib.merge(e, e) == (-math.inf, 0.0, 0.0)
    m, l, u = oracle_lib.merge(e, a)
    assert (m, l, u) == pytest.approx(a)
    m, l, u = oracle_lib.merge(a, e)
    assert (m, l, u) == pytest.approx(a)
    assert oracle_lib.block_summary([-math.inf, -math.inf], [1.0, 2.0]) == (-math.inf, 0.0, 0.0)


# ---------------------------------------------------------------- backward

def test_backward_matches_finite_differences(oracle_lib):
    B, H, N, d = 1, 2, 5, 3
    q, k, v = _rand((B, H, N, d), 50), _rand((B, H, N, d), 51), _rand((B, H, N, d), 52)
    do = _rand((B, H, N, d), 53)
    mask = np.zeros((B, N, N)); mask[0, 1, 3] = -np.inf; mask[0, 4, 0] = 0.7
    for causal in (False, True):
        dq, dk, dv = oracle_lib.attention_bwd(q, k, v, do, mask=mask, scale=0.6, causal=causal)

        def f(qq, kk, vv):
            o, _ = oracle_lib.attention(qq, kk, vv, mask=mask, scale=0.6, causal=causal)
            return float((o * do).sum())

        eps = 1e-6
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy(); xp[idx] += eps
                xm = x.copy(); xm[idx] -= eps
                args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
                ap = [xp if n == name else a for n, a in zip("qkv", args)]
                am = [xm if n == name else a for n, a in zip("qkv", args)]
                num[idx] = (f(*ap) - f(*am)) / (2 * eps)
            np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=f"d{name} causal={causal}")


def test_backward_zero_scale_closed_form(oracle_lib):
    B, H, N, d = 1, 1, 6, 4
    q, k, v, do = (_rand((B, H, N, d), s) for s in (60, 61, 62, 63))
    dq, dk, dv = oracle_lib.attention_bwd(q, k, v, do, scale=0.0)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)
    # uniform weights 1/N: every key collects the mean of dO
    np.testing.assert_allclose(dv, np.repeat(do.mean(axis=2, keepdims=True), N, axis=2), rtol=1e-13)


def test_rejects_bad_shapes(oracle_lib):
    q = np.zeros((1, 1, 4, 8))
    with pytest.raises(ValueError):
        oracle_lib.attention(q, np.zeros((1, 1, 4, 4)), np.zeros((1, 1, 4, 4)))
    with pytest.raises(ValueError):
        oracle_lib.attention(q, q, q, mask=np.zeros((1, 4, 5)))


# ---------------------------------------------------------------- dropout
# The keep stream is Philox4x64-10 (Salmon et al., SC 2011); numpy's Philox bit
# generator is an independent implementation of the same published algorithm. It
# advances its counter once before producing a block, so its output for counter c is
# the block of counter c + 1.

@pytest.mark.parametrize("counter,key", [
    ([0, 0, 0, 0], [0, 0]),
    ([7, 11, 13, 17], [3, 5]),
    ([2**64 - 2, 2**64 - 1, 5, 2**63], [2**64 - 1, 12345]),  # carry out of word 0 into word 1
    ([123456789, 0, 42, 9], [0xDEADBEEF, 0]),
])
def test_philox_matches_numpy(oracle_lib, counter, key):
    assert list(oracle_lib.philox4x64_10(counter, key)) == _numpy_philox_block(counter, key)


def _as_int(words):
    return sum(int(w) << (64 * n) for n, w in enumerate(words))


def _numpy_philox_block(counter, key):
    """numpy's Philox output for the block at `counter` (it steps the 256-bit counter by
    one first; counter and key are passed as Python integers, which numpy takes exactly)."""
    bg = np.random.Philox(key=_as_int(key), counter=(_as_int(counter) - 1) % 2**256)
    return [int(x) for x in bg.random_raw(4)]


def test_dropout_keep_stream_through_numpy(oracle_lib):
    """Every keep decision of a small problem, recomputed from numpy's Philox with the
    stated counter layout {i, j div 32, b*H + h, offset}, key {seed, 0}, bytes from
    the low byte of word 0 upward."""
    B, H, Nq, Nk, p, seed, offset = 2, 3, 5, 70, 0.3, 987654321, 17
    keep = oracle_lib.dropout_keep(B, H, Nq, Nk, p, seed, offset)
    t = oracle_lib.dropout_threshold(p)
    assert t == 179  # 0.7 * 256 = 179.2
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                for g in range((Nk + 31) // 32):
                    words = _numpy_philox_block([i, g, b * H + h, offset], [seed, 0])
                    for tt in range(min(32, Nk - 32 * g)):
                        byte = (words[tt // 8] >> (8 * (tt % 8))) & 0xFF
                        assert keep[b, h, i, 32 * g + tt] == (byte < t), (b, h, i, g, tt)


def test_dropout_threshold_rounding(oracle_lib):
    assert oracle_lib.dropout_threshold(0.0) == 256
    assert oracle_lib.dropout_threshold(0.5) == 128
    assert oracle_lib.dropout_threshold(0.1) == 230  # 230.4
    assert oracle_lib.dropout_threshold(1 - 0.5 / 256) == 1  # 0.5 rounds up
    with pytest.raises(ValueError):
        oracle_lib.dropout_threshold(0.999)  # keeps nothing
    with pytest.raises(ValueError):
        oracle_lib.dropout_threshold(-0.001)


def test_dropout_zero_is_attention(oracle_lib):
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((2, 2, 37, 16)) for _ in range(3))
    for causal in (False, True):
        o0, l0 = oracle_lib.attention(q, k, v, scale=0.3, causal=causal)
        o1, l1 = oracle_lib.attention_dropout(q, k, v, 0.0, seed=5, scale=0.3, causal=causal)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_dropout_weights_through_identity_values(oracle_lib):
    """With V = I (Nk = d) each output row is the row's weights: the undropped
    softmax probabilities times keep / q, not renormalised over the kept keys; lse is
    the undropped one."""
    rng = np.random.default_rng(4)
    B, H, N = 1, 2, 48
    q, k = rng.standard_normal((B, H, N, N)), rng.standard_normal((B, H, N, N))
    v = np.broadcast_to(np.eye(N), (B, H, N, N)).copy()
    for causal in (False, True):
        P, l0 = oracle_lib.attention(q, k, v, scale=0.2, causal=causal)  # V = I: out is P
        o, l1 = oracle_lib.attention_dropout(q, k, v, 0.25, seed=77, offset=3, scale=0.2, causal=causal)
        keep = oracle_lib.dropout_keep(B, H, N, N, 0.25, 77, 3)
        assert np.array_equal(l0, l1)
        np.testing.assert_allclose(o, P * keep * (256 / 192), rtol=1e-12, atol=1e-15)


def test_dropout_is_unbiased_over_seeds(oracle_lib):
    """The mean over many seeds approaches the undropped output (E[keep / q] = 1)."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 1, 8, 8)) for _ in range(3))
    o0, _ = oracle_lib.attention(q, k, v, scale=0.5)
    acc = np.zeros_like(o0)
    n = 3000
    for s in range(n):
        acc += oracle_lib.attention_dropout(q, k, v, 0.5, seed=s, scale=0.5)[0]
    assert np.max(np.abs(acc / n - o0)) < 0.08


def test_dropout_keep_fraction(oracle_lib):
    keep = oracle_lib.dropout_keep(2, 4, 256, 256, 0.2, seed=2024)
    t = oracle_lib.dropout_threshold(0.2)
    frac, n = keep.mean(), keep.size
    assert abs(frac - t / 256) < 5 * math.sqrt((t / 256) * (1 - t / 256) / n)
    # different seeds, offsets and heads give different streams
    assert not np.array_equal(keep, oracle_lib.dropout_keep(2, 4, 256, 256, 0.2, seed=2025))
    assert not np.array_equal(keep, oracle_lib.dropout_keep(2, 4, 256, 256, 0.2, seed=2024, offset=1))
    assert not np.array_equal(keep[0, 0], keep[0, 1])
