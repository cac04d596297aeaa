"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print for a worked example (``tests/golden``), closed forms, invariants
stated on the pages, finite differences of the forward, or a small
independent brute force.  Chosen so that a dropped term, a wrong sign, a
wrong mask direction, a transposed operand or a missing scale factor anywhere
in the oracle fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import (
    attention_backward,
    attention_backward_head,
    attention_backward_rows,
    attention_forward,
    attention_forward_head,
    attention_forward_rows,
    causal_mask,
    matmul_backward,
    merge_outputs,
    merge_partials,
    merge_stats,
    naive_softmax,
    online_softmax_steps,
    softmax_3pass,
    softmax_backward,
    tiled_forward_head,
)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- online softmax


def test_worked_example_online_steps(golden_dir):
    """Flash Attention page, 2.Online Softmax §六: step table for x = [1, 3, 2, 5]."""
    g = _load(golden_dir, "online_softmax_worked_example.json")
    tol = 0.5 * 10 ** -g["printed_decimals"] + 1e-12
    steps = online_softmax_steps(g["x"])
    assert len(steps) == len(g["steps"])
    for (m, factor, ell), want in zip(steps, g["steps"]):
        assert m == want["m"]
        assert abs(factor - want["factor"]) <= tol
        assert abs(ell - want["l"]) <= tol
    # the standard (3-pass) column of the same example
    y, m3, l3 = softmax_3pass(np.array(g["x"], dtype=float))
    assert m3 == g["standard"]["m"]
    assert abs(l3 - g["standard"]["l"]) <= tol
    for t, want in zip(np.exp(np.array(g["x"]) - m3), g["standard"]["terms"]):
        assert abs(t - want) <= tol
    # exactness claim (§五): online and 3-pass agree to rounding
    assert abs(steps[-1][2] - l3) <= 1e-12
    assert abs(y.sum() - 1.0) <= 1e-15


def test_merge_associative_and_equal_to_3pass():
    """2.Online Softmax §3.1: the two-block merge is associative and exact."""
    rng = _rng(11)
    x = rng.uniform(-50.0, 50.0, size=1000)
    _, m_ref, l_ref = softmax_3pass(x)
    cuts = np.sort(rng.choice(np.arange(1, 1000), size=17, replace=False))
    blocks = np.split(x, cuts)
    stats = [(b.max(), np.exp(b - b.max()).sum()) for b in blocks]

    left = (-math.inf, 0.0)
    for s in stats:
        left = merge_stats(*left, *s)
    right = (-math.inf, 0.0)
    for s in reversed(stats):
        right = merge_stats(*s, *right)

    def tree(items):
        if len(items) == 1:
            return items[0]
        mid = len(items) // 2
        return merge_stats(*tree(items[:mid]), *tree(items[mid:]))

    for m, ell in (left, right, tree(stats)):
        assert m == m_ref
        assert abs(ell - l_ref) <= 1e-13 * l_ref


def test_merge_outputs_matches_definition():
    """2.Online Softmax §4.1: merging unnormalised outputs gives softmax(x)·V."""
    rng = _rng(12)
    x = rng.normal(size=300) * 5
    v = rng.normal(size=(300, 7))
    y, _, _ = softmax_3pass(x)
    a, b = slice(0, 113), slice(113, 300)
    ma, mb = x[a].max(), x[b].max()
    la, lb = np.exp(x[a] - ma).sum(), np.exp(x[b] - mb).sum()
    oa, ob = np.exp(x[a] - ma) @ v[a], np.exp(x[b] - mb) @ v[b]
    m, ell, o = merge_outputs(ma, la, oa, mb, lb, ob)
    np.testing.assert_allclose(o / ell, y @ v, rtol=0, atol=1e-13)
    # an empty block (-inf, 0, 0) is the identity of the merge
    m2, l2, o2 = merge_outputs(-math.inf, 0.0, np.zeros(7), ma, la, oa)
    assert m2 == ma and l2 == la
    np.testing.assert_array_equal(o2, oa)


def test_softmax_rows_sum_to_one():
    """附录A 结论二 一: Σ_i p_i = 1 and p_i > 0."""
    rng = _rng(13)
    x = rng.normal(size=(64, 333)) * 20
    y, _, _ = softmax_3pass(x)
    assert np.all(y > 0)
    assert np.max(np.abs(y.sum(axis=1) - 1.0)) <= 1e-12


def test_overflow_and_shift_invariance():
    """2.Online Softmax §1.2-1.3 and the cnnetsun.cn page §2.1: x = 1000 overflows
    the naive form; the max-subtracted form is finite and shift invariant."""
    x = np.array([1000.0, 999.0, 10.0, -1000.0])
    assert not np.all(np.isfinite(naive_softmax(x)))      # negative control
    y, m, ell = softmax_3pass(x)
    assert np.all(np.isfinite(y)) and m == 1000.0
    y2, _, _ = softmax_3pass(x - 777.25)
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=0)
    # attention level: adding t·e_0 to every key shifts row i's scores by
    # scale·t·q_i0, a per-row constant, so O is unchanged and LSE moves by it.
    rng = _rng(14)
    n, d = 40, 16
    scale = d ** -0.5
    q, k, v = rng.normal(size=(n, d)), rng.normal(size=(n, d)), rng.normal(size=(n, d))
    q[:, 0] = rng.choice([-1.0, 1.0], size=n) * rng.uniform(0.5, 1.0, size=n)
    t = 4000.0
    k2 = k.copy()
    k2[:, 0] += t
    for causal in (False, True):
        o, lse = attention_forward_head(q, k, v, scale, causal)
        o2, lse2 = attention_forward_head(q, k2, v, scale, causal)
        assert np.all(np.isfinite(o2)) and np.all(np.isfinite(lse2))
        assert np.max(np.abs(scale * t * q[:, 0])) > 1e3 * 0.9
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-9)
        np.testing.assert_allclose(lse2 - scale * t * q[:, 0], lse, rtol=1e-12, atol=1e-9)


# ---------------------------------------------------------------- forward closed forms


def test_two_key_worked_example(golden_dir):
    """附录A 结论二 七's numbers embedded in one head pin the scale, O, LSE and all
    three gradients (see the fixture's construction)."""
    g = _load(golden_dir, "attention_two_key_example.json")
    q, k, v, do = (np.array(g[x], dtype=float) for x in ("q", "k", "v", "do"))
    o, lse = attention_forward_head(q, k, v, g["scale"])
    dq, dk, dv = attention_backward_head(q, k, v, do, g["scale"])
    e = g["expected"]
    tol = g["tolerance"]
    np.testing.assert_allclose(o, e["O"], atol=tol, rtol=0)
    np.testing.assert_allclose(lse, e["LSE"], atol=tol, rtol=0)
    np.testing.assert_allclose(dv, e["dV"], atol=tol, rtol=0)
    np.testing.assert_allclose(dq, e["dQ"], atol=tol, rtol=0)
    np.testing.assert_allclose(dk, e["dK"], atol=tol, rtol=0)


def test_two_key_closed_form():
    """Two visible keys: p_1 is the logistic of the score gap, LSE = ln(e^{s1}+e^{s2})."""
    rng = _rng(15)
    d = 8
    scale = 0.37
    q, k, v = rng.normal(size=(1, d)), rng.normal(size=(2, d)), rng.normal(size=(2, d))
    s1, s2 = scale * float(q[0] @ k[0]), scale * float(q[0] @ k[1])
    p1 = 1.0 / (1.0 + math.exp(s2 - s1))
    o, lse = attention_forward_head(q, k, v, scale)
    np.testing.assert_allclose(o[0], p1 * v[0] + (1 - p1) * v[1], atol=1e-14, rtol=0)
    assert abs(lse[0] - math.log(math.exp(s1) + math.exp(s2))) <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    """Rows of P sum to one, so V_j = c for all j gives O_i = c."""
    rng = _rng(16)
    n, d = 50, 12
    q, k = rng.normal(size=(n, d)) * 3, rng.normal(size=(n, d)) * 3
    c = rng.normal(size=d)
    o, _ = attention_forward_head(q, k, np.tile(c, (n, 1)), d ** -0.5, causal)
    assert np.max(np.abs(o - c)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_v(causal):
    """K_j = k for all j makes P uniform over the visible keys: O_i = mean_{j visible} V_j."""
    rng = _rng(17)
    n, d = 45, 10
    q = rng.normal(size=(n, d))
    k = np.tile(rng.normal(size=d), (n, 1))
    v = rng.normal(size=(n, d))
    o, lse = attention_forward_head(q, k, v, d ** -0.5, causal)
    if causal:
        want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
        count = np.arange(1, n + 1)
    else:
        want = np.tile(v.mean(axis=0), (n, 1))
        count = np.full(n, n)
    assert np.max(np.abs(o - want)) <= 1e-12
    s = (d ** -0.5) * (q @ k[0])
    np.testing.assert_allclose(lse, s + np.log(count), atol=1e-12, rtol=0)


def test_causal_mask_direction():
    """Key j is visible to query i iff j <= i; the first query sees only key 0."""
    m = causal_mask(4, 4)
    assert m[0].tolist() == [True, False, False, False]
    assert m[3].tolist() == [True, True, True, True]
    rng = _rng(18)
    q, k, v = rng.normal(size=(6, 4)), rng.normal(size=(6, 4)), rng.normal(size=(6, 4))
    o, lse = attention_forward_head(q, k, v, 0.5, causal=True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15, rtol=0)
    assert abs(lse[0] - 0.5 * float(q[0] @ k[0])) <= 1e-15


def _brute_force_head(q, k, v, scale, causal):
    """Scalar loops with math.exp; independent of numpy's vectorised path.
    With fewer queries than keys, query i stands at position i + len(k) - len(q)."""
    n, d = len(q), len(q[0])
    pos0 = len(k) - n
    o, lse = [], []
    for i in range(n):
        keys = [j for j in range(len(k)) if (not causal or j <= i + pos0)]
        s = [scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in keys]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        z = math.fsum(w)
        o.append([math.fsum(w[a] * v[j][t] for a, j in enumerate(keys)) / z for t in range(len(v[0]))])
        lse.append(mx + math.log(z))
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_scalar_brute_force(causal):
    rng = _rng(19)
    q, k, v = rng.normal(size=(7, 5)), rng.normal(size=(7, 5)), rng.normal(size=(7, 5))
    o, lse = attention_forward_head(q, k, v, 0.61, causal)
    ob, lseb = _brute_force_head(q.tolist(), k.tolist(), v.tolist(), 0.61, causal)
    np.testing.assert_allclose(o, ob, atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse, lseb, atol=1e-14, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 7, 32, 64, 300])
def test_tiled_algorithm_equals_definition(causal, block):
    """2.Online Softmax §4.2 + §五: the one-pass tiled forward reaches the same O and
    LSE as the materialised definition (ragged last block included)."""
    rng = _rng(20 + block)
    n, d = 150, 16
    q, k, v = rng.normal(size=(n, d)) * 2, rng.normal(size=(n, d)) * 2, rng.normal(size=(n, d))
    o, lse = attention_forward_head(q, k, v, d ** -0.5, causal)
    ot, lset = tiled_forward_head(q, k, v, d ** -0.5, block, causal)
    np.testing.assert_allclose(ot, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lset, lse, atol=1e-12, rtol=0)


def test_self_test_shape_of_cnnetsun_page():
    """cnnetsun.cn page §4 self-test shape (1, 256, 64), scale 64^-0.5, block 128."""
    rng = _rng(42)
    q, k, v = rng.normal(size=(256, 64)), rng.normal(size=(256, 64)), rng.normal(size=(256, 64))
    o, lse = attention_forward_head(q, k, v, 64 ** -0.5)
    ot, lset = tiled_forward_head(q, k, v, 64 ** -0.5, 128)
    assert np.max(np.abs(o - ot)) <= 1e-13 and np.max(np.abs(lse - lset)) <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_row_subset_equals_full(causal):
    rng = _rng(21)
    q, k, v = rng.normal(size=(64, 8)), rng.normal(size=(64, 8)), rng.normal(size=(64, 8))
    rows = [0, 5, 17, 63]
    o, lse = attention_forward_head(q, k, v, 0.3, causal)
    orow, lserow = attention_forward_rows(q, k, v, rows, 0.3, causal)
    np.testing.assert_allclose(orow, o[rows], atol=1e-14, rtol=0)
    np.testing.assert_allclose(lserow, lse[rows], atol=1e-14, rtol=0)


# ---------------------------------------------------------------- backward pins


def test_matmul_gradient_example(golden_dir):
    """附录A 结论一 七 (1x2 example) and the 八 table row for Y = A Bᵀ."""
    g = _load(golden_dir, "matmul_gradient_worked_example.json")
    da, db = matmul_backward(g["A"], g["B"], g["dY"])
    np.testing.assert_array_equal(da, g["dA"])
    np.testing.assert_array_equal(db, g["dB"])
    rng = _rng(22)
    a, b, dy = rng.normal(size=(3, 4)), rng.normal(size=(5, 4)), rng.normal(size=(3, 5))
    da, dbt = matmul_backward(a, b.T, dy)       # Y = A Bᵀ
    np.testing.assert_allclose(da, dy @ b, atol=1e-14, rtol=0)
    np.testing.assert_allclose(dbt.T, dy.T @ a, atol=1e-14, rtol=0)


def test_softmax_backward_example(golden_dir):
    """附录A 结论二 七: s = (1, 2), dp = (1, 0) gives ds ≈ (0.197, -0.197)."""
    g = _load(golden_dir, "softmax_backward_worked_example.json")
    tol = 0.5 * 10 ** -g["printed_decimals"] + 1e-12
    p, _, _ = softmax_3pass(np.array(g["s"], dtype=float))
    np.testing.assert_allclose(p, g["p"], atol=tol, rtol=0)
    ds = softmax_backward(p, np.array(g["dp"], dtype=float))
    np.testing.assert_allclose(ds, g["ds"], atol=tol, rtol=0)
    assert abs(float(p @ np.array(g["dp"])) - g["rho"]) <= tol
    # the exact value: p1 (1 - p1) = e / (1 + e)^2
    exact = math.e / (1.0 + math.e) ** 2
    assert abs(ds[0] - exact) <= 1e-15 and abs(ds[1] + exact) <= 1e-15
    # the Jacobian built column by column from unit upstream gradients
    jac = np.stack([softmax_backward(p, np.eye(2)[c]) for c in range(2)], axis=1)
    np.testing.assert_allclose(jac, g["J"], atol=tol, rtol=0)


def test_softmax_jacobian_properties():
    """附录A 结论二 2.4 / 5.3 / 九: column sums of J are 0, constant dp gives ds = 0,
    and the cross-entropy upstream gradient gives ds = p - y."""
    rng = _rng(23)
    s = rng.normal(size=9) * 3
    p, _, _ = softmax_3pass(s)
    jac = np.stack([softmax_backward(p, np.eye(9)[c]) for c in range(9)], axis=1)
    np.testing.assert_allclose(jac, np.diag(p) - np.outer(p, p), atol=1e-15, rtol=0)
    assert np.max(np.abs(jac.sum(axis=0))) <= 1e-15
    assert np.max(np.abs(softmax_backward(p, np.full(9, 3.7)))) <= 1e-14
    y = np.zeros(9)
    y[4] = 1.0
    np.testing.assert_allclose(softmax_backward(p, -y / p), p - y, atol=1e-14, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_d_identity(causal):
    """"反向传播的公式推导" 五: rowsum(dP ⊙ P) = rowsum(dO ⊙ O)."""
    rng = _rng(24)
    n, d = 70, 16
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    o, _ = attention_forward_head(q, k, v, d ** -0.5, causal)
    *_, mid = attention_backward_head(q, k, v, do, d ** -0.5, causal, return_intermediates=True)
    lhs = (mid["dP"] * mid["P"]).sum(axis=1)
    rhs = (do * o).sum(axis=1)
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * max(1.0, np.max(np.abs(rhs)))


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    """Σ_j dS_ij = 0 (constant-dp invariance), hence Σ_j dK_j = 0; rows of P sum to
    one, hence Σ_j dV_j = Σ_i dO_i."""
    rng = _rng(25)
    n, d = 60, 16
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    dq, dk, dv, mid = attention_backward_head(q, k, v, do, d ** -0.5, causal, return_intermediates=True)
    assert np.max(np.abs(mid["dS"].sum(axis=1))) <= 1e-12
    assert np.max(np.abs(dk.sum(axis=0))) <= 1e-11
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-11, rtol=0)


def _loss(q, k, v, do, scale, causal):
    o, _ = attention_forward_head(q, k, v, scale, causal)
    return float((do * o).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [4, 8])
def test_finite_difference_gradients(causal, n):
    """Central differences of L = Σ dO ⊙ O (h = 1e-6) against dQ, dK, dV."""
    rng = _rng(26 + n)
    d = 4
    scale = 0.7
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    grads = attention_backward_head(q, k, v, do, scale, causal)
    h = 1e-6
    for which, g in zip(range(3), grads):
        fd = np.zeros((n, d))
        for i in range(n):
            for t in range(d):
                args = [q.copy(), k.copy(), v.copy()]
                args[which][i, t] += h
                up = _loss(*args, do, scale, causal)
                args[which][i, t] -= 2 * h
                dn = _loss(*args, do, scale, causal)
                fd[i, t] = (up - dn) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert err <= 1e-6, (which, err)


@pytest.mark.parametrize("causal", [False, True])
def test_row_block_backward_sums_to_full(causal):
    """Row blocks of the backward: dQ rows are exact and the dK, dV shares of a
    partition of the rows add up to the full gradients."""
    rng = _rng(27)
    n, d = 48, 8
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    dq, dk, dv = attention_backward_head(q, k, v, do, 0.4, causal)
    dk_sum, dv_sum = np.zeros_like(dk), np.zeros_like(dv)
    for block in (np.arange(0, 5), np.arange(5, 31), np.arange(31, 48)):
        dq_r, dk_r, dv_r = attention_backward_rows(q, k, v, do, block, 0.4, causal)
        np.testing.assert_allclose(dq_r, dq[block], atol=1e-14, rtol=0)
        dk_sum += dk_r
        dv_sum += dv_r
    np.testing.assert_allclose(dk_sum, dk, atol=1e-13, rtol=0)
    np.testing.assert_allclose(dv_sum, dv, atol=1e-13, rtol=0)


# ---------------------------------------------------------------- fewer queries than keys, merges


def test_causal_mask_with_fewer_queries_than_keys():
    """Queries are the last positions: 3 queries over 5 keys see 3, 4 and 5 keys;
    the square mask is the lower triangle; more queries than keys is rejected."""
    assert causal_mask(3, 5).astype(int).tolist() == [[1, 1, 1, 0, 0], [1, 1, 1, 1, 0], [1, 1, 1, 1, 1]]
    assert np.array_equal(causal_mask(6, 6), np.tril(np.ones((6, 6), dtype=bool)))
    with pytest.raises(ValueError):
        causal_mask(4, 3)


@pytest.mark.parametrize("causal", [False, True])
def test_fewer_queries_matches_scalar_brute_force(causal):
    rng = _rng(40)
    q, k, v = rng.normal(size=(4, 5)), rng.normal(size=(9, 5)), rng.normal(size=(9, 6))
    o, lse = attention_forward_head(q, k, v, 0.55, causal)
    ob, lseb = _brute_force_head(q.tolist(), k.tolist(), v.tolist(), 0.55, causal)
    np.testing.assert_allclose(o, ob, atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse, lseb, atol=1e-14, rtol=0)


def test_suffix_queries_equal_rows_of_the_square_problem():
    """The last n_q queries of a square causal problem, run alone over all keys,
    give that problem's last n_q rows of O and LSE; with dO zero on the other
    rows, its dQ rows and its whole dK, dV as well."""
    rng = _rng(41)
    n, n_q, d = 40, 13, 8
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    do[: n - n_q] = 0.0
    o, lse = attention_forward_head(q, k, v, 0.4, causal=True)
    dq, dk, dv = attention_backward_head(q, k, v, do, 0.4, causal=True)
    o_s, lse_s = attention_forward_head(q[n - n_q:], k, v, 0.4, causal=True)
    dq_s, dk_s, dv_s = attention_backward_head(q[n - n_q:], k, v, do[n - n_q:], 0.4, causal=True)
    np.testing.assert_allclose(o_s, o[n - n_q:], atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse_s, lse[n - n_q:], atol=1e-14, rtol=0)
    np.testing.assert_allclose(dq_s, dq[n - n_q:], atol=1e-13, rtol=0)
    np.testing.assert_allclose(dk_s, dk, atol=1e-13, rtol=0)
    np.testing.assert_allclose(dv_s, dv, atol=1e-13, rtol=0)


def test_single_query_causal_sees_every_key():
    """One query after n_k - 1 cached keys (a decode step) sees all keys."""
    rng = _rng(42)
    q, k, v = rng.normal(size=(1, 8)), rng.normal(size=(30, 8)), rng.normal(size=(30, 8))
    o_c, lse_c = attention_forward_head(q, k, v, 0.3, causal=True)
    o_n, lse_n = attention_forward_head(q, k, v, 0.3, causal=False)
    np.testing.assert_allclose(o_c, o_n, atol=0, rtol=0)
    np.testing.assert_allclose(lse_c, lse_n, atol=0, rtol=0)


@pytest.mark.parametrize("block", [1, 6, 32])
def test_tiled_algorithm_with_fewer_queries(block):
    rng = _rng(43 + block)
    q, k, v = rng.normal(size=(21, 8)) * 2, rng.normal(size=(70, 8)) * 2, rng.normal(size=(70, 8))
    o, lse = attention_forward_head(q, k, v, 8 ** -0.5, causal=True)
    ot, lset = tiled_forward_head(q, k, v, 8 ** -0.5, block, causal=True)
    np.testing.assert_allclose(ot, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lset, lse, atol=1e-12, rtol=0)


def test_row_subsets_with_fewer_queries():
    rng = _rng(44)
    q, k, v, do = rng.normal(size=(20, 8)), rng.normal(size=(50, 8)), rng.normal(size=(50, 8)), rng.normal(size=(20, 8))
    rows = np.array([0, 7, 19])
    o, lse = attention_forward_head(q, k, v, 0.3, causal=True)
    orow, lserow = attention_forward_rows(q, k, v, rows, 0.3, causal=True)
    np.testing.assert_allclose(orow, o[rows], atol=1e-14, rtol=0)
    np.testing.assert_allclose(lserow, lse[rows], atol=1e-14, rtol=0)
    dq, dk, dv = attention_backward_head(q, k, v, do, 0.3, causal=True)
    dk_sum, dv_sum = np.zeros_like(dk), np.zeros_like(dv)
    for block in (np.arange(0, 9), np.arange(9, 20)):
        dq_r, dk_r, dv_r = attention_backward_rows(q, k, v, do, block, 0.3, causal=True)
        np.testing.assert_allclose(dq_r, dq[block], atol=1e-14, rtol=0)
        dk_sum += dk_r
        dv_sum += dv_r
    np.testing.assert_allclose(dk_sum, dk, atol=1e-13, rtol=0)
    np.testing.assert_allclose(dv_sum, dv, atol=1e-13, rtol=0)


def test_finite_difference_gradients_fewer_queries():
    """Central differences for 3 causal queries over 6 keys (h = 1e-6)."""
    rng = _rng(45)
    n_q, n_k, d, scale = 3, 6, 4, 0.7
    q, do = rng.normal(size=(n_q, d)), rng.normal(size=(n_q, d))
    k, v = rng.normal(size=(n_k, d)), rng.normal(size=(n_k, d))
    grads = attention_backward_head(q, k, v, do, scale, causal=True)
    h = 1e-6
    for which, g in zip(range(3), grads):
        fd = np.zeros(g.shape)
        for i in range(g.shape[0]):
            for t in range(d):
                args = [q.copy(), k.copy(), v.copy()]
                args[which][i, t] += h
                up = _loss(*args, do, scale, True)
                args[which][i, t] -= 2 * h
                dn = _loss(*args, do, scale, True)
                fd[i, t] = (up - dn) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert err <= 1e-6, (which, err)


def test_merge_partials_over_key_ranges_equals_full():
    """2.Online Softmax §七: attention over disjoint key sets, merged, is attention
    over all the keys (contiguous ranges and an interleaved partition)."""
    rng = _rng(46)
    q, k, v = rng.normal(size=(9, 6)) * 3, rng.normal(size=(31, 6)) * 3, rng.normal(size=(31, 5))
    o, lse = attention_forward_head(q, k, v, 0.5)
    for parts in ([np.arange(0, 10), np.arange(10, 11), np.arange(11, 31)],
                  [np.arange(0, 31, 3), np.arange(1, 31, 3), np.arange(2, 31, 3)]):
        outs = [attention_forward_head(q, k[p], v[p], 0.5) for p in parts]
        om, lsem = merge_partials([x[0] for x in outs], [x[1] for x in outs])
        np.testing.assert_allclose(om, o, atol=1e-13, rtol=0)
        np.testing.assert_allclose(lsem, lse, atol=1e-13, rtol=0)


def test_merge_partials_streaming_prefix_then_new_keys():
    """Prefix caching: new causal queries over cached keys (every cached key
    visible) merged with the same queries over the new keys under the causal
    mask equal the causal problem over the whole sequence."""
    rng = _rng(47)
    n_cache, n_new, d = 25, 7, 8
    q = rng.normal(size=(n_new, d))
    k, v = rng.normal(size=(n_cache + n_new, d)), rng.normal(size=(n_cache + n_new, d))
    o, lse = attention_forward_head(q, k, v, 0.35, causal=True)
    o_a, lse_a = attention_forward_head(q, k[:n_cache], v[:n_cache], 0.35, causal=False)
    o_b, lse_b = attention_forward_head(q, k[n_cache:], v[n_cache:], 0.35, causal=True)
    om, lsem = merge_partials([o_a, o_b], [lse_a, lse_b])
    np.testing.assert_allclose(om, o, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lsem, lse, atol=1e-13, rtol=0)


def test_merge_partials_ignores_parts_that_saw_nothing():
    rng = _rng(48)
    o1, lse1 = rng.normal(size=(3, 4)), rng.normal(size=3)
    junk = rng.normal(size=(3, 4))
    lse_none = np.full(3, -np.inf)
    om, lsem = merge_partials([junk, o1, junk], [lse_none, lse1, lse_none])
    np.testing.assert_allclose(om, o1, atol=1e-15, rtol=0)
    np.testing.assert_allclose(lsem, lse1, atol=1e-15, rtol=0)
    om, lsem = merge_partials([junk, junk], [lse_none, lse_none])
    assert np.all(om == 0.0) and np.all(lsem == -np.inf)


def test_merge_partials_two_parts_closed_form():
    """Two parts with LSE a and b: weights e^a/(e^a+e^b) and e^b/(e^a+e^b),
    LSE = ln(e^a + e^b) — written out directly."""
    o_a, o_b = np.array([[1.0, -2.0]]), np.array([[3.0, 0.5]])
    a, b = 0.3, -1.1
    om, lsem = merge_partials([o_a, o_b], [np.array([a]), np.array([b])])
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(om, wa * o_a + (1 - wa) * o_b, atol=1e-15, rtol=0)
    assert abs(lsem[0] - math.log(math.exp(a) + math.exp(b))) <= 1e-15


# ---------------------------------------------------------------- batched wrappers over [B, H, N, d]
#
# "1.FlashAttention 整体结构" 一 states attention per head; a [B, H, N, d] call is
# that definition applied to every (batch, head) slice independently.  Each head
# below gets its own values, so a swapped b/h index, a slice written to the
# wrong head or an output slot left unfilled fails one of these.

_BATCH_SHAPE = (2, 3, 9, 4)   # B, H, N, d: six heads that differ


def _distinct_heads(seed):
    rng = _rng(seed)
    B, H, n, d = _BATCH_SHAPE
    q, k, v, do = (rng.normal(size=_BATCH_SHAPE) for _ in range(4))
    # scale every head differently so that no two heads can stand in for each other
    for b in range(B):
        for h in range(H):
            f = 1.0 + 0.25 * (H * b + h)
            q[b, h] *= f
            v[b, h] += 3.0 * (H * b + h)
            do[b, h] -= 2.0 * (H * b + h)
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
def test_batched_wrappers_equal_the_per_head_definition(causal):
    """Every [b, h] slice of the batched result is the per-head result of that slice, bit for bit."""
    q, k, v, do = _distinct_heads(40)
    scale = _BATCH_SHAPE[3] ** -0.5
    o, lse = attention_forward(q, k, v, scale, causal)
    dq, dk, dv = attention_backward(q, k, v, do, scale, causal)
    assert o.shape == q.shape and lse.shape == q.shape[:3]
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    for b in range(_BATCH_SHAPE[0]):
        for h in range(_BATCH_SHAPE[1]):
            ro, rl = attention_forward_head(q[b, h], k[b, h], v[b, h], scale, causal)
            rdq, rdk, rdv = attention_backward_head(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
            assert np.array_equal(o[b, h], ro) and np.array_equal(lse[b, h], rl)
            assert np.array_equal(dq[b, h], rdq) and np.array_equal(dk[b, h], rdk) and np.array_equal(dv[b, h], rdv)


@pytest.mark.parametrize("causal", [False, True])
def test_batched_constant_v_per_head(causal):
    """V[b, h, j] = c_bh for every key gives O[b, h, i] = c_bh (rows of P sum to one),
    with a different constant vector in each head."""
    q, k, _, _ = _distinct_heads(41)
    B, H, n, d = _BATCH_SHAPE
    c = np.arange(B * H * d, dtype=np.float64).reshape(B, H, 1, d) * 0.37 - 5.0
    v = np.broadcast_to(c, (B, H, n, d)).copy()
    o, _ = attention_forward(q, k, v, d ** -0.5, causal)
    assert np.max(np.abs(o - c)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_batched_identical_keys_per_head(causal):
    """K[b, h, j] = k_bh for every key makes P uniform over the visible keys of that
    head: O is the (running, under the mask) mean of that head's V, LSE is
    scale·q·k_bh + ln(count), dQ = 0 (Σ_j dS_ij = 0 and every key is the same),
    and without the mask dV[b, h, j] = mean_i dO[b, h, i] for every key."""
    q, _, v, do = _distinct_heads(42)
    B, H, n, d = _BATCH_SHAPE
    rng = _rng(43)
    kvec = rng.normal(size=(B, H, 1, d))
    k = np.broadcast_to(kvec, (B, H, n, d)).copy()
    scale = d ** -0.5
    o, lse = attention_forward(q, k, v, scale, causal)
    dq, dk, dv = attention_backward(q, k, v, do, scale, causal)
    count = np.arange(1, n + 1) if causal else np.full(n, n)
    for b in range(B):
        for h in range(H):
            if causal:
                want = np.cumsum(v[b, h], axis=0) / count[:, None]
            else:
                want = np.tile(v[b, h].mean(axis=0), (n, 1))
            assert np.max(np.abs(o[b, h] - want)) <= 1e-12
            s = scale * (q[b, h] @ kvec[b, h, 0])
            np.testing.assert_allclose(lse[b, h], s + np.log(count), atol=1e-12, rtol=0)
            assert np.max(np.abs(dq[b, h])) <= 1e-12
            if not causal:
                np.testing.assert_allclose(dv[b, h], np.tile(do[b, h].mean(axis=0), (n, 1)), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_batched_gradient_invariants_per_head(causal):
    """Per head: Σ_j dV_j = Σ_i dO_i (rows of P sum to one) and Σ_j dK_j = 0; each
    head's dO is shifted differently, so dV's column sums identify the head."""
    q, k, v, do = _distinct_heads(44)
    B, H, n, d = _BATCH_SHAPE
    dq, dk, dv = attention_backward(q, k, v, do, d ** -0.5, causal)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(dv[b, h].sum(axis=0), do[b, h].sum(axis=0), atol=1e-10, rtol=0)
            assert np.max(np.abs(dk[b, h].sum(axis=0))) <= 1e-10
