"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a worked
example the pages print, a closed form, an invariant of the mathematics, a
special case with a textbook answer, brute force on a tiny input, or central
finite differences for the backward pass.  The cases are chosen so that a
dropped scale, a wrong sign, a transposed operand, an off-by-one causal mask or
a missing rowsum term each fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from tests.golden_io import load

F = oracle.attention_forward
BWD = oracle.attention_backward


def rnd(T, Hq, Hkv, d, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((T, Hq, d)), r.standard_normal((T, Hkv, d)),
            r.standard_normal((T, Hkv, d)), r.standard_normal((T, Hq, d)))


# ---------------------------------------------------------------- worked examples

def test_online_softmax_two_blocks_example():
    """"Attention 算子优化…" section 三: [1,2] then [3,1] give l ~= 1.638."""
    g = load("online_softmax_two_blocks.txt")
    scores = g["scores_block1"] + g["scores_block2"]
    # scores as q.k with d = 1, scale = 1
    n = len(scores)
    q = np.ones((n, 1, 1))
    k = np.array(scores, float).reshape(n, 1, 1)
    v = np.zeros((n, 1, 1))
    _, lse = F(q, k, v, [0, n], 1.0, False)
    ell = math.exp(lse[0, 0] - g["page_m_final"])
    # the page sums terms already rounded to 3 decimals, so its figure is good
    # to one unit in the last printed digit (exact: 1.63855)
    assert abs(ell - g["page_l_new"]) <= 10.0 ** -g["page_digits"]
    assert ell == pytest.approx(g["exact_l_new"], rel=1e-14)
    # the page's intermediate numbers, recomputed by the recurrence it describes
    b1, b2 = g["scores_block1"], g["scores_block2"]
    m_old = max(b1)
    l_old = sum(math.exp(s - m_old) for s in b1)
    assert round(l_old, 3) == g["page_l_old"]
    m_new = max(m_old, max(b2))
    corr = math.exp(m_old - m_new)
    assert round(corr, 3) == g["page_correction"]
    l_new = corr * l_old + sum(math.exp(s - m_new) for s in b2)
    assert l_new == pytest.approx(ell, rel=1e-15, abs=1e-15)


def test_online_softmax_value_example():
    """"FlashAttention：从 Safe Softmax 到分块计算" section 3.3:
    [1,2] then [3], v = [10,20,30]: o = u / l with the page's closed forms."""
    g = load("online_softmax_value_example.txt")
    n = len(g["scores"])
    q = np.ones((n, 1, 1))
    k = np.array(g["scores"], float).reshape(n, 1, 1)
    v = np.array(g["values"], float).reshape(n, 1, 1)
    o, lse = F(q, k, v, [0, n], 1.0, False)
    # every row sees the same scores (non-causal, identical queries)
    assert o[0, 0, 0] == pytest.approx(g["merged_u"] / g["merged_l"], rel=1e-14)
    assert lse[0, 0] == pytest.approx(g["m_final"] + math.log(g["merged_l"]), rel=1e-14)
    # the merge of block states equals the one-pass state (page's identity)
    assert g["merged_l"] == pytest.approx(sum(math.exp(s - 3) for s in g["scores"]), rel=1e-15)
    assert g["merged_u"] == pytest.approx(
        sum(math.exp(s - 3) * x for s, x in zip(g["scores"], g["values"])), rel=1e-15)
    # a transposed or reversed value order would give another number
    assert o[0, 0, 0] == pytest.approx(25.752104, abs=1e-6)


def test_safe_softmax_example_probabilities():
    """Same page, section 2.1: [1,2,3] -> (e^-2, e^-1, 1) / sum; V = I reads P."""
    g = load("safe_softmax_example.txt")
    n = 3
    q = np.zeros((n, 1, 3)); q[:, 0, 0] = 1.0
    k = np.zeros((n, 1, 3)); k[:, 0, 0] = g["scores"]
    v = np.eye(3).reshape(3, 1, 3)
    o, _ = F(q, k, v, [0, n], 1.0, False)
    e = np.array(g["shifted_exp"])
    np.testing.assert_allclose(o[0, 0], e / e.sum(), rtol=1e-14)


# ---------------------------------------------------------------- hand N=4, d=2

def test_hand_zero_query_uniform():
    """Q = 0: every score is 0, P is uniform, O = column mean of V, LSE = ln 4."""
    q = np.zeros((4, 1, 2))
    k = np.array([[1, 2], [3, -1], [0, 5], [-2, 2]], float)[:, None, :]
    v = np.array([[1, 0], [2, 4], [3, 8], [6, -4]], float)[:, None, :]
    o, lse = F(q, k, v, [0, 4], 0.5, False)
    np.testing.assert_allclose(o[:, 0, :], np.tile([3.0, 2.0], (4, 1)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0], np.full(4, math.log(4)), rtol=1e-15)


def test_hand_equal_keys_uniform():
    """All K rows equal: scores equal along each row, same uniform result."""
    q = np.array([[1, 2], [0, 1], [-3, 1], [2, 2]], float)[:, None, :]
    k = np.tile([[2.0, -1.0]], (4, 1))[:, None, :]
    v = np.array([[1, 0], [2, 4], [3, 8], [6, -4]], float)[:, None, :]
    o, lse = F(q, k, v, [0, 4], 1.0, False)
    np.testing.assert_allclose(o[:, 0, :], np.tile([3.0, 2.0], (4, 1)), atol=1e-14)
    expect = [1 * 2 - 2 + math.log(4), -1 + math.log(4), -6 - 1 + math.log(4), 4 - 2 + math.log(4)]
    np.testing.assert_allclose(lse[0], expect, rtol=1e-14)


def test_hand_causal_zero_query_prefix_means():
    """Causal with Q = 0: O_i = mean(V[0..i]) and LSE_i = ln(i+1) (diagonal visible)."""
    q = np.zeros((4, 1, 2))
    k = np.array([[1, 2], [3, -1], [0, 5], [-2, 2]], float)[:, None, :]
    v = np.array([[1, 0], [2, 4], [3, 8], [6, -4]], float)[:, None, :]
    o, lse = F(q, k, v, [0, 4], 1.0, True)
    want = np.array([[1, 0], [1.5, 2], [2, 4], [3, 2]], float)
    np.testing.assert_allclose(o[:, 0, :], want, atol=1e-15)
    np.testing.assert_allclose(lse[0], [math.log(i + 1) for i in range(4)], rtol=1e-15, atol=1e-15)


def test_hand_exponential_weights():
    """q = [1,0], keys [j,0]: p_j = e^j / sum e^j; with V = [j, 1] O = (E[j], 1)."""
    q = np.tile([[1.0, 0.0]], (4, 1))[:, None, :]
    k = np.array([[j, 0] for j in range(4)], float)[:, None, :]
    v = np.array([[j, 1] for j in range(4)], float)[:, None, :]
    o, lse = F(q, k, v, [0, 4], 1.0, False)
    Z = sum(math.exp(j) for j in range(4))
    mean_j = sum(j * math.exp(j) for j in range(4)) / Z
    np.testing.assert_allclose(o[:, 0, 0], mean_j, rtol=1e-14)
    np.testing.assert_allclose(o[:, 0, 1], 1.0, rtol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(Z), rtol=1e-15)
    # causal: row i sees keys 0..i only
    o, lse = F(q, k, v, [0, 4], 1.0, True)
    for i in range(4):
        Zi = sum(math.exp(j) for j in range(i + 1))
        assert o[i, 0, 0] == pytest.approx(sum(j * math.exp(j) for j in range(i + 1)) / Zi, rel=1e-14)
        assert lse[0, i] == pytest.approx(math.log(Zi), rel=1e-14, abs=1e-15)


def test_scale_applies_to_scores():
    """scale multiplies the scores: scale = 2 on keys [j,0] gives weights e^(2j)."""
    q = np.tile([[1.0, 0.0]], (3, 1))[:, None, :]
    k = np.array([[j, 0] for j in range(3)], float)[:, None, :]
    v = np.array([[j, 1] for j in range(3)], float)[:, None, :]
    o, lse = F(q, k, v, [0, 3], 2.0, False)
    Z = sum(math.exp(2 * j) for j in range(3))
    assert o[0, 0, 0] == pytest.approx(sum(j * math.exp(2 * j) for j in range(3)) / Z, rel=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(Z), rel=1e-15)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    """With V = I (L = d) the output rows are the rows of P: >= 0, sum 1."""
    L = 16
    r = np.random.default_rng(1)
    q = r.standard_normal((L, 1, L)) * 3
    k = r.standard_normal((L, 1, L))
    v = np.eye(L).reshape(L, 1, L)
    o, _ = F(q, k, v, [0, L], 0.7, causal)
    P = o[:, 0, :]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-14)
    assert (P >= 0).all()
    if causal:
        assert np.all(np.triu(P, 1) == 0)
        assert np.all(np.diag(P) > 0)


def test_permuting_keys_and_values_together():
    q, k, v, _ = rnd(40, 2, 2, 8, 2)
    perm = np.random.default_rng(3).permutation(40)
    o1, l1 = F(q, k, v, [0, 40], 0.3, False)
    o2, l2 = F(q, k[perm], v[perm], [0, 40], 0.3, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13)
    # permuting only V changes the output (catches a mis-paired PV product)
    o3, _ = F(q, k, v[perm], [0, 40], 0.3, False)
    assert np.abs(o3 - o1).max() > 1e-3


def test_constant_values_reproduce_value():
    q, k, _, _ = rnd(33, 3, 1, 8, 4)
    vrow = np.linspace(-2, 3, 8)
    v = np.tile(vrow, (33, 1, 1))
    for causal in (False, True):
        o, _ = F(q, k, v, [0, 33], 0.35, causal)
        np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), rtol=1e-13, atol=1e-13)


def test_key_shift_invariance_and_lse_shift():
    """k_j -> k_j + c leaves O unchanged and moves LSE_i by scale * q_i . c."""
    q, k, v, _ = rnd(24, 2, 2, 8, 5)
    c = np.random.default_rng(6).standard_normal(8)
    scale = 0.4
    for causal in (False, True):
        o1, l1 = F(q, k, v, [0, 24], scale, causal)
        o2, l2 = F(q, k + c, v, [0, 24], scale, causal)
        np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-12)
        shift = scale * np.einsum("thd,d->ht", q, c)
        np.testing.assert_allclose(l2 - l1, shift, rtol=1e-10, atol=1e-11)


def test_last_causal_row_equals_full_row_and_first_row_is_v0():
    q, k, v, _ = rnd(20, 2, 2, 4, 7)
    oc, lc = F(q, k, v, [0, 20], 0.5, True)
    of, lf = F(q, k, v, [0, 20], 0.5, False)
    np.testing.assert_allclose(oc[-1], of[-1], rtol=1e-14)
    np.testing.assert_allclose(lc[:, -1], lf[:, -1], rtol=1e-14)
    np.testing.assert_allclose(oc[0], v[0], rtol=1e-14)
    np.testing.assert_allclose(lc[:, 0], 0.5 * np.einsum("hd,hd->h", q[0], k[0]), rtol=1e-13)
    assert np.abs(oc[:-1] - of[:-1]).max() > 1e-3


@pytest.mark.parametrize("case", ["wide", "same_query", "query_matches_keys"])
def test_stress_cases_stay_finite(case):
    """Wide score range, identical queries, a query equal to every key."""
    q, k, v, _ = rnd(64, 2, 2, 16, 8)
    if case == "wide":
        q = q * 100
    elif case == "same_query":
        q = np.broadcast_to(q[:1], q.shape).copy()
    else:
        k = np.broadcast_to(k[:1], k.shape).copy() * 30
        q = np.broadcast_to(k[:1], q.shape).copy()
    for causal in (False, True):
        o, lse = F(q, k, v, [0, 64], 0.25, causal)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        assert np.abs(o).max() <= np.abs(v).max() + 1e-12  # convex combination of V rows


# ---------------------------------------------------------------- structure

def test_gqa_equals_repeated_heads():
    q, k, v, do = rnd(30, 8, 2, 8, 9)
    rep = lambda x: np.repeat(x, 4, axis=1)  # consecutive grouping: kv = h // 4
    for causal in (False, True):
        o1, l1 = F(q, k, v, [0, 30], 0.3, causal)
        o2, l2 = F(q, rep(k), rep(v), [0, 30], 0.3, causal)
        np.testing.assert_allclose(o1, o2, rtol=1e-14)
        np.testing.assert_allclose(l1, l2, rtol=1e-14)
        dq1, dk1, dv1 = BWD(q, k, v, do, [0, 30], 0.3, causal)
        dq2, dk2, dv2 = BWD(q, rep(k), rep(v), do, [0, 30], 0.3, causal)
        np.testing.assert_allclose(dq1, dq2, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dk1, dk2.reshape(30, 2, 4, 8).sum(2), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv1, dv2.reshape(30, 2, 4, 8).sum(2), rtol=1e-12, atol=1e-13)


def test_varlen_equals_independent_sequences():
    lengths = [5, 1, 17, 9]
    cu = oracle.cu_from_lengths(lengths)
    q, k, v, do = rnd(int(cu[-1]), 4, 2, 8, 10)
    for causal in (False, True):
        o, lse = F(q, k, v, cu, 0.3, causal)
        dq, dk, dv = BWD(q, k, v, do, cu, 0.3, causal)
        for s in range(len(lengths)):
            a, b = cu[s], cu[s + 1]
            os_, ls_ = F(q[a:b], k[a:b], v[a:b], [0, b - a], 0.3, causal)
            np.testing.assert_allclose(o[a:b], os_, rtol=1e-14)
            np.testing.assert_allclose(lse[:, a:b], ls_, rtol=1e-14)
            g = BWD(q[a:b], k[a:b], v[a:b], do[a:b], [0, b - a], 0.3, causal)
            for x, y in zip((dq, dk, dv), g):
                np.testing.assert_allclose(x[a:b], y, rtol=1e-13, atol=1e-14)


def test_empty_sequence_and_single_token():
    cu = oracle.cu_from_lengths([0, 1, 0, 3])
    q, k, v, do = rnd(4, 2, 1, 4, 11)
    o, lse = F(q, k, v, cu, 0.5, True)
    np.testing.assert_allclose(o[0], np.repeat(v[0], 2, axis=0), rtol=1e-14)  # one key: O = v
    np.testing.assert_allclose(lse[:, 0], 0.5 * (q[0] @ k[0, 0]), rtol=1e-14)


def test_rows_function_matches_full():
    lengths = [37, 130, 64]
    cu = oracle.cu_from_lengths(lengths)
    q, k, v, _ = rnd(int(cu[-1]), 4, 2, 16, 12)
    o, lse = F(q, k, v, cu, 0.25, True)
    toks = np.array([0, 36, 37, 100, 166, 170, 230])
    heads = np.array([0, 3, 1, 2, 3, 0, 1])
    o_r, l_r = oracle.attention_forward_rows(q, k, v, cu, 0.25, True, toks, heads)
    np.testing.assert_allclose(o_r, o[toks, heads], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l_r, lse[heads, toks], rtol=1e-14)


# ---------------------------------------------------------------- backward

def _loss(q, k, v, do, cu, scale, causal):
    o, _ = F(q, k, v, cu, scale, causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (3, 1)])
def test_backward_matches_finite_differences(causal, heads):
    """Central differences (h = 1e-6, fp64) of L = sum(dO * O)."""
    Hq, Hkv = heads
    cu = oracle.cu_from_lengths([5, 3])
    q, k, v, do = rnd(8, Hq, Hkv, 3, 13)
    scale = 0.8
    grads = BWD(q, k, v, do, cu, scale, causal)
    h = 1e-6
    for which, g in zip(range(3), grads):
        args = [q, k, v]
        fd = np.zeros_like(args[which])
        it = np.nditer(args[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = (_loss(*plus, do, cu, scale, causal) - _loss(*minus, do, cu, scale, causal)) / (2 * h)
        err = np.linalg.norm(fd - g) / np.linalg.norm(g)
        assert err <= 1e-6, (which, err)


def test_backward_sum_identities():
    """rowsum(dP*P) = rowsum(dO*O); sum_j dS_ij = 0 so sum_j dK_j = 0 per
    (sequence, kv head)."""
    lengths = [50, 13]
    cu = oracle.cu_from_lengths(lengths)
    q, k, v, do = rnd(63, 4, 2, 8, 14)
    for causal in (False, True):
        o, _ = F(q, k, v, cu, 0.3, causal)
        dq, dk, dv, rs = BWD(q, k, v, do, cu, 0.3, causal, return_rowsum=True)
        np.testing.assert_allclose(rs, np.einsum("thd,thd->ht", do, o), rtol=1e-11, atol=1e-12)
        for s in range(2):
            a, b = cu[s], cu[s + 1]
            assert np.abs(dk[a:b].sum(axis=0)).max() < 1e-11 * max(1.0, np.abs(dk).max())


def test_backward_single_key_gradients_vanish():
    """One visible key: P = 1 exactly, so dS = 0 and dQ = dK = 0, dV = dO."""
    q, k, v, do = rnd(1, 2, 1, 4, 15)
    dq, dk, dv = BWD(q, k, v, do, [0, 1], 0.5, True)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    np.testing.assert_allclose(dv[0, 0], do[0].sum(axis=0), rtol=1e-15)


# ---------------------------------------------------------------- tile counts

@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 256, 300, 511, 513, 1000, 1706, 4096])
def test_tile_counts_closed_form_matches_brute_force(L):
    for causal in (False, True):
        assert oracle.tile_counts([L], causal)[0] == oracle.tile_counts_closed_form(L, causal)


def test_causal_skips_about_half_of_the_tiles():
    """"Attention 算子优化…" section 四: about half of the tiles are skipped."""
    full = oracle.tile_counts([4096], False)[0]
    causal = oracle.tile_counts([4096], True)[0]
    assert full == 32 * 32
    assert causal == 32 * 33 // 2
    assert 0.5 <= causal / full < 0.52


# ---------------------------------------------------------------- decode

DEC = oracle.attention_decode


def test_decode_value_example():
    """The section 3.3 example of "FlashAttention：从 Safe Softmax 到分块计算"
    as one decoding step: a query q = [1] against cached keys [1], [2], [3]
    (d = 1, scale = 1) with values 10, 20, 30."""
    g = load("online_softmax_value_example.txt")
    n = len(g["scores"])
    q = np.ones((1, 1, 1))
    k = np.array(g["scores"], float).reshape(n, 1, 1)
    v = np.array(g["values"], float).reshape(n, 1, 1)
    o, lse = DEC(q, k, v, [0, n], 1.0)
    assert o[0, 0, 0] == pytest.approx(g["merged_u"] / g["merged_l"], rel=1e-14)
    assert lse[0, 0] == pytest.approx(g["m_final"] + math.log(g["merged_l"]), rel=1e-14)


def test_decode_equals_last_causal_row():
    """A decoding step is the last row of causal attention over the sequence
    whose newest token carries the query."""
    lengths = [7, 1, 30, 12]
    cu = oracle.cu_from_lengths(lengths)
    q, k, v, _ = rnd(int(cu[-1]), 8, 2, 16, 20)
    o_full, l_full = F(q, k, v, cu, 0.3, True)
    last = cu[1:] - 1
    o, lse = DEC(q[last], k, v, cu, 0.3)
    np.testing.assert_allclose(o, o_full[last], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, l_full[:, last], rtol=1e-14)


def test_decode_zero_query_means_and_degenerate_caches():
    """q = 0: uniform weights, O = mean of the cached V rows, LSE = ln L; an
    empty cache gives O = 0, LSE = -inf; one cached key gives O = v_0."""
    lengths = [5, 0, 1, 9]
    cu = oracle.cu_from_lengths(lengths)
    _, k, v, _ = rnd(int(cu[-1]), 2, 2, 4, 21)
    q = np.zeros((4, 2, 4))
    o, lse = DEC(q, k, v, cu, 0.7)
    for b, L in enumerate(lengths):
        a = cu[b]
        if L == 0:
            assert (o[b] == 0).all() and np.isneginf(lse[:, b]).all()
        else:
            np.testing.assert_allclose(o[b], v[a:a + L].mean(axis=0), rtol=1e-14)
            np.testing.assert_allclose(lse[:, b], math.log(L), rtol=1e-14)
    q1 = np.random.default_rng(3).standard_normal((4, 2, 4))
    o1, l1 = DEC(q1, k, v, cu, 0.7)
    np.testing.assert_allclose(o1[2], v[cu[2]], rtol=1e-14)
    np.testing.assert_allclose(l1[:, 2], 0.7 * np.einsum("hd,hd->h", q1[2], k[cu[2]]), rtol=1e-13)


def test_decode_gqa_equals_repeated_heads():
    cu = oracle.cu_from_lengths([11, 6])
    _, k, v, _ = rnd(17, 8, 2, 8, 22)
    q = np.random.default_rng(4).standard_normal((2, 8, 8))
    rep = lambda x: np.repeat(x, 4, axis=1)
    o1, l1 = DEC(q, k, v, cu, 0.4)
    o2, l2 = DEC(q, rep(k), rep(v), cu, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


# ---------------------------------------------------------------- FP8 (E4M3) K/V cache

from oracle import quant as Q8  # noqa: E402


def test_e4m3_decoding_of_every_code_matches_torch():
    """All 256 codes against torch's float8_e4m3fn, a library implementation
    of the same format (NaN codes: 0x7F and 0xFF)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = Q8.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert (nan == np.isnan(got)).all() and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_rounding_matches_torch_and_round_trips():
    """Every grid point, every midpoint (ties go to the even code) and random
    float32 values within the range where torch does not overflow."""
    import torch
    grid = Q8.e4m3_decode(np.arange(256, dtype=np.uint8))
    grid = np.unique(grid[np.isfinite(grid)])
    mids = (grid[1:] + grid[:-1]) / 2
    rnd = np.random.default_rng(0).uniform(-464, 464, 20000)
    small = np.random.default_rng(1).uniform(-0.05, 0.05, 20000)
    x = np.concatenate([grid, mids, [464.0, -464.0], rnd, small]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(Q8.e4m3_round(x.astype(np.float64)), ref)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(Q8.e4m3_encode(Q8.e4m3_decode(codes)), codes)


def test_e4m3_saturates_and_rounds_ties_to_even():
    assert Q8.e4m3_round(np.array([449.0, 470.0, 1e6, -500.0])).tolist() == [448.0, 448.0, 448.0, -448.0]
    # 1.0625 lies halfway between 1.0 (mantissa 0) and 1.125 (mantissa 1): to 1.0
    # 1.1875 lies halfway between 1.125 and 1.25 (mantissa 2): to 1.25
    assert Q8.e4m3_round(np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10])).tolist() == [
        1.0, 1.25, 0.0, 2.0 ** -8]


def test_row_quantisation_scale_rule_and_error_bound():
    r = np.random.default_rng(2)
    x = r.standard_normal((40, 3, 64)).astype(np.float32)
    x[5, 1] = 0.0  # an all-zero row
    x[7, 2] *= 1e-3
    codes, s = Q8.quantize_rows_fp8(x)
    assert codes.dtype == np.uint8 and s.dtype == np.float32 and s.shape == (40, 3)
    deq = Q8.dequantize_rows_fp8(codes, s)
    amax = np.abs(x).max(axis=-1)
    live = amax > 0
    np.testing.assert_array_equal(s[live], (amax[live] / np.float32(448)).astype(np.float32))
    assert s[5, 1] == 1.0 and (codes[5, 1] == 0).all()
    # the row's largest element lands on +-448 (to float32 rounding of x / s)
    top = np.take_along_axis(np.abs(deq), np.abs(x).argmax(-1)[..., None], -1)[..., 0]
    np.testing.assert_allclose(top[live], amax[live], rtol=2e-7)
    # half a quantum: 2^-4 relative in the normal range, 2^-10 s below it
    err = np.abs(deq - x)
    assert (err <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s[..., None] * (1 + 1e-6)).all()


# ---------------------------------------------------------------- paged K/V cache

def _paged_case(lengths, page, Hkv=2, d=8, seed=30, shuffle=True):
    """A packed cache cut into pages, placed at random physical pages of a
    pool that also holds garbage pages; returns (packed k, v, cu, pages, table)."""
    r = np.random.default_rng(seed)
    cu = oracle.cu_from_lengths(lengths)
    T = int(cu[-1])
    k = r.standard_normal((T, Hkv, d))
    v = r.standard_normal((T, Hkv, d))
    npg = [(L + page - 1) // page for L in lengths]
    total = sum(npg) + 5
    phys = r.permutation(total) if shuffle else np.arange(total)
    kp = r.standard_normal((total, page, Hkv, d)) * 100  # garbage everywhere first
    vp = r.standard_normal((total, page, Hkv, d)) * 100
    table = np.full((len(lengths), max(npg + [1]) + 2), -7, dtype=np.int64)  # unused entries: junk
    nxt = 0
    for b, L in enumerate(lengths):
        for j in range(npg[b]):
            pg = phys[nxt]
            nxt += 1
            table[b, j] = pg
            a, e = cu[b] + j * page, min(cu[b] + (j + 1) * page, cu[b + 1])
            kp[pg, :e - a] = k[a:e]
            vp[pg, :e - a] = v[a:e]
    return k, v, cu, kp, vp, table


@pytest.mark.parametrize("page", [1, 4, 16])
def test_paged_decode_equals_packed_decode(page):
    """Any page size, any placement of the pages in the pool and junk in the
    unused table entries and page tails give the packed cache's result."""
    lengths = [37, 0, 16, 5, 64]
    k, v, cu, kp, vp, table = _paged_case(lengths, page)
    q = np.random.default_rng(31).standard_normal((5, 4, 8))
    o_ref, l_ref = DEC(q, k, v, cu, 0.35)
    o, l = oracle.attention_decode_paged(q, kp, vp, table, lengths, 0.35)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(l, l_ref)


def test_paged_decode_reads_the_right_pages():
    """Attention over a cache is invariant under permuting its keys, so a
    swap of two full pages changes nothing; swapping the partly filled last
    page with a full one makes the gather read other rows (garbage past the
    cache) and changes that sequence's result, and only that one."""
    lengths = [44, 40]  # page 8: sequence 0 has 6 pages, the last with 4 rows
    k, v, cu, kp, vp, table = _paged_case(lengths, 8, seed=32)
    q = np.random.default_rng(33).standard_normal((2, 2, 8))
    o1, _ = oracle.attention_decode_paged(q, kp, vp, table, lengths, 0.5)
    t_full = table.copy()
    t_full[0, [0, 3]] = t_full[0, [3, 0]]
    o2, _ = oracle.attention_decode_paged(q, kp, vp, t_full, lengths, 0.5)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    t_tail = table.copy()
    t_tail[0, [0, 5]] = t_tail[0, [5, 0]]
    o3, _ = oracle.attention_decode_paged(q, kp, vp, t_tail, lengths, 0.5)
    assert np.abs(o1[0] - o3[0]).max() > 1e-3
    np.testing.assert_array_equal(o1[1], o3[1])


# ---------------------------------------------------------------- paged prefill

def _prefill_pages(seq_kv, page, Hkv, d, seed):
    """Lays per-sequence K/V arrays (list of [Lk, Hkv, d]) out as a shuffled
    page pool with garbage in every unused row and junk table entries."""
    r = np.random.default_rng(seed)
    npg = [(len(kv) + page - 1) // page for kv in seq_kv]
    total = sum(npg) + 3
    phys = r.permutation(total)
    pool = r.standard_normal((total, page, Hkv, d)) * 50
    table = np.full((len(seq_kv), max(npg + [1]) + 1), -3, dtype=np.int64)
    nxt = 0
    for b, kv in enumerate(seq_kv):
        for j in range(npg[b]):
            pg = phys[nxt]
            nxt += 1
            table[b, j] = pg
            rows = kv[j * page:(j + 1) * page]
            pool[pg, :len(rows)] = rows
    return pool, table


def _prefill_case(Lk, Lq, Hq=4, Hkv=2, d=8, page=4, seed=50):
    """Full per-sequence q, k, v (all Lk tokens) and the paged inputs of the
    chunk made of each sequence's last Lq tokens."""
    r = np.random.default_rng(seed)
    qs = [r.standard_normal((L, Hq, d)) for L in Lk]
    ks = [r.standard_normal((L, Hkv, d)) for L in Lk]
    vs = [r.standard_normal((L, Hkv, d)) for L in Lk]
    kp, table = _prefill_pages(ks, page, Hkv, d, seed + 1)
    # the value pool uses the same pages as the key pool
    vp = np.random.default_rng(seed + 2).standard_normal(kp.shape) * 50
    for b, vv in enumerate(vs):
        for j in range((len(vv) + page - 1) // page):
            rows = vv[j * page:(j + 1) * page]
            vp[table[b, j], :len(rows)] = rows
    q_chunk = np.concatenate([q[len(q) - lq:] for q, lq in zip(qs, Lq)], axis=0)
    return qs, ks, vs, kp, vp, table, q_chunk, oracle.cu_from_lengths(Lq)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("page", [1, 4, 16])
def test_paged_prefill_without_prefix_equals_packed_forward(causal, page):
    """Lk = Lq: the paged prefill is the packed forward over the same keys."""
    L = [37, 0, 16, 5, 64]
    qs, ks, vs, kp, vp, table, qc, cu = _prefill_case(L, L, page=page, seed=51)
    o, l = oracle.attention_forward_paged(qc, kp, vp, table, cu, L, 0.3, causal)
    k = np.concatenate(ks, axis=0)
    v = np.concatenate(vs, axis=0)
    o_ref, l_ref = F(qc, k, v, cu, 0.3, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, l_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("Lq", [[1, 5, 3], [7, 12, 30], [40, 17, 9]])
def test_paged_prefill_with_cached_prefix_equals_rows_of_full_causal(Lq):
    """Chunked prefill: the chunk of the newest Lq tokens, with the first
    Lk - Lq tokens already in the cache, gives exactly the last Lq rows of
    causal attention over the whole sequence (which pins the mask alignment:
    a mask aligned at the first token would differ)."""
    Lk = [40, 17, 30]
    qs, ks, vs, kp, vp, table, qc, cu = _prefill_case(Lk, Lq, seed=52)
    o, l = oracle.attention_forward_paged(qc, kp, vp, table, cu, Lk, 0.4, True)
    for b in range(len(Lk)):
        o_full, l_full = F(qs[b], ks[b], vs[b], [0, Lk[b]], 0.4, True)
        a, e = int(cu[b]), int(cu[b + 1])
        np.testing.assert_allclose(o[a:e], o_full[Lk[b] - Lq[b]:], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l[:, a:e], l_full[:, Lk[b] - Lq[b]:], rtol=1e-12, atol=1e-13)
    # top-left alignment (query i sees keys j <= i) is a different result
    if any(lq < lk for lq, lk in zip(Lq, Lk)):
        wrong, _ = F(qc, np.concatenate([k[:lq] for k, lq in zip(ks, Lq)], axis=0),
                       np.concatenate([v[:lq] for v, lq in zip(vs, Lq)], axis=0), cu, 0.4, True)
        assert np.abs(wrong - o).max() > 1e-3


def test_paged_prefill_single_query_equals_paged_decode():
    """Lq = 1 at the end of the cache is one decoding step (every key visible),
    with or without the mask."""
    Lk = [9, 33, 1]
    qs, ks, vs, kp, vp, table, qc, cu = _prefill_case(Lk, [1, 1, 1], seed=53)
    for causal in (False, True):
        o, l = oracle.attention_forward_paged(qc, kp, vp, table, cu, Lk, 0.5, causal)
        o_ref, l_ref = oracle.attention_decode_paged(qc.reshape(3, 4, 8), kp, vp, table, Lk, 0.5)
        np.testing.assert_allclose(o, o_ref.reshape(3, 4, 8), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, l_ref, rtol=1e-12, atol=1e-13)


def test_paged_prefill_non_causal_rows_are_decode_steps():
    """Without the mask each query row sees the whole cache: row i equals a
    decoding step of that query over the sequence's Lk keys."""
    Lk, Lq = [23, 8], [5, 8]
    qs, ks, vs, kp, vp, table, qc, cu = _prefill_case(Lk, Lq, seed=54)
    o, l = oracle.attention_forward_paged(qc, kp, vp, table, cu, Lk, 0.3, False)
    for b in range(2):
        a, e = int(cu[b]), int(cu[b + 1])
        cache_cu = oracle.cu_from_lengths([Lk[b]] * (e - a))
        kk = np.concatenate([ks[b]] * (e - a), axis=0)
        vv = np.concatenate([vs[b]] * (e - a), axis=0)
        o_ref, l_ref = DEC(qc[a:e], kk, vv, cache_cu, 0.3)
        np.testing.assert_allclose(o[a:e], o_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l[:, a:e], l_ref, rtol=1e-12, atol=1e-13)


def test_paged_prefill_rows_without_visible_keys_and_page_swaps():
    """Causal with fewer cached keys than queries: the first Lq - Lk rows see
    no key (O = 0, LSE = -inf).  Swapping the partly filled last page with a
    full one changes that sequence's result and no other."""
    Lk, Lq = [3, 12], [6, 12]
    qs, ks, vs, kp, vp, table, qc, cu = _prefill_case(Lk, [3, 12], seed=55)
    q6 = np.concatenate([np.random.default_rng(56).standard_normal((3, 4, 8)), qc], axis=0)
    cu6 = oracle.cu_from_lengths(Lq)
    o, l = oracle.attention_forward_paged(q6, kp, vp, table, cu6, Lk, 0.3, True)
    assert np.all(o[:3] == 0.0) and np.all(np.isneginf(l[:, :3]))
    assert np.all(np.isfinite(l[:, 3:]))
    t2 = table.copy()
    t2[1, [0, 2]] = t2[1, [2, 0]]  # sequence 1: 12 rows in pages of 4, all full
    o2, _ = oracle.attention_forward_paged(q6, kp, vp, t2, cu6, Lk, 0.3, True)
    np.testing.assert_array_equal(o2[:6], o[:6])
    assert np.abs(o2[6:] - o[6:]).max() > 1e-3  # causal: key order matters
    o3, _ = oracle.attention_forward_paged(q6, kp, vp, t2, cu6, Lk, 0.3, False)
    o4, _ = oracle.attention_forward_paged(q6, kp, vp, table, cu6, Lk, 0.3, False)
    np.testing.assert_allclose(o3[6:], o4[6:], rtol=1e-12, atol=1e-13)  # no mask: a key set
