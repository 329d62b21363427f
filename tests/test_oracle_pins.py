"""Pins for the CPU oracle: checks against what the AnchorFormer construction and plain
mathematics fix, never against the oracle's own formula retyped.

Source of the definition: pith.science verdict on arXiv 2505.16463 ("core_discovery",
"key_machinery", the referee summary of Eq. 11/12 and the desk editor's note that
S_t = A Delta^{-1} A^T is row-stochastic, S_t 1 = 1).

Each pin is chosen so that a plausible slip in the oracle fails at least one:
  softmax over the wrong axis         -> closed forms, hard assignment, ratio property
  scale dropped or applied twice      -> closed form with scale 1/2, ratio property
  Delta from rows instead of columns  -> closed forms, Markov route, constant-V
  A^T V transposed / wrong index      -> reassociation, brute-force path sum
  U indexed per (batch, head)         -> layout pin
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- closed forms

def test_closed_form_two_tokens_two_anchors(oracle_mod):
    """Hand-derived case (exact rationals).

    n=2, m=2, d=1, scale=1, u_1=1, u_2=0, q_1=ln 3, q_2=0, V=(1, 0).
    Token 1 scores (ln 3, 0) -> A_1 = (3/4, 1/4); token 2 scores (0, 0) -> A_2 = (1/2, 1/2).
    Delta = (5/4, 3/4); A^T V = (3/4, 1/4); W' = (3/5, 1/3);
    H_1 = 3/4*3/5 + 1/4*1/3 = 8/15,  H_2 = 1/2*3/5 + 1/2*1/3 = 7/15.
    """
    Q = np.array([[[[math.log(3.0)], [0.0]]]])
    U = np.array([[[1.0], [0.0]]])
    V = np.array([[[[1.0], [0.0]]]])
    H = oracle_mod.forward(Q, U, V, 1.0)
    expect = [Fraction(8, 15), Fraction(7, 15)]
    for i in range(2):
        assert abs(H[0, 0, i, 0] - float(expect[i])) < 1e-15


def test_closed_form_scale_and_two_columns(oracle_mod):
    """Same A as above reached through scale=1/2 and d=2, with a second value column.

    u_1=(2,0), u_2=(0,2); q_1=(ln 3, 0) -> scaled scores (ln 3, 0); q_2=(1,1) -> (1, 1).
    V = [[1, 2], [0, -4]].  Column 0 as above.  Column 1: A^T V = (-1/2, -3/2),
    W' = (-2/5, -2), H = (3/4*(-2/5) + 1/4*(-2), 1/2*(-2/5) + 1/2*(-2)) = (-4/5, -6/5).
    """
    Q = np.array([[[[math.log(3.0), 0.0], [1.0, 1.0]]]])
    U = np.array([[[2.0, 0.0], [0.0, 2.0]]])
    V = np.array([[[[1.0, 2.0], [0.0, -4.0]]]])
    H = oracle_mod.forward(Q, U, V, 0.5)
    expect = np.array([[8 / 15, -4 / 5], [7 / 15, -6 / 5]])
    np.testing.assert_allclose(H[0, 0], expect, rtol=0, atol=2e-15)


def test_hard_assignment_gives_cluster_means(oracle_mod):
    """When every token's score for its own anchor exceeds the others by ~500, A is a
    0/1 assignment; S_t then averages V over the tokens sharing an anchor."""
    c = [0, 1, 0, 2, 1, 0, 2, 2, 0]
    n, m, d = len(c), 3, 4
    U = 10.0 * np.eye(m)
    U = np.concatenate([U, np.zeros((m, d - m))], axis=1)
    Q = np.zeros((n, d))
    for i, ci in enumerate(c):
        Q[i, ci] = 50.0
    rng = np.random.default_rng(1)
    V = _rand(rng, n, d)
    H = oracle_mod.forward(Q[None, None], U[None], V[None, None], 1.0)[0, 0]
    for i in range(n):
        members = [t for t in range(n) if c[t] == c[i]]
        np.testing.assert_allclose(H[i], V[members].mean(axis=0), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- A itself

def test_softmax_ratio_property(oracle_mod):
    """Defining property of a softmax over anchors: each row of A is positive, sums to one,
    and log A_ij - log A_ik = scale * q_i . (u_j - u_k)."""
    rng = np.random.default_rng(2)
    n, m, d, s = 13, 7, 5, 0.37
    Q, U, V = _rand(rng, n, d), _rand(rng, m, d), _rand(rng, n, d)
    A = oracle_mod.slice_forward(Q, U, V, s)["A"]
    assert (A > 0).all()
    np.testing.assert_allclose(A.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    for j in range(m):
        for k in range(m):
            lhs = np.log(A[:, j]) - np.log(A[:, k])
            rhs = s * (Q @ (U[j] - U[k]))
            np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- the product

def test_reassociation_matches_explicit_St(oracle_mod):
    """Eq. 11 == Eq. 12: forming the n x n S_t = A Delta^{-1} A^T and applying it to V gives
    the factored A (Delta^{-1} (A^T V))."""
    rng = np.random.default_rng(3)
    for n, m, d in [(1, 1, 1), (5, 3, 2), (40, 9, 6), (97, 16, 8)]:
        Q, U, V = _rand(rng, n, d), _rand(rng, m, d), _rand(rng, n, d)
        o = oracle_mod.slice_forward(Q, U, V, 1 / math.sqrt(d))
        A = o["A"]
        np.testing.assert_allclose(o["delta"], A.sum(axis=0), rtol=1e-14)
        np.testing.assert_allclose(o["W"], A.T @ V, rtol=1e-12, atol=1e-13)
        St = A @ np.diag(1.0 / A.sum(axis=0)) @ A.T
        np.testing.assert_allclose(o["H"], St @ V, rtol=1e-11, atol=1e-13)


def test_row_stochastic_constant_value_is_fixed(oracle_mod):
    """S_t 1 = 1: every row of S_t sums to one, so a V whose columns are constant comes back
    unchanged."""
    rng = np.random.default_rng(4)
    n, m, d = 31, 6, 4
    Q, U = _rand(rng, n, d), _rand(rng, m, d)
    cst = _rand(rng, d)
    V = np.tile(cst, (n, 1))
    o = oracle_mod.slice_forward(Q, U, V, 0.5)
    A = o["A"]
    St = A @ np.diag(1.0 / A.sum(axis=0)) @ A.T
    np.testing.assert_allclose(St.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o["H"], V, rtol=0, atol=1e-14)


@pytest.mark.parametrize("case", ["m1", "identical_anchors", "zero_queries"])
def test_degenerate_cases_give_the_mean(oracle_mod, case):
    """One anchor, all anchors equal, or Q = 0: every row of A is the same, S_t = 11^T / n,
    so every H_i is the mean of V's rows."""
    rng = np.random.default_rng(5)
    n, d = 23, 5
    m = 1 if case == "m1" else 6
    Q = np.zeros((n, d)) if case == "zero_queries" else _rand(rng, n, d)
    U = np.tile(_rand(rng, 1, d), (m, 1)) if case == "identical_anchors" else _rand(rng, m, d)
    V = _rand(rng, n, d)
    H = oracle_mod.slice_forward(Q, U, V, 0.7)["H"]
    np.testing.assert_allclose(H, np.tile(V.mean(axis=0), (n, 1)), rtol=0, atol=1e-14)


def test_brute_force_path_sum_eq8(oracle_mod):
    """Eq. 8 written out as a path sum over anchors, scalar by scalar:
    p(v_j | v_i) = sum_l p(v_j | u_l) p(u_l | v_i), with p(u_l | v_i) the softmax of
    token i over anchors and p(v_j | u_l) = A_jl / sum_t A_tl; H_i = sum_j p(v_j|v_i) V_j."""
    rnd = random.Random(6)
    for _ in range(25):
        n, m, d = rnd.randint(1, 8), rnd.randint(1, 4), rnd.randint(1, 3)
        s = rnd.uniform(0.1, 1.5)
        Q = [[rnd.gauss(0, 1) for _ in range(d)] for _ in range(n)]
        U = [[rnd.gauss(0, 1) for _ in range(d)] for _ in range(m)]
        V = [[rnd.gauss(0, 1) for _ in range(d)] for _ in range(n)]
        p_ul_vi = []
        for i in range(n):
            e = [math.exp(s * math.fsum(Q[i][k] * U[l][k] for k in range(d))) for l in range(m)]
            z = math.fsum(e)
            p_ul_vi.append([x / z for x in e])
        col = [math.fsum(p_ul_vi[t][l] for t in range(n)) for l in range(m)]
        H = oracle_mod.forward(np.array(Q)[None, None], np.array(U)[None], np.array(V)[None, None], s)[0, 0]
        for i in range(n):
            for k in range(d):
                terms = []
                for j in range(n):
                    pji = math.fsum(p_ul_vi[j][l] / col[l] * p_ul_vi[i][l] for l in range(m))
                    terms.append(pji * V[j][k])
                assert abs(H[i, k] - math.fsum(terms)) < 1e-13


def test_markov_route_F_squared(oracle_mod):
    """Bipartite token-anchor graph G = [[0, A], [A^T, 0]], D = diag(G 1), F = D^{-1} G:
    the token block of F^2 is S_t, and applying it to V gives H."""
    rng = np.random.default_rng(7)
    n, m, d = 17, 5, 3
    Q, U, V = _rand(rng, n, d), _rand(rng, m, d), _rand(rng, n, d)
    o = oracle_mod.slice_forward(Q, U, V, 0.8)
    A = o["A"]
    G = np.zeros((n + m, n + m))
    G[:n, n:] = A
    G[n:, :n] = A.T
    F = G / G.sum(axis=1, keepdims=True)
    F2 = F @ F
    np.testing.assert_allclose(F2[:n, :n] @ V, o["H"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(G.sum(axis=1)[n:], o["delta"], rtol=1e-14)


# ---------------------------------------------------------------- invariants

def test_invariants(oracle_mod):
    """Consequences of S_t being symmetric, doubly stochastic, non-negative and of rank <= m."""
    rng = np.random.default_rng(8)
    n, m, d, s = 29, 4, 6, 0.6
    Q, U, V = _rand(rng, n, d), _rand(rng, m, d), _rand(rng, n, d)
    H = lambda Qx, Ux, Vx: oracle_mod.slice_forward(Qx, Ux, Vx, s)["H"]
    h = H(Q, U, V)
    # column sums preserved (S_t^T 1 = 1)
    np.testing.assert_allclose(h.sum(axis=0), V.sum(axis=0), rtol=1e-12, atol=1e-12)
    # convex combinations of V's rows
    assert (h <= V.max(axis=0) + 1e-12).all() and (h >= V.min(axis=0) - 1e-12).all()
    # linear in V, shift-equivariant
    V2 = _rand(rng, n, d)
    np.testing.assert_allclose(H(Q, U, 2.5 * V - 0.5 * V2), 2.5 * h - 0.5 * H(Q, U, V2), atol=1e-12)
    c = _rand(rng, d)
    np.testing.assert_allclose(H(Q, U, V + c), h + c, atol=1e-12)
    # token permutation equivariance, anchor permutation invariance
    p = rng.permutation(n)
    np.testing.assert_allclose(H(Q[p], U, V[p]), h[p], atol=1e-12)
    np.testing.assert_allclose(H(Q, U[rng.permutation(m)], V), h, atol=1e-12)
    # S_t symmetric with rank <= m
    A = oracle_mod.slice_forward(Q, U, V, s)["A"]
    St = A @ np.diag(1.0 / A.sum(axis=0)) @ A.T
    np.testing.assert_allclose(St, St.T, atol=1e-15)
    assert np.linalg.matrix_rank(St, tol=1e-10) <= m


def test_zero_degree_anchor_drops_out(oracle_mod):
    """Reading for Delta_j = 0 (silent on the pages): an anchor no token reaches
    (every A_ij underflows to exactly 0) contributes nothing; H equals the forward without it."""
    Q = np.array([[1.0], [2.0], [3.0], [0.5]])
    V = np.array([[1.0, -1.0], [2.0, 0.0], [4.0, 3.0], [-2.0, 1.0]])
    U = np.array([[0.0], [-2000.0]])  # score <= -1000: exp underflows to 0 in double
    Qd = np.concatenate([Q, np.zeros((4, 1))], axis=1)
    Ud = np.concatenate([U, np.zeros((2, 1))], axis=1)
    o = oracle_mod.slice_forward(Qd, Ud, V, 1.0)
    assert o["delta"][1] == 0.0 and (o["Wp"][1] == 0).all()
    np.testing.assert_allclose(o["H"], np.tile(V.mean(axis=0), (4, 1)), atol=1e-15)


def test_layout_batch_heads_and_shared_anchors(oracle_mod):
    """[B][heads][n][d] layout with U [heads][m][d] shared by every batch entry."""
    rng = np.random.default_rng(9)
    B, heads, n, m, d = 2, 3, 11, 4, 5
    Q, V = _rand(rng, B, heads, n, d), _rand(rng, B, heads, n, d)
    U = _rand(rng, heads, m, d)
    Q[1], V[1] = Q[0], V[0]
    H = oracle_mod.forward(Q, U, V, 0.45)
    np.testing.assert_array_equal(H[1], H[0])
    for b in range(B):
        for h in range(heads):
            np.testing.assert_allclose(H[b, h], oracle_mod.slice_forward(Q[b, h], U[h], V[b, h], 0.45)["H"],
                                       rtol=0, atol=0)
    assert not np.allclose(H[0, 0], H[0, 1])


def test_scale_multiplies_scores(oracle_mod):
    rng = np.random.default_rng(10)
    n, m, d = 19, 5, 8
    Q, U, V = _rand(rng, 1, 1, n, d), _rand(rng, 1, m, d), _rand(rng, 1, 1, n, d)
    np.testing.assert_allclose(oracle_mod.forward(Q, U, V, 0.3), oracle_mod.forward(0.3 * Q, U, V, 1.0),
                               atol=1e-13)


def test_sampled_rows_route(oracle_mod):
    rng = np.random.default_rng(11)
    n, m, d = 50, 7, 4
    Q, U, V = _rand(rng, n, d), _rand(rng, m, d), _rand(rng, n, d)
    rows = [0, 3, 49, 17]
    np.testing.assert_array_equal(oracle_mod.slice_rows(Q, U, V, 0.5, rows),
                                  oracle_mod.slice_forward(Q, U, V, 0.5)["H"][rows])


def test_bad_arguments_raise(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.slice_rows(np.zeros((3, 2)), np.zeros((1, 2)), np.zeros((3, 2)), 1.0, [5])
    with pytest.raises(ValueError):
        oracle_mod.forward(np.zeros((1, 1, 3, 2)), np.zeros((1, 0, 2)), np.zeros((1, 1, 3, 2)), 1.0)
