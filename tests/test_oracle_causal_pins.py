"""Pins for the oracle's masked (causal) variant of the anchor construction: token i's anchor
summaries include only tokens j <= i (one of the pith.science verdict's inferences on arXiv
2505.16463: A can be masked against later tokens).  Checked against what the
definition fixes, not against the prefix loop retyped:

  the last token sees every token: its row equals the unmasked forward's last row;
  the first token sees only itself: H[0] = V[0];
  no token draws on a later one: changing Q or V of later tokens leaves earlier rows alone;
  the masked S_t keeps rows summing to one: a constant V comes back unchanged;
  one anchor: A is all ones and H[i] is the mean of V[0..i];
  the explicit masked n x n S_t[i][j] = sum_l A[i][l] A[j][l] / Delta^(i)_l (j <= i) times V,
  built here from the forward oracle's A, equals the prefix evaluation.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(seed, B, heads, n, m, d, qscale=1.0):
    r = np.random.default_rng(seed)
    return qscale * r.standard_normal((B, heads, n, d)), r.standard_normal((heads, m, d)), r.standard_normal((B, heads, n, d))


def test_last_row_is_the_unmasked_forward(oracle_mod):
    Q, U, V = _rand(1, 2, 3, 11, 4, 5)
    Hc = oracle_mod.causal(Q, U, V, 0.6)
    Hf = oracle_mod.forward(Q, U, V, 0.6)
    assert np.allclose(Hc[:, :, -1], Hf[:, :, -1], atol=1e-13, rtol=0)
    assert not np.allclose(Hc[:, :, 3], Hf[:, :, 3], atol=1e-6, rtol=0)  # earlier rows do differ


def test_first_row_is_its_own_value(oracle_mod):
    Q, U, V = _rand(2, 2, 2, 6, 5, 3)
    Hc = oracle_mod.causal(Q, U, V, 0.8)
    assert np.allclose(Hc[:, :, 0], V[:, :, 0], atol=1e-14, rtol=0)


def test_causality(oracle_mod):
    Q, U, V = _rand(3, 1, 2, 9, 4, 4)
    Hc = oracle_mod.causal(Q, U, V, 0.5)
    Q2, V2 = Q.copy(), V.copy()
    Q2[:, :, 6:] += 3.0
    V2[:, :, 6:] -= 2.0
    Hc2 = oracle_mod.causal(Q2, U, V2, 0.5)
    assert np.array_equal(Hc[:, :, :6], Hc2[:, :, :6])
    assert not np.allclose(Hc[:, :, 6:], Hc2[:, :, 6:])


def test_constant_values_are_kept(oracle_mod):
    Q, U, V = _rand(4, 2, 2, 10, 6, 4)
    Vc = np.broadcast_to(V[:, :, :1, :], V.shape).copy()
    assert np.allclose(oracle_mod.causal(Q, U, Vc, 0.7), Vc, atol=1e-13, rtol=0)


def test_one_anchor_is_a_prefix_mean(oracle_mod):
    Q, U, V = _rand(5, 1, 2, 8, 1, 3)
    Hc = oracle_mod.causal(Q, U, V, 0.9)
    ref = np.cumsum(V, axis=2) / np.arange(1, 9)[None, None, :, None]
    assert np.allclose(Hc, ref, atol=1e-14, rtol=0)


def test_explicit_masked_matrix(oracle_mod):
    Q, U, V = _rand(6, 1, 1, 7, 3, 2, qscale=2.0)
    A = oracle_mod.slice_forward(Q[0, 0], U[0], V[0, 0], 0.5)["A"]
    n = A.shape[0]
    S = np.zeros((n, n))
    for i in range(n):
        dl = A[: i + 1].sum(axis=0)
        for j in range(i + 1):
            S[i, j] = float(np.sum(A[i] * A[j] / dl))
    assert np.allclose(S.sum(axis=1), 1.0, atol=1e-14, rtol=0)
    assert np.allclose(oracle_mod.causal(Q, U, V, 0.5)[0, 0], S @ V[0, 0], atol=1e-13, rtol=0)
