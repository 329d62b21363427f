"""Pins for the oracle's backward (gradients of a loss with upstream gradient dH with respect
to Q, U and V).  They check against what the mathematics fixes, never against the
backward's own formula retyped:

  central finite differences of L = sum(dH * H) through the FORWARD oracle (a separate code
  path): every gradient entry, on shapes small enough to perturb each input once;
  dH with constant rows: L = sum_k c_k sum_i V_ik (S_t preserves column sums for any Q, U),
      so dQ = dU = 0 exactly and dV = dH;
  one anchor: A is all ones, H is the mean of V, so dQ = dU = 0 and dV_i = mean of dH;
  an anchor that no token reaches (its A column underflows) gets a zero dU row;
  L depends on Q and U only through S = scale Q U^T, so sum(Q dQ) = sum(U dU) (both equal
      sum(S dS)); softmax rows are invariant to shifting every anchor by one vector, so the
      anchors' dU rows sum to zero;
  dU of a head is the sum over the batch entries that share its anchors; linearity in dH.

Source: the anchors are fitted by gradient descent (pith.science verdict on arXiv 2505.16463,
"core_discovery"; the arXiv abstract, where the anchors are weights of a trainable layer).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(seed, B, heads, n, m, d, qscale=1.0):
    rng = np.random.default_rng(seed)
    Q = qscale * rng.standard_normal((B, heads, n, d))
    U = rng.standard_normal((heads, m, d))
    V = rng.standard_normal((B, heads, n, d))
    dH = rng.standard_normal((B, heads, n, d))
    return Q, U, V, dH


def _finite_differences(orc, Q, U, V, dH, scale, eps=1e-6):
    def loss(q, u, v):
        return float((orc.forward(q, u, v, scale) * dH).sum())

    out = []
    for which in range(3):
        X = (Q, U, V)[which]
        G = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args = [Q, U, V]
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args[which] = Xp
            lp = loss(*args)
            args[which] = Xm
            lm = loss(*args)
            G[idx] = (lp - lm) / (2 * eps)
        out.append(G)
    return out


@pytest.mark.parametrize("shape,scale,qscale", [((1, 1, 5, 3, 4), 0.5, 1.0), ((2, 2, 4, 2, 3), 1.0, 1.0),
                                                ((1, 2, 6, 4, 2), 0.7, 3.0), ((2, 1, 3, 5, 2), 0.25, 1.0)])
def test_gradients_match_finite_differences(oracle_mod, shape, scale, qscale):
    Q, U, V, dH = _inputs(sum(shape), *shape, qscale=qscale)
    dQ, dU, dV = oracle_mod.backward(Q, U, V, dH, scale)
    nQ, nU, nV = _finite_differences(oracle_mod, Q, U, V, dH, scale)
    for name, g, num in (("dQ", dQ, nQ), ("dU", dU, nU), ("dV", dV, nV)):
        err = np.abs(g - num).max()
        assert err <= 1e-6 * max(1.0, np.abs(num).max()), f"{name}: max |analytic - finite difference| = {err:.3e}"


def test_constant_upstream_rows_leave_q_and_u_flat(oracle_mod):
    Q, U, V, _ = _inputs(3, 2, 3, 9, 5, 4)
    c = np.array([0.5, -1.25, 2.0, 0.75])
    dH = np.broadcast_to(c, Q.shape).copy()
    dQ, dU, dV = oracle_mod.backward(Q, U, V, dH, 0.6)
    assert np.abs(dQ).max() < 1e-12 and np.abs(dU).max() < 1e-12
    assert np.allclose(dV, dH, atol=1e-12, rtol=0)


def test_one_anchor(oracle_mod):
    Q, U, V, dH = _inputs(4, 2, 2, 7, 1, 3)
    dQ, dU, dV = oracle_mod.backward(Q, U, V, dH, 0.9)
    assert np.abs(dQ).max() < 1e-13 and np.abs(dU).max() < 1e-13
    assert np.allclose(dV, np.broadcast_to(dH.mean(axis=2, keepdims=True), dV.shape), atol=1e-13, rtol=0)


def test_unreached_anchor_has_zero_gradient(oracle_mod):
    Q, U, V, dH = _inputs(5, 1, 1, 6, 4, 3)
    Q[..., 0] = np.abs(Q[..., 0]) + 1.0
    U[0, 2] = [-3000.0, 0.0, 0.0]  # scores <= -3000 * scale: exp underflows to 0 for every token
    dQ, dU, dV = oracle_mod.backward(Q, U, V, dH, 0.5)
    assert np.all(dU[0, 2] == 0.0)
    assert np.isfinite(dQ).all() and np.isfinite(dV).all()


def test_q_and_u_gradients_balance(oracle_mod):
    """L depends on Q and U only through S = scale Q U^T: sum(Q dQ) = sum(S dS) = sum(U dU)."""
    Q, U, V, dH = _inputs(6, 3, 2, 11, 6, 5, qscale=2.0)
    dQ, dU, _ = oracle_mod.backward(Q, U, V, dH, 0.4)
    lhs, rhs = float((Q * dQ).sum()), float((U * dU).sum())
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs)), (lhs, rhs)


def test_anchor_gradients_sum_to_zero(oracle_mod):
    """Shifting every anchor of a head by one vector leaves each softmax row unchanged."""
    Q, U, V, dH = _inputs(7, 2, 3, 8, 5, 4)
    _, dU, _ = oracle_mod.backward(Q, U, V, dH, 0.8)
    assert np.abs(dU.sum(axis=1)).max() < 1e-12


def test_batch_entries_share_the_anchor_gradient(oracle_mod):
    Q, U, V, dH = _inputs(8, 3, 2, 6, 4, 3)
    dQ, dU, dV = oracle_mod.backward(Q, U, V, dH, 0.5)
    total = np.zeros_like(U)
    for b in range(3):
        for h in range(2):
            q, u, v = oracle_mod.slice_backward(Q[b, h], U[h], V[b, h], dH[b, h], 0.5)
            assert np.allclose(q, dQ[b, h], atol=1e-13, rtol=0) and np.allclose(v, dV[b, h], atol=1e-13, rtol=0)
            total[h] += u
    assert np.allclose(total, dU, atol=1e-12, rtol=0)


def test_linear_in_the_upstream_gradient(oracle_mod):
    Q, U, V, dH = _inputs(9, 1, 2, 7, 3, 4)
    dH2 = np.random.default_rng(10).standard_normal(dH.shape)
    g1 = oracle_mod.backward(Q, U, V, dH, 0.5)
    g2 = oracle_mod.backward(Q, U, V, dH2, 0.5)
    g12 = oracle_mod.backward(Q, U, V, 2.0 * dH - 3.0 * dH2, 0.5)
    for a, b, c in zip(g1, g2, g12):
        assert np.allclose(c, 2.0 * a - 3.0 * b, atol=1e-11, rtol=0)
