"""Pins for the oracle's full softmax attention and relative Frobenius error, used by the
approximation-error diagnostic (how far anchor attention is from full attention when the
anchors are rows of the keys: the skeptic's concrete test in the pith.science verdict on
arXiv 2505.16463).  Checked against closed forms and invariants, not against the formula
retyped.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(seed, B, heads, n, d):
    r = np.random.default_rng(seed)
    return r.standard_normal((B, heads, n, d)), r.standard_normal((heads, n, d)), r.standard_normal((B, heads, n, d))


def test_closed_form(oracle_mod):
    """Keys (1, 0), V = (1, 0): query ln 3 weighs them 3/4 and 1/4 (H = 3/4); query 0 evenly (1/2)."""
    Q = np.array([[[[math.log(3.0)], [0.0]]]])
    K = np.array([[[1.0], [0.0]]])
    V = np.array([[[[1.0], [0.0]]]])
    H = oracle_mod.full_attention(Q, K, V, 1.0)
    assert abs(H[0, 0, 0, 0] - 0.75) < 1e-15 and abs(H[0, 0, 1, 0] - 0.5) < 1e-15


def test_constant_values_and_zero_scale(oracle_mod):
    Q, K, V = _rand(1, 2, 2, 9, 4)
    Vc = np.broadcast_to(V[:, :, :1, :], V.shape).copy()
    assert np.allclose(oracle_mod.full_attention(Q, K, Vc, 0.7), Vc, atol=1e-14, rtol=0)
    H0 = oracle_mod.full_attention(Q, K, V, 0.0)
    assert np.allclose(H0, np.broadcast_to(V.mean(axis=2, keepdims=True), V.shape), atol=1e-14, rtol=0)


def test_dominant_key_selects_its_value(oracle_mod):
    """Each head's keys are shared by the batch: with key 4 of head 0 and key 1 of head 1
    scoring far above the rest, every query of (b, 0) takes V[b, 0, 4] and of (b, 1) V[b, 1, 1]."""
    Q, K, V = _rand(2, 2, 2, 6, 3)
    Q[..., 0] = np.abs(Q[..., 0]) + 1.0
    K[0, 4] = [800.0, 0.0, 0.0]  # scores >= 800 * scale above every other key of the head
    K[1, 1] = [800.0, 0.0, 0.0]
    H = oracle_mod.full_attention(Q, K, V, 1.0)
    for b in range(2):
        assert np.allclose(H[b, 0], np.broadcast_to(V[b, 0, 4], H[b, 0].shape), atol=1e-12, rtol=0)
        assert np.allclose(H[b, 1], np.broadcast_to(V[b, 1, 1], H[b, 1].shape), atol=1e-12, rtol=0)


def test_permutations(oracle_mod):
    Q, K, V = _rand(3, 1, 2, 8, 5)
    H = oracle_mod.full_attention(Q, K, V, 0.5)
    p = np.random.default_rng(4).permutation(8)
    # the same permutation of keys and values leaves H unchanged, and of the queries permutes its rows
    Hk = oracle_mod.full_attention(Q, K[:, p], V[:, :, p], 0.5)
    assert np.allclose(Hk, H, atol=1e-12, rtol=0)
    Hq = oracle_mod.full_attention(Q[:, :, p], K, V, 0.5)
    assert np.allclose(Hq, H[:, :, p], atol=1e-12, rtol=0)


def test_identical_keys_agree_with_one_anchor(oracle_mod):
    """All keys equal: full attention averages V; so does anchor attention with one anchor."""
    Q, K, V = _rand(5, 2, 1, 7, 4)
    Kc = np.broadcast_to(K[:, :1, :], K.shape).copy()
    Hf = oracle_mod.full_attention(Q, Kc, V, 0.9)
    Ha = oracle_mod.forward(Q, K[:, :1, :], V, 0.9)
    assert np.allclose(Hf, Ha, atol=1e-14, rtol=0)


def test_relative_frobenius(oracle_mod):
    Q, K, V = _rand(6, 2, 3, 5, 4)
    H = oracle_mod.full_attention(Q, K, V, 0.5)
    assert np.all(oracle_mod.relative_frobenius(H, H) == 0.0)
    assert np.allclose(oracle_mod.relative_frobenius(H, np.zeros_like(H)), 1.0, atol=1e-15, rtol=0)
    assert np.allclose(oracle_mod.relative_frobenius(H, 2.0 * H), 1.0, atol=1e-15, rtol=0)
    assert np.allclose(oracle_mod.relative_frobenius(H, 1.25 * H), 0.25, atol=1e-15, rtol=0)
    assert oracle_mod.relative_frobenius(H, H).shape == (2, 3)
