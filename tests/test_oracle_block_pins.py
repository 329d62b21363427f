"""Pins for the oracle's block front end: in an AnchorFormer layer the anchor attention takes
the place of a ViT block's self-attention, so each head's queries and values are linear
projections of the token embeddings, Q = X Wq^T and V = X Wv^T, and the forward follows.
Checked against the forward (pinned on its own), closed forms and invariants, with the
projections formed here by indexing or by a library contraction, never by the oracle's loop.
"""
import math

import numpy as np
import pytest


def _rand(seed, B, heads, n, m, d, dm):
    r = np.random.default_rng(seed)
    X = r.standard_normal((B, n, dm))
    Wq = r.standard_normal((heads, d, dm)) / math.sqrt(dm)
    Wv = r.standard_normal((heads, d, dm)) / math.sqrt(dm)
    U = r.standard_normal((heads, m, d))
    return X, Wq, Wv, U


def test_signed_column_selection_is_the_forward(oracle_mod):
    """With each weight row a signed unit vector, Q[b, h, i, k] = s_hk X[b, i, p_h(k)]: a
    gather, so the block must equal the forward on the gathered Q and V."""
    B, heads, n, m, d, dm = 2, 3, 11, 5, 4, 12
    r = np.random.default_rng(7)
    X = r.standard_normal((B, n, dm))
    U = r.standard_normal((heads, m, d))
    Wq, Wv = np.zeros((heads, d, dm)), np.zeros((heads, d, dm))
    Q, V = np.empty((B, heads, n, d)), np.empty((B, heads, n, d))
    for h in range(heads):
        pq, pv = r.permutation(dm)[:d], r.permutation(dm)[:d]
        sq, sv = r.choice([-1.0, 1.0], d), r.choice([-1.0, 1.0], d)
        for k in range(d):
            Wq[h, k, pq[k]] = sq[k]
            Wv[h, k, pv[k]] = sv[k]
            Q[:, h, :, k] = sq[k] * X[:, :, pq[k]]
            V[:, h, :, k] = sv[k] * X[:, :, pv[k]]
    H = oracle_mod.block(X, Wq, Wv, U, 0.6)
    assert np.allclose(H, oracle_mod.forward(Q, U, V, 0.6), atol=1e-13, rtol=0)


def test_zero_query_projection_averages_the_values(oracle_mod):
    """Wq = 0: every score is 0, A is uniform, and each row of H is the token mean of V,
    i.e. (mean over tokens of X) Wv^T, summed here with fsum."""
    B, heads, n, m, d, dm = 2, 2, 6, 3, 3, 5
    X, _, Wv, U = _rand(3, B, heads, n, m, d, dm)
    H = oracle_mod.block(X, np.zeros_like(Wv), Wv, U, 0.8)
    for b in range(B):
        for h in range(heads):
            for k in range(d):
                want = math.fsum(X[b, i, c] * Wv[h, k, c] for i in range(n) for c in range(dm)) / n
                assert np.allclose(H[b, h, :, k], want, atol=1e-13, rtol=0)


def test_matches_a_library_projection(oracle_mod):
    X, Wq, Wv, U = _rand(4, 2, 3, 17, 6, 8, 24)
    Q = np.einsum("bic,hkc->bhik", X, Wq)
    V = np.einsum("bic,hkc->bhik", X, Wv)
    assert np.allclose(oracle_mod.block(X, Wq, Wv, U, 0.35), oracle_mod.forward(Q, U, V, 0.35), atol=1e-12, rtol=0)


def test_linear_in_the_value_projection(oracle_mod):
    X, Wq, Wv, U = _rand(5, 1, 2, 9, 4, 4, 10)
    Wv2 = np.random.default_rng(6).standard_normal(Wv.shape)
    H1 = oracle_mod.block(X, Wq, Wv, U, 0.5)
    H2 = oracle_mod.block(X, Wq, Wv2, U, 0.5)
    H = oracle_mod.block(X, Wq, 2.0 * Wv - 0.5 * Wv2, U, 0.5)
    assert np.allclose(H, 2.0 * H1 - 0.5 * H2, atol=1e-12, rtol=0)


def test_token_permutation_permutes_rows(oracle_mod):
    X, Wq, Wv, U = _rand(8, 2, 2, 10, 3, 4, 6)
    p = np.random.default_rng(9).permutation(10)
    H = oracle_mod.block(X, Wq, Wv, U, 0.7)
    Hp = oracle_mod.block(X[:, p], Wq, Wv, U, 0.7)
    assert np.allclose(Hp, H[:, :, p], atol=1e-12, rtol=0)


def test_batch_entries_share_the_weights(oracle_mod):
    """Batch entries with the same tokens give the same output; heads differ."""
    X, Wq, Wv, U = _rand(10, 3, 2, 8, 3, 4, 6)
    X[2] = X[0]
    H = oracle_mod.block(X, Wq, Wv, U, 0.9)
    assert np.array_equal(H[2], H[0])
    assert not np.allclose(H[0, 0], H[0, 1])


def test_slice_entry_matches_the_batched_one(oracle_mod):
    X, Wq, Wv, U = _rand(11, 2, 3, 7, 4, 4, 8)
    H = oracle_mod.block(X, Wq, Wv, U, 0.4)
    assert np.array_equal(oracle_mod.block_slice(X[1], Wq[2], Wv[2], U[2], 0.4), H[1, 2])


def test_bad_arguments_raise(oracle_mod):
    X, Wq, Wv, U = _rand(12, 1, 1, 4, 2, 2, 3)
    with pytest.raises(ValueError):
        oracle_mod.block(X, Wq, Wv, U[:, :0], 0.5)
