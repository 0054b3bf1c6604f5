"""Pins of the oracle's backward pass (dQ, dK, dV of <dOut, Z_K>).

The Diffuser notes (sec 2.6) train through the same unrolled K-hop recursion,
so the gradient is the exact derivative of the forward.  The oracle's
backward is pinned to things other than its own chain-rule code: central
finite differences of the oracle's forward, the exact linear map from V to
Z_K given by the finite-K expansion (sec 2.5) with dense matrix powers, the
softmax's shift invariance, the special cases K = 0 and alpha = 1, and the
causal graph's lower-triangular structure (sec 2.6).
"""
import numpy as np
import pytest

import oracle
from tests import golden

PINS = golden.pins()


def qkv_g(n, d, seed, units=1):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((units, n, d)) for _ in range(4))


def loss(Q, K, V, W, row_ptr, col, hops, alpha):
    return float((oracle.forward(Q, K, V, row_ptr, col, hops, alpha) * W).sum())


def dense(A, row_ptr, col, n):
    M = np.zeros((n, n))
    for i in range(n):
        M[i, col[row_ptr[i]:row_ptr[i + 1]]] = A[row_ptr[i]:row_ptr[i + 1]]
    return M


@pytest.mark.parametrize("causal", [False, True], ids=["bidirectional", "causal"])
@pytest.mark.parametrize("hops,alpha", [(1, 0.0), (3, 0.2), (5, 0.1)])
def test_backward_matches_central_differences(hops, alpha, causal):
    # d L / d x for L = <W, Z_K>, x a sampled entry of Q, K or V:
    # (L(x + h) - L(x - h)) / 2h has error O(h^2) ~ 1e-10 relative at h = 1e-5
    n, d = 40, 8
    row_ptr, col = oracle.token_graph(n, 2, 2, 3, seed=5, globals_idx=[3, 30], causal=causal)
    Q, K, V, W = qkv_g(n, d, 17 + hops)
    dQ, dK, dV = oracle.backward(Q, K, V, W, row_ptr, col, hops, alpha)
    rng = np.random.default_rng(hops)
    h = 1e-5
    for X, dX in ((Q, dQ), (K, dK), (V, dV)):
        for _ in range(12):
            i, c = int(rng.integers(n)), int(rng.integers(d))
            keep = X[0, i, c]
            X[0, i, c] = keep + h
            lp = loss(Q, K, V, W, row_ptr, col, hops, alpha)
            X[0, i, c] = keep - h
            lm = loss(Q, K, V, W, row_ptr, col, hops, alpha)
            X[0, i, c] = keep
            fd = (lp - lm) / (2 * h)
            assert abs(fd - dX[0, i, c]) <= 1e-7 * max(1.0, abs(fd)), (i, c, fd, dX[0, i, c])


def test_dv_is_the_transposed_finite_k_map():
    # [D] sec 2.5: Z_5 = M V with M = sum_k c_k A^k (c = 0.1, 0.09, ..., 0.59049 for
    # alpha = 0.1), so dV = M^T dOut exactly, whatever the weights
    c = PINS["finiteK5_alpha01_coeffs"]
    n, d = 50, 6
    row_ptr, col = oracle.token_graph(n, 3, 2, 4, seed=2)
    Q, K, V, G = qkv_g(n, d, 3)
    A = oracle.attention_weights(Q[0], K[0], row_ptr, col)
    M = sum(ck * np.linalg.matrix_power(dense(A, row_ptr, col, n), k) for k, ck in enumerate(c))
    _, _, dV = oracle.backward(Q, K, V, G, row_ptr, col, 5, 0.1)
    np.testing.assert_allclose(dV[0], M.T @ G[0], rtol=1e-12, atol=1e-13)


def test_dk_sums_to_zero():
    # adding one vector to every key shifts each row's scores by a constant, which
    # the row softmax ignores: the gradient along that direction, sum_j dK_j, is 0
    n, d = 64, 8
    row_ptr, col = oracle.token_graph(n, 4, 3, 6, seed=9)
    Q, K, V, G = qkv_g(n, d, 4, units=2)
    dQ, dK, _ = oracle.backward(Q, K, V, G, row_ptr, col, 4, 0.15)
    scale = np.abs(dK).max()
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, atol=1e-12 * max(scale, 1.0) * n)
    assert np.abs(dQ).max() > 1e-3


def test_special_cases_have_no_weight_gradient():
    # K = 0 returns V, and alpha = 1 returns V at every hop: dV = dOut, dQ = dK = 0
    n, d = 30, 4
    row_ptr, col = oracle.token_graph(n, 2, 1, 3, seed=1)
    Q, K, V, G = qkv_g(n, d, 6)
    for hops, alpha in ((0, 0.1), (4, 1.0)):
        dQ, dK, dV = oracle.backward(Q, K, V, G, row_ptr, col, hops, alpha)
        np.testing.assert_array_equal(dV, G)
        np.testing.assert_array_equal(dQ, 0.0)
        np.testing.assert_array_equal(dK, 0.0)


def test_causal_gradient_never_reaches_the_future():
    # [D] sec 2.6: on the lower-triangular graph, output rows < p read no position
    # >= p, so a loss on those rows has exactly zero gradient at positions >= p
    n, d, p = 80, 8, 33
    row_ptr, col = oracle.token_graph(n, 5, 2, 6, seed=4, globals_idx=[10, 60], causal=True)
    Q, K, V, G = qkv_g(n, d, 8)
    G[:, p:] = 0.0
    dQ, dK, dV = oracle.backward(Q, K, V, G, row_ptr, col, 5, 0.1)
    for dX in (dQ, dK, dV):
        np.testing.assert_array_equal(dX[:, p:], 0.0)
        assert np.abs(dX[:, :p]).max() > 1e-4


def test_backward_units_are_independent():
    n, d = 32, 8
    row_ptr, col = oracle.token_graph(n, 3, 1, 2, seed=3)
    Q, K, V, G = qkv_g(n, d, 10, units=3)
    all3 = oracle.backward(Q, K, V, G, row_ptr, col, 3, 0.3)
    for u in range(3):
        one = oracle.backward(Q[u], K[u], V[u], G[u], row_ptr, col, 3, 0.3)
        for a, b in zip(all3, one):
            np.testing.assert_array_equal(a[u], b)
