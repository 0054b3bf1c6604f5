"""Pins of the oracle's diffusion module with its projections (Diffuser notes
sec 2.1: per-head Q, K, V projections, concatenation, output projection W_O)."""
import numpy as np

import oracle


def weights(D, H, d, seed):
    rng = np.random.default_rng(seed)
    s = 1.0 / np.sqrt(D)
    return (rng.standard_normal((H, D, d)) * s, rng.standard_normal((H, D, d)) * s,
            rng.standard_normal((H, D, d)) * s, rng.standard_normal((H * d, D)) / np.sqrt(H * d))


def test_single_head_identity_projections_is_the_module():
    n, d = 48, 16
    X = np.random.default_rng(1).standard_normal((2, n, d))
    row_ptr, col = oracle.token_graph(n, 3, 2, 4, seed=5)
    I = np.eye(d)
    got = oracle.layer_forward(X, I[None], I[None], I[None], I, row_ptr, col, 5, 0.1)
    want = oracle.forward(X[:, None], X[:, None], X[:, None], row_ptr, col, 5, 0.1)[:, 0]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)


def test_zero_query_key_projections_give_uniform_weights():
    # all scores 0: each row's weights are 1/|N(i)|; then Z_K = sum_k c_k A^k V with the
    # finite-K coefficients c_k = alpha (1-alpha)^k (k < K), (1-alpha)^K (notes sec 2.5)
    n, D, H, d, K, alpha = 40, 12, 2, 4, 4, 0.2
    X = np.random.default_rng(2).standard_normal((1, n, D))
    Wq, Wk, Wv, Wo = weights(D, H, d, 3)
    row_ptr, col = oracle.token_graph(n, 2, 1, 3, seed=7)
    got = oracle.layer_forward(X, 0 * Wq, 0 * Wk, Wv, Wo, row_ptr, col, K, alpha)
    A = np.zeros((n, n))
    for i in range(n):
        nb = col[row_ptr[i]:row_ptr[i + 1]]
        A[i, nb] = 1.0 / len(nb)
    M = sum(alpha * (1 - alpha) ** k * np.linalg.matrix_power(A, k) for k in range(K))
    M = M + (1 - alpha) ** K * np.linalg.matrix_power(A, K)
    heads = np.concatenate([M @ (X[0] @ Wv[h]) for h in range(H)], axis=1)
    np.testing.assert_allclose(got[0], heads @ Wo, rtol=1e-12, atol=1e-13)


def test_head_order_does_not_matter():
    # permuting the heads and the matching row blocks of W_O leaves the output unchanged
    n, D, H, d = 36, 16, 3, 8
    X = np.random.default_rng(4).standard_normal((2, n, D))
    Wq, Wk, Wv, Wo = weights(D, H, d, 5)
    row_ptr, col = oracle.token_graph(n, 3, 1, 2, seed=1)
    perm = [2, 0, 1]
    Wo_p = np.concatenate([Wo[h * d:(h + 1) * d] for h in perm], axis=0)
    a = oracle.layer_forward(X, Wq, Wk, Wv, Wo, row_ptr, col, 3, 0.1)
    b = oracle.layer_forward(X, Wq[perm], Wk[perm], Wv[perm], Wo_p, row_ptr, col, 3, 0.1)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_linear_in_the_value_and_output_projections():
    n, D, H, d = 30, 8, 2, 4
    X = np.random.default_rng(6).standard_normal((1, n, D))
    Wq, Wk, Wv, Wo = weights(D, H, d, 7)
    row_ptr, col = oracle.token_graph(n, 2, 1, 2, seed=3)
    base = oracle.layer_forward(X, Wq, Wk, Wv, Wo, row_ptr, col, 5, 0.1)
    np.testing.assert_allclose(oracle.layer_forward(X, Wq, Wk, 2 * Wv, Wo, row_ptr, col, 5, 0.1),
                               2 * base, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(oracle.layer_forward(X, Wq, Wk, Wv, -3 * Wo, row_ptr, col, 5, 0.1),
                               -3 * base, rtol=1e-13, atol=1e-14)


def test_round_bf16_matches_torch_and_ties_to_even():
    import torch
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-6, 6, 10000),
                        [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(2.0 + 2 ** -7), 0.0, 2 ** -100]])
    want = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), want)
    # ties go to the even neighbour
    assert oracle.round_bf16(np.array([1.0 + 2 ** -8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1.0 + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6


def test_bf16_interfaces_with_no_hops_are_two_rounded_products():
    # hops = 0: Z = V, so the module is round(round(round(X W_V) concatenated) W_O)
    n, D, H, d = 20, 16, 2, 8
    rng = np.random.default_rng(6)
    X = rng.standard_normal((2, n, D))
    Wq, Wk, Wv, Wo = weights(D, H, d, 7)
    row_ptr, col = oracle.token_graph(n, 2, 1, 2, seed=1)
    got = oracle.layer_forward(X, Wq, Wk, Wv, Wo, row_ptr, col, 0, 0.1, bf16_interfaces=True)
    import torch
    def rb(t):
        return torch.tensor(t, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    V = rb(np.stack([X @ Wv[h] for h in range(H)], axis=1))          # [B][H][n][d]
    heads = np.concatenate([V[:, h] for h in range(H)], axis=-1)
    np.testing.assert_array_equal(got, rb(heads @ Wo))
