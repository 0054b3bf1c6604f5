"""Pins of the oracle's graph variants beyond the three basic graphs:

* uniform-spaced extras ("w uni." of the Diffuser notes, sec 4.5, Tab S.7:
  the random edges' positions are taken at uniform spacing; the reading is
  j_t = (i + floor((2t + 1) n / (2R))) mod n, t < R);
* one graph per head (Diffuser notes sec 2.2: the random sets may differ per
  layer and per head).

Each is pinned by a hand-derived example or by a computation that shares no
step with the oracle's (Python sets, dense numpy matrices).
"""
import numpy as np
import pytest

import oracle


def brute_uniform_graph(n, r, G, R, causal):
    """Neighbour sets from the definition, as Python sets."""
    G = set(G)
    rows = []
    for i in range(n):
        if i in G:
            s = set(range(n))
        else:
            s = set(range(max(0, i - r), min(n, i + r + 1))) | G
            s |= {(i + ((2 * t + 1) * n) // (2 * R)) % n for t in range(R)}
        if causal:
            s = {j for j in s if j <= i}
        rows.append(sorted(s))
    return rows


def csr_rows(row_ptr, col):
    return [list(col[row_ptr[i]:row_ptr[i + 1]]) for i in range(len(row_ptr) - 1)]


def test_uniform_grid_worked_example():
    # n = 16, R = 4: the grid offsets are floor((2t + 1) 16 / 8) = 2, 6, 10, 14
    row_ptr, col = oracle.uniform_graph(16, 1, 0, 4)
    rows = csr_rows(row_ptr, col)
    assert rows[0] == [0, 1, 2, 6, 10, 14]
    assert rows[5] == [3, 4, 5, 6, 7, 11, 15]        # window 4..6, grid 7, 11, 15, 3
    assert rows[15] == [1, 5, 9, 13, 14, 15]         # window 14..15, grid 1, 5, 9, 13


@pytest.mark.parametrize("n,r,G,R,causal", [
    (16, 1, [], 4, False), (37, 3, [0, 5], 5, False), (100, 7, [3], 9, True),
    (257, 20, [0, 1, 2], 32, False), (64, 0, [], 1, True), (9, 30, [8], 3, False)])
def test_uniform_graph_brute_force(n, r, G, R, causal):
    row_ptr, col = oracle.uniform_graph(n, r, len(G), R, globals_idx=G or None, causal=causal)
    assert csr_rows(row_ptr, col) == brute_uniform_graph(n, r, G, R, causal)


@pytest.mark.parametrize("n,R", [(64, 4), (96, 8), (4096, 32)])
def test_uniform_extras_are_equally_spaced(n, R):
    # r = 0, no globals: row i is {i} plus R positions n/R apart, none of them i
    row_ptr, col = oracle.uniform_graph(n, 0, 0, R)
    step = n // R
    for i in (0, 1, n // 3, n - 1):
        row = col[row_ptr[i]:row_ptr[i + 1]]
        assert len(row) == R + 1 and i in row
        offs = sorted((int(j) - i) % n for j in row if j != i)
        assert np.all(np.diff(offs) == step) and offs[0] == step // 2


def test_causal_uniform_graph_is_the_lower_triangle():
    n, r, G, R = 200, 6, [0, 7], 16
    bp, bc = oracle.uniform_graph(n, r, len(G), R, globals_idx=G)
    cp, cc = oracle.uniform_graph(n, r, len(G), R, globals_idx=G, causal=True)
    assert csr_rows(cp, cc) == [[j for j in row if j <= i] for i, row in enumerate(csr_rows(bp, bc))]


def dense_head_forward(Q, K, V, row_ptr, col, hops, alpha):
    """One head from the definitions with dense matrices: masked row softmax of
    QK^T / sqrt(d), then Z <- (1 - alpha) A Z + alpha V, hops times."""
    n, d = Q.shape
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        mask[i, col[row_ptr[i]:row_ptr[i + 1]]] = True
    S = np.where(mask, Q @ K.T / np.sqrt(d), -np.inf)
    E = np.exp(S - S.max(axis=1, keepdims=True))
    A = E / E.sum(axis=1, keepdims=True)
    Z = V.copy()
    for _ in range(hops):
        Z = (1 - alpha) * (A @ Z) + alpha * V
    return Z


def per_head_inputs(B, H, n, d, seed):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((B, H, n, d)) for _ in range(3))


def test_per_head_forward_matches_dense_heads():
    B, H, n, d = 2, 3, 60, 8
    Q, K, V = per_head_inputs(B, H, n, d, 1)
    graphs = [oracle.token_graph(n, 4, 1, 3, seed=s << 16) for s in (11, 12, 13)]
    got = oracle.forward_per_head(Q, K, V, graphs, 4, 0.15)
    for b in range(B):
        for h in range(H):
            want = dense_head_forward(Q[b, h], K[b, h], V[b, h], *graphs[h], 4, 0.15)
            np.testing.assert_allclose(got[b, h], want, rtol=1e-12, atol=1e-13)


def test_per_head_forward_heads_are_independent():
    B, H, n, d = 1, 2, 50, 8
    Q, K, V = per_head_inputs(B, H, n, d, 2)
    # (seeds that differ only below R = 4 permute a row's own keys i R + t: same draws)
    g0, g1 = oracle.token_graph(n, 3, 1, 4, seed=1 << 20), oracle.token_graph(n, 3, 1, 4, seed=2 << 20)
    assert not np.array_equal(g0[1], g1[1])
    a = oracle.forward_per_head(Q, K, V, [g0, g1], 5, 0.1)
    b = oracle.forward_per_head(Q, K, V, [g0, g0], 5, 0.1)
    assert np.array_equal(a[:, 0], b[:, 0])            # head 0 sees only its own graph
    assert not np.allclose(a[:, 1], b[:, 1])           # head 1 does see its graph change
    shared = oracle.forward(Q, K, V, *g0, 5, 0.1)
    assert np.array_equal(b, shared)                   # one graph for all heads: the shared forward
