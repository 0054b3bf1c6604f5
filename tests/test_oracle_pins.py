"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Nothing here compares the oracle with itself: every expected value is a number
the pages print, a closed form, a textbook routine (dense softmax, a dense
linear solve, matrix powers) or a brute-force construction written a different
way (Python sets).  Page titles:
  [D] "Diffuser: modelling long sequences with multi-hop attention diffusion"
  [S] "1.2.1 Static sparsity: Longformer, BigBird and sliding windows"
"""
import math

import numpy as np
import pytest

import oracle
from sparse_long_sequence_gb300 import synthetic, workloads
from tests import golden

PINS = golden.pins()
MASK64 = (1 << 64) - 1


# ---------------------------------------------------------------- helpers
def sm64_py(x: int) -> int:
    """SplitMix64 output function, in Python integers (pinned below)."""
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def brute_token_graph(n, r, G, R, seed):
    """Neighbour sets as Python sets: [S] eq 5 window, eq 12 globals, random draws."""
    G = set(G)
    rows = []
    for i in range(n):
        if i in G:
            s = set(range(n))
        else:
            s = {j for j in range(max(0, i - r), min(n, i + r + 1))}
            s |= G
            s |= {sm64_py(seed ^ (i * R + t)) % n for t in range(R)}
        rows.append(sorted(s))
    return rows


def brute_causal_token_graph(n, r, G, R, seed):
    """Causal neighbour sets from the text: [S] sec 1.1 window of the r+1 history
    positions; [D] sec 2.6 every global and random edge obeys j <= i."""
    rows = []
    for i in range(n):
        if i in G:
            s = set(range(i + 1))
        else:
            s = set(range(max(0, i - r), i + 1))
            s |= {g for g in G if g <= i}
            for t in range(R):
                j = sm64_py(seed ^ (i * R + t)) % n
                if j <= i:
                    s.add(j)
        rows.append(sorted(s))
    return rows


def brute_block_graph(n, b, c, s, gb, seed):
    nb = -(-n // b)
    half = (c - 1) // 2
    allowed = []
    for J in range(nb):
        if J < gb:
            a = set(range(nb))
        else:
            a = {x for x in range(J - half, J + half + 1) if 0 <= x < nb}
            a |= set(range(gb))
            a |= {sm64_py(seed ^ (J * s + t)) % nb for t in range(s)}
        allowed.append(a)
    rows = [sorted(j for j in range(n) if j // b in allowed[i // b]) for i in range(n)]
    return rows, allowed


def csr_rows(row_ptr, col):
    return [list(col[row_ptr[i]:row_ptr[i + 1]]) for i in range(len(row_ptr) - 1)]


def dense_from_csr(A, row_ptr, col, n):
    M = np.zeros((n, n))
    for i in range(n):
        for e in range(row_ptr[i], row_ptr[i + 1]):
            M[i, col[e]] = A[e]
    return M


def random_qkv(n, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))


# ---------------------------------------------------------------- generator
def test_splitmix64_published_stream():
    # Seed-0 SplitMix64 stream: output k is the mix of state (k+1)*gamma, i.e.
    # the output function applied to k*gamma.
    expected = PINS["splitmix64_seed0_outputs"]
    gamma = 0x9E3779B97F4A7C15
    for k, want in enumerate(expected):
        assert oracle.splitmix64((k * gamma) & MASK64) == want
        assert sm64_py((k * gamma) & MASK64) == want


# ---------------------------------------------------------------- graph builder
def test_eight_position_pair_counts():
    # [S] Fig 1: 64 / 22 / 32 allowed pairs (global position 4 is index 3).
    assert oracle.token_graph(8, 7, 0, 0)[0][-1] == PINS["n8_full_pairs"][0]
    assert oracle.token_graph(8, 1, 0, 0)[0][-1] == PINS["n8_window_r1_pairs"][0]
    assert oracle.token_graph(8, 1, 0, 0, globals_idx=[3])[0][-1] == \
        PINS["n8_window_r1_global4_pairs"][0]
    # any interior position gives 32 too; a position at an end gives fewer overlaps
    for gpos in range(1, 7):
        assert oracle.token_graph(8, 1, 0, 0, globals_idx=[gpos])[0][-1] == 32


@pytest.mark.parametrize("n,r", [(1, 0), (5, 0), (8, 1), (9, 4), (64, 3), (100, 7), (513, 32),
                                 (1000, 99)])
def test_window_count_closed_form(n, r):
    # [S] eq 6, n >= 2r+1: |E_local| = n(2r+1) - r(r+1)
    assert n >= 2 * r + 1
    row_ptr, col = oracle.token_graph(n, r, 0, 0)
    assert row_ptr[-1] == n * (2 * r + 1) - r * (r + 1)


@pytest.mark.parametrize("n,r", [(4, 3), (10, 6), (7, 100)])
def test_window_short_sequence(n, r):
    # n < 2r+1: every row is truncated at one or both ends; sum the interval lengths
    want = sum(min(n - 1, i + r) - max(0, i - r) + 1 for i in range(n))
    assert oracle.token_graph(n, r, 0, 0)[0][-1] == want


def _window_plus_globals(n, r, g):
    total = 0
    for i in range(n):
        if i < g:
            total += n
            continue
        lo, hi = max(0, i - r), min(n - 1, i + r)
        total += (hi - lo + 1) + sum(1 for j in range(g) if j < lo or j > hi)
    return total


def test_workload_edge_counts():
    counts = golden.edge_counts()
    for w in workloads.ALL:
        c = counts[w.name]
        if w.kind == "token":
            n, r, g = w.n, w.r, w.n_globals
            assert c["window_edges"] == n * (2 * r + 1) - r * (r + 1)
            assert oracle.token_graph(n, r, 0, 0)[0][-1] == c["window_edges"]
            assert _window_plus_globals(n, r, g) == c["window_plus_globals"]
            assert oracle.token_graph(n, r, g, 0)[0][-1] == c["window_plus_globals"]
            row_ptr, col = oracle.token_graph(**w.graph_args())
        else:
            row_ptr, col = oracle.block_graph(**w.graph_args())
        assert row_ptr[-1] == c["total"], w.name


@pytest.mark.parametrize("n,r,G,R,seed", [
    (1, 0, [], 0, 0), (1, 3, [0], 5, 0), (2, 0, [], 3, 7), (17, 2, [0, 1], 4, 0),
    (33, 1, [5, 20], 6, 123), (40, 0, [], 8, 99), (64, 5, [0, 31, 63], 16, 2**63 + 5),
    (50, 30, [10], 3, 1), (96, 4, [], 40, 42),
])
def test_token_graph_brute_force(n, r, G, R, seed):
    row_ptr, col = oracle.token_graph(n, r, len(G), R, seed=seed, globals_idx=G)
    assert csr_rows(row_ptr, col) == brute_token_graph(n, r, G, R, seed)


def test_token_graph_dedup_and_order():
    # [S] sec 2.1: a key that is both window and global, or drawn twice, enters once.
    row_ptr, col = oracle.token_graph(64, 4, 8, 32, seed=11)
    for i in range(64):
        row = col[row_ptr[i]:row_ptr[i + 1]]
        assert np.all(np.diff(row) > 0)
        assert i in row  # self is always a neighbour ([D] sec 2.1 symbol table)


def test_block_example_twelve_blocks():
    # [S] sec 2: N=12 blocks of b=4, c=3 window, s=2 random, g_b=1 global.
    n, b = 48, 4
    row_ptr, col = oracle.block_graph(n, b, 3, 2, 1, seed=0)
    per_row = np.diff(row_ptr)
    block_pairs = [int(per_row[J * b:(J + 1) * b].sum()) for J in range(12)]
    assert block_pairs[0] == PINS["block12_global_row_pairs"][0]
    assert all(p <= PINS["block12_ordinary_row_pairs"][0] for p in block_pairs[1:])
    assert row_ptr[-1] <= PINS["block12_upper_bound"][0]
    assert 11 * PINS["block12_ordinary_row_pairs"][0] + PINS["block12_global_row_pairs"][0] == \
        PINS["block12_upper_bound"][0]
    # with every block allowed the pattern is full attention
    full_ptr, _ = oracle.block_graph(n, b, 23, 0, 0)
    assert full_ptr[-1] == PINS["block12_full_pairs"][0]
    rows, allowed = brute_block_graph(n, b, 3, 2, 1, 0)
    assert csr_rows(row_ptr, col) == rows
    assert block_pairs == [16 * len(a) for a in allowed]


@pytest.mark.parametrize("n,b,c,s,gb,seed", [
    (50, 16, 3, 1, 1, 0), (7, 4, 1, 0, 0, 3), (130, 64, 3, 3, 2, 0), (64, 8, 5, 2, 0, 9),
    (1, 64, 3, 3, 1, 0), (200, 8, 3, 4, 2, 77),
])
def test_block_graph_brute_force_ragged(n, b, c, s, gb, seed):
    # ragged last block ([S] sec 1.1 block padding): truncated, never padded
    row_ptr, col = oracle.block_graph(n, b, c, s, gb, seed=seed)
    rows, _ = brute_block_graph(n, b, c, s, gb, seed)
    assert csr_rows(row_ptr, col) == rows


# ---------------------------------------------------------------- softmax weights
def test_eight_position_one_hop_example():
    # [S] eq 8-10, position 4 of n=8 (index 3), r=1, scale already in the scores:
    # s = (0, ln2, 0) -> weights (1/4, 1/2, 1/4); o_4 = (1, 1.5).
    n, d = 8, 64
    Q = np.zeros((n, d)); K = np.zeros((n, d)); V = np.zeros((n, d))
    ln2 = PINS["onehop_scores"][1]
    K[3, 0] = 1.0
    Q[3, 0] = math.sqrt(d) * ln2          # q.k / sqrt(d) = ln 2
    V[2, :2] = PINS["onehop_v3"]; V[3, :2] = PINS["onehop_v4"]; V[4, :2] = PINS["onehop_v5"]
    row_ptr, col = oracle.token_graph(n, 1, 0, 0)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    assert list(col[row_ptr[3]:row_ptr[4]]) == [2, 3, 4]
    np.testing.assert_allclose(A[row_ptr[3]:row_ptr[4]], PINS["onehop_weights"], rtol=0, atol=1e-15)
    Z = oracle.diffuse(A, row_ptr, col, V, hops=1, alpha=0.0)
    np.testing.assert_allclose(Z[3, :2], PINS["onehop_out"], rtol=0, atol=1e-14)
    assert np.all(Z[3, 2:] == 0)


@pytest.mark.parametrize("seed", [0, 1])
def test_weights_equal_dense_masked_softmax(seed):
    # [S] sec 2.1 equivalence recipe: same boolean mask, dense reference with -inf
    # outside it; [S] eq 2-3.
    n, d = 40, 16
    Q, K, _ = random_qkv(n, d, seed)
    row_ptr, col = oracle.token_graph(n, 3, 2, 5, seed=seed)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    mask = np.full((n, n), -np.inf)
    for i in range(n):
        mask[i, col[row_ptr[i]:row_ptr[i + 1]]] = 0.0
    S = Q @ K.T / np.sqrt(d) + mask
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(dense_from_csr(A, row_ptr, col, n), P, rtol=1e-13, atol=1e-15)


def test_weights_rows_stochastic():
    # [D] after eq S.5: each row is non-negative and sums to 1
    n, d = 300, 64
    Q, K, _ = random_qkv(n, d, 5)
    Q *= 3.0  # spread the scores
    row_ptr, col = oracle.token_graph(n, 8, 3, 7, seed=3)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    assert np.all(A >= 0)
    sums = np.add.reduceat(A, row_ptr[:-1])
    np.testing.assert_allclose(sums, 1.0, rtol=0, atol=1e-14)


def test_full_graph_one_hop_is_dense_attention():
    # a full graph with hops=1, alpha=0 is textbook softmax(Q K^T / sqrt(d)) V
    n, d = 37, 64
    Q, K, V = random_qkv(n, d, 9)
    row_ptr, col = oracle.token_graph(n, n, 0, 0)
    out = oracle.forward(Q[None], K[None], V[None], row_ptr, col, hops=1, alpha=0.0)[0]
    S = Q @ K.T / np.sqrt(d)
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(out, P @ V, rtol=1e-12, atol=1e-13)


def test_scale_is_inverse_sqrt_head_width():
    # [S] eq 1: s_ij = q_i.k_j / sqrt(d_h) -- with d=16 a wrong scale changes the weights
    n, d = 3, 16
    Q = np.zeros((n, d)); K = np.zeros((n, d))
    Q[0, 0] = 4.0 * math.log(3.0)   # s_00 = ln 3 with scale 1/4
    K[0, 0] = 1.0
    row_ptr, col = oracle.token_graph(n, 2, 0, 0)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    np.testing.assert_allclose(A[:3], [3 / 5, 1 / 5, 1 / 5], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- diffusion
def test_three_token_example():
    # [D] sec 2.5: A = [[1/2,1/2,0],[0,1/2,1/2],[0,0,1]], alpha=0.1, K=2:
    # Z_(2),1 = 0.3475 V1 + 0.45 V2 + 0.2025 V3.
    A_dense = np.array(PINS["three_token_A"])
    row_ptr = np.array([0, 2, 4, 5]); col = np.array([0, 1, 1, 2, 2], dtype=np.int32)
    A = np.array([A_dense[i, j] for i in range(3) for j in col[row_ptr[i]:row_ptr[i + 1]]])
    Z = oracle.diffuse(A, row_ptr, col, np.eye(3), hops=int(PINS["three_token_hops"][0]),
                       alpha=PINS["three_token_alpha"][0])
    np.testing.assert_allclose(Z[0], PINS["three_token_row1"], rtol=0, atol=1e-15)


def test_finite_k_expansion_coefficients():
    # [D] sec 2.5: Z_(5) = (0.1 I + 0.09 A + 0.081 A^2 + 0.0729 A^3 + 0.06561 A^4
    #                       + 0.59049 A^5) V  for K=5, alpha=0.1; coefficients sum to 1.
    c = PINS["finiteK5_alpha01_coeffs"]
    assert abs(sum(c) - 1.0) < 1e-15
    n, d = 50, 8
    Q, K, V = random_qkv(n, d, 4)
    row_ptr, col = oracle.token_graph(n, 2, 2, 3, seed=8)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    M = dense_from_csr(A, row_ptr, col, n)
    want = sum(ck * np.linalg.matrix_power(M, k) for k, ck in enumerate(c)) @ V
    got = oracle.diffuse(A, row_ptr, col, V, hops=5, alpha=0.1)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_many_hops_reach_ppr_closed_form():
    # [D] sec 2.4: infinite-hop limit alpha [I - (1-alpha) A]^-1 V; 0.9^400 ~ 5e-19
    n, d = 48, 6
    Q, K, V = random_qkv(n, d, 6)
    row_ptr, col = oracle.token_graph(n, 3, 1, 4, seed=2)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    M = dense_from_csr(A, row_ptr, col, n)
    alpha = 0.1
    want = alpha * np.linalg.solve(np.eye(n) - (1 - alpha) * M, V)
    got = oracle.diffuse(A, row_ptr, col, V, hops=400, alpha=alpha)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_diffusion_special_cases():
    n, d = 30, 5
    Q, K, V = random_qkv(n, d, 7)
    row_ptr, col = oracle.token_graph(n, 2, 1, 3, seed=1)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    # eq S.7 with no iterations returns V
    np.testing.assert_array_equal(oracle.diffuse(A, row_ptr, col, V, hops=0, alpha=0.1), V)
    # alpha = 1 returns V ([D] sec 2.4)
    np.testing.assert_allclose(oracle.diffuse(A, row_ptr, col, V, hops=4, alpha=1.0), V,
                               rtol=0, atol=0)
    # a constant V is a fixed point: A is row-stochastic
    Vc = np.full((n, d), 2.5)
    np.testing.assert_allclose(oracle.diffuse(A, row_ptr, col, Vc, hops=6, alpha=0.3), Vc,
                               rtol=1e-14, atol=0)
    # alpha = 0, one hop is plain sparse attention A V ([S] eq 4)
    np.testing.assert_allclose(oracle.diffuse(A, row_ptr, col, V, hops=1, alpha=0.0),
                               dense_from_csr(A, row_ptr, col, n) @ V, rtol=1e-13, atol=1e-14)


def test_forward_units_and_threads_independent():
    # units are independent; splitting them over threads changes nothing
    B, H, n, d = 2, 3, 64, 64
    Q, K, V = synthetic.qkv(B, H, n, d, "fp32", seed=3)
    row_ptr, col = oracle.token_graph(n, 4, 2, 5)
    Q64, K64, V64 = (oracle.widen(x, "fp32") for x in (Q, K, V))
    one = oracle.forward(Q64, K64, V64, row_ptr, col, hops=3, alpha=0.2, nthreads=1)
    many = oracle.forward(Q64, K64, V64, row_ptr, col, hops=3, alpha=0.2, nthreads=4)
    np.testing.assert_array_equal(one, many)
    for b in range(B):
        for h in range(H):
            A = oracle.attention_weights(Q64[b, h], K64[b, h], row_ptr, col)
            Z = oracle.diffuse(A, row_ptr, col, V64[b, h], hops=3, alpha=0.2)
            np.testing.assert_array_equal(one[b, h], Z)


# ---------------------------------------------------------------- input generator
def test_synthetic_inputs_are_standard_normal_and_seeded():
    Q, K, V = synthetic.qkv(1, 2, 256, 64, "fp32", seed=0)
    allz = np.concatenate([Q.ravel(), K.ravel(), V.ravel()]).astype(np.float64)
    assert abs(allz.mean()) < 0.02 and abs(allz.std() - 1.0) < 0.02
    Q2, _, _ = synthetic.qkv(1, 2, 256, 64, "fp32", seed=0)
    np.testing.assert_array_equal(Q, Q2)
    Q3, _, _ = synthetic.qkv(1, 2, 256, 64, "fp32", seed=1)
    assert not np.array_equal(Q, Q3)


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0],
                 dtype=np.float32)
    bits = synthetic.to_bf16_bits(x)
    back = synthetic.bf16_bits_to_f32(bits)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 is a tie -> even (1+2^-6)
    np.testing.assert_array_equal(back, np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0],
                                                 dtype=np.float32))
    np.testing.assert_array_equal(oracle.widen(bits, "bf16"), back.astype(np.float64))


# ---------------------------------------------------------------- causal graph
@pytest.mark.parametrize("n,r", [(1, 0), (8, 1), (9, 4), (64, 3), (513, 32), (1000, 99)])
def test_causal_window_count_closed_form(n, r):
    # [S] sec 1.1: a causal window row holds at most r+1 history positions;
    # rows i < r hold i+1, so |E| = n(r+1) - r(r+1)/2 for n > r
    assert n > r
    row_ptr, _ = oracle.token_graph(n, r, 0, 0, causal=True)
    assert row_ptr[-1] == n * (r + 1) - r * (r + 1) // 2


@pytest.mark.parametrize("n,r,G,R,seed", [
    (1, 0, [], 0, 0), (1, 3, [0], 5, 0), (2, 0, [], 3, 7), (17, 2, [0, 1], 4, 0),
    (33, 1, [5, 20], 6, 123), (40, 0, [], 8, 99), (64, 5, [0, 31, 63], 16, 2**63 + 5),
    (50, 30, [10], 3, 1), (96, 4, [], 40, 42),
])
def test_causal_token_graph_brute_force(n, r, G, R, seed):
    row_ptr, col = oracle.token_graph(n, r, len(G), R, seed=seed, globals_idx=G, causal=True)
    assert csr_rows(row_ptr, col) == brute_causal_token_graph(n, r, G, R, seed)


def test_causal_graph_is_masked_bidirectional_graph():
    # [D] sec 2.6: the causal graph is the lower triangle of the same edge set;
    # every row keeps its self edge, so no softmax row is empty
    n = 200
    rp_b, col_b = oracle.token_graph(n, 6, 4, 5, seed=3, globals_idx=[0, 50, 120, 199])
    rp_c, col_c = oracle.token_graph(n, 6, 4, 5, seed=3, globals_idx=[0, 50, 120, 199],
                                     causal=True)
    for i, (rb, rc) in enumerate(zip(csr_rows(rp_b, col_b), csr_rows(rp_c, col_c))):
        assert rc == [j for j in rb if j <= i]
        assert rc[-1] == i
    # position 4 cannot read the future global 8 ([S] sec 1.2, causal remark)
    rp, col = oracle.token_graph(16, 1, 0, 0, causal=True, globals_idx=[8])
    assert 8 not in csr_rows(rp, col)[4] and 8 in csr_rows(rp, col)[9]


def test_causal_full_graph_one_hop_is_dense_causal_attention():
    # r >= n: every row reads all of its history; hops=1, alpha=0 is textbook
    # causal softmax(Q K^T / sqrt(d) + upper-triangular -inf) V
    n, d = 37, 64
    Q, K, V = random_qkv(n, d, 19)
    row_ptr, col = oracle.token_graph(n, n, 0, 0, causal=True)
    out = oracle.forward(Q[None], K[None], V[None], row_ptr, col, hops=1, alpha=0.0)[0]
    S = Q @ K.T / np.sqrt(d)
    S[np.triu_indices(n, 1)] = -np.inf
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(out, P @ V, rtol=1e-12, atol=1e-13)


def test_causal_diffusion_never_reads_the_future():
    # [D] sec 2.6: A lower-triangular => every A^k and the PPR sum are too, so
    # changing position p's Q, K or V leaves output rows < p exactly unchanged
    n, d, p = 96, 16, 40
    Q, K, V = random_qkv(n, d, 21)
    row_ptr, col = oracle.token_graph(n, 5, 2, 6, seed=4, globals_idx=[10, 70], causal=True)
    base = oracle.forward(Q[None], K[None], V[None], row_ptr, col, hops=5, alpha=0.1)[0]
    for X in (Q, K, V):
        Xp = X.copy()
        Xp[p] += 1.0
        args = [Q, K, V]
        args[[id(Q), id(K), id(V)].index(id(X))] = Xp
        pert = oracle.forward(*(a[None] for a in args), row_ptr, col, hops=5, alpha=0.1)[0]
        np.testing.assert_array_equal(pert[:p], base[:p])
        assert np.abs(pert[p:] - base[p:]).max() > 1e-6
    # row 0 reads only itself: A_00 = 1, so Z_k row 0 is V row 0 for every K
    np.testing.assert_allclose(base[0], V[0], rtol=0, atol=1e-15)
    A = oracle.attention_weights(Q, K, row_ptr, col)
    M = dense_from_csr(A, row_ptr, col, n)
    assert not np.triu(np.linalg.matrix_power(M, 5), 1).any()


# ---------------------------------------------------------------- dilated window
def test_dilated_window_page_example():
    # [S] sec 1.2 eq 11: r = 2, dilation 3 - position 10 reads 4, 7, 10, 13, 16 and not 9 or 11
    row_ptr, col = oracle.dilated_graph(40, 2, 3, 0, 0)
    assert list(col[row_ptr[10]:row_ptr[11]]) == [4, 7, 10, 13, 16]


@pytest.mark.parametrize("n,r,dl,G,R,seed,causal", [
    (50, 2, 3, [], 0, 0, False), (97, 4, 5, [0, 60], 6, 3, False), (64, 3, 7, [5], 4, 1, True),
    (20, 9, 4, [], 3, 2, False), (33, 1, 1, [2, 20], 5, 9, True),
])
def test_dilated_graph_brute_force(n, r, dl, G, R, seed, causal):
    rows = []
    for i in range(n):
        if i in G:
            s = set(range(n))
        else:
            s = {i + k * dl for k in range(-r, r + 1) if 0 <= i + k * dl < n}
            s |= set(G)
            s |= {sm64_py(seed ^ (i * R + t)) % n for t in range(R)}
        if causal:
            s = {j for j in s if j <= i}
        rows.append(sorted(s))
    row_ptr, col = oracle.dilated_graph(n, r, dl, len(G), R, seed=seed, globals_idx=G, causal=causal)
    assert csr_rows(row_ptr, col) == rows


def test_dilation_one_is_the_sliding_window():
    for causal in (False, True):
        a = oracle.dilated_graph(300, 7, 1, 3, 5, seed=4, causal=causal)
        b = oracle.token_graph(300, 7, 3, 5, seed=4, causal=causal)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def _components(row_ptr, col, n):
    parent = list(range(n))

    def find(x):
        while parent[x] != x:
            parent[x] = parent[parent[x]]
            x = parent[x]
        return x
    for i in range(n):
        for j in col[row_ptr[i]:row_ptr[i + 1]]:
            parent[find(i)] = find(int(j))
    return len({find(i) for i in range(n)})


def test_dilation_splits_the_graph_by_residue():
    # [S] sec 1.2: with one dilation 3 and nothing else, edges join only positions that
    # agree mod 3 - three components; one global token reconnects them
    assert _components(*oracle.dilated_graph(60, 2, 3, 0, 0), 60) == 3
    assert _components(*oracle.dilated_graph(60, 2, 3, 1, 0), 60) == 1


def test_twelve_layer_reach_example():
    # [S] sec 2.1: 12 layers reaching distance 900 need r >= 75 (12 * 75 = 900); for
    # n = 8192 the page counts 8192 * 151 = 1,236,992 local edges ignoring the ends,
    # against 8192^2 = 67,108,864 for full attention (about 1.84 %); the ends remove
    # r(r+1) = 5,700 of them ([S] eq 6)
    r = -(-900 // 12)
    assert r == 75
    nominal = 8192 * (2 * r + 1)
    assert nominal == 1_236_992 and round(100 * nominal / 8192 ** 2, 2) == 1.84
    row_ptr, _ = oracle.token_graph(8192, r, 0, 0)
    assert row_ptr[-1] == nominal - r * (r + 1) == 1_231_292
