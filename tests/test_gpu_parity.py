"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Graphs must match bit for bit; outputs within the tolerances in helpers.py.
Small cases span several tiles and ragged tails; the full-size workloads run
in the benchmark's launch configuration and are compared on sampled units
(whole (batch, head) units, which the oracle computes independently), plus
properties that hold at any size for every unit.
"""
import math

import numpy as np
import pytest

import oracle
from sparse_long_sequence_gb300 import synthetic, workloads
from tests.helpers import check_output, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_long_sequence_gb300 import binding
    return binding


def oracle_graph(w_or_args, kind="token"):
    if kind == "token":
        return oracle.token_graph(**w_or_args)
    return oracle.block_graph(**w_or_args)


def build_graph(dl, args, kind="token"):
    if kind == "token":
        a = dict(args)
        gi = a.pop("globals_idx", None)
        return dl.diffuser_build_graph(a["n"], a["r"], a["n_globals"], global_idx=gi,
                                       rand_per_row=a["rand_per_row"], seed=a["seed"])
    return dl.diffuser_build_block_graph(**args)


# ---------------------------------------------------------------- graphs (bit-exact)
TOKEN_CASES = [
    dict(n=1, r=0, n_globals=0, rand_per_row=0, seed=0),
    dict(n=1, r=5, n_globals=1, rand_per_row=3, seed=0),
    dict(n=2, r=0, n_globals=0, rand_per_row=3, seed=7),
    dict(n=17, r=2, n_globals=2, rand_per_row=4, seed=0),
    dict(n=300, r=8, n_globals=3, rand_per_row=5, seed=0),
    dict(n=500, r=0, n_globals=0, rand_per_row=40, seed=99),
    dict(n=640, r=600, n_globals=5, rand_per_row=2, seed=3),
    dict(n=1000, r=31, n_globals=0, rand_per_row=0, seed=0),
    dict(n=777, r=13, n_globals=4, rand_per_row=9, seed=2 ** 63 + 11, globals_idx=[0, 100, 401, 776]),
    dict(n=4096, r=256, n_globals=16, rand_per_row=32, seed=1),
]
BLOCK_CASES = [
    dict(n=50, block=16, window_blocks=3, rand_blocks=1, global_blocks=1, seed=0),
    dict(n=1000, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=0),
    dict(n=48, block=4, window_blocks=3, rand_blocks=2, global_blocks=1, seed=0),
    dict(n=130, block=64, window_blocks=5, rand_blocks=3, global_blocks=0, seed=5),
    dict(n=7, block=64, window_blocks=1, rand_blocks=0, global_blocks=1, seed=0),
]


@pytest.mark.parametrize("args", TOKEN_CASES)
def test_token_graph_bit_exact(dl, args):
    g = build_graph(dl, args)
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    o_ptr, o_col = oracle_graph(args)
    np.testing.assert_array_equal(row_ptr, o_ptr)
    np.testing.assert_array_equal(col, o_col)


@pytest.mark.parametrize("args", BLOCK_CASES)
def test_block_graph_bit_exact(dl, args):
    g = build_graph(dl, args, "block")
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    o_ptr, o_col = oracle_graph(args, "block")
    np.testing.assert_array_equal(row_ptr, o_ptr)
    np.testing.assert_array_equal(col, o_col)


@pytest.mark.parametrize("w", workloads.ALL, ids=lambda w: w.name)
def test_workload_graph_bit_exact(dl, w):
    g = build_graph(dl, w.graph_args(), w.kind)
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    o_ptr, o_col = oracle_graph(w.graph_args(), w.kind)
    assert g.nnz == o_ptr[-1]
    np.testing.assert_array_equal(row_ptr, o_ptr)
    np.testing.assert_array_equal(col, o_col)


# ---------------------------------------------------------------- pins on the device
def test_eight_position_one_hop_example_on_device(dl):
    # "1.2.1 Static sparsity", eq 8-10: weights (1/4, 1/2, 1/4), o_4 = (1, 1.5)
    import torch
    n, d = 8, 64
    Q = np.zeros((1, 1, n, d), np.float32); K = np.zeros_like(Q); V = np.zeros_like(Q)
    K[0, 0, 3, 0] = 1.0
    Q[0, 0, 3, 0] = 8.0 * math.log(2.0)
    V[0, 0, 2, :2] = (2, 0); V[0, 0, 3, :2] = (0, 2); V[0, 0, 4, :2] = (2, 2)
    g = dl.diffuser_build_graph(n, 1, 0, rand_per_row=0)
    Qd, Kd, Vd = (to_device(x, "fp32") for x in (Q, K, V))
    A = dl.diffuser_attention_weights(Qd, Kd, g)
    out = dl.diffuser_forward(Qd, Kd, Vd, g, hops=1, alpha=0.0)
    torch.cuda.synchronize()
    row_ptr, _ = dl.diffuser_graph_copy_csr(g)
    np.testing.assert_allclose(A[0, row_ptr[3]:row_ptr[4]].cpu().numpy(), [0.25, 0.5, 0.25],
                               atol=1e-7)
    np.testing.assert_allclose(out[0, 0, 3, :2].cpu().numpy(), [1.0, 1.5], atol=1e-6)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_three_token_example_on_device(dl, dtype):
    # Diffuser notes sec 2.5: Z_(2),1 = 0.3475 V1 + 0.45 V2 + 0.2025 V3
    import torch
    g = dl.diffuser_build_graph(3, 1, 0, rand_per_row=0)
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    dense = np.array([[0.5, 0.5, 0], [0, 0.5, 0.5], [0, 0, 1]])
    A = np.array([dense[i, j] for i in range(3) for j in col[row_ptr[i]:row_ptr[i + 1]]],
                 np.float32)
    V = np.zeros((1, 1, 3, 64), np.float32)
    V[0, 0, 0, 0] = V[0, 0, 1, 1] = V[0, 0, 2, 2] = 1.0
    Vd = to_device(synthetic.to_bf16_bits(V) if dtype == "bf16" else V, dtype)
    out = dl.diffuser_diffuse_csr(g, torch.from_numpy(A).cuda(), Vd, hops=2, alpha=0.1)
    torch.cuda.synchronize()
    got = to_f64(out)[0, 0, 0, :3]
    tol = 1e-6 if dtype == "fp32" else 2e-3
    np.testing.assert_allclose(got, [0.3475, 0.45, 0.2025], atol=tol)


# ---------------------------------------------------------------- forward parity, small
SMALL = [
    # (B, H, n, r, g, R, hops, alpha)
    (1, 1, 1, 0, 0, 0, 5, 0.1),
    (1, 2, 300, 8, 3, 5, 5, 0.1),
    (2, 3, 257, 32, 4, 8, 5, 0.1),
    (1, 2, 1000, 64, 8, 16, 3, 0.25),
    (1, 1, 640, 640, 0, 0, 1, 0.0),      # full graph, one hop, alpha 0: dense attention
    (2, 2, 513, 20, 2, 4, 2, 1.0),       # alpha 1 returns V
    (1, 4, 700, 17, 5, 3, 0, 0.1),       # hops 0 returns V
    (1, 1, 389, 128, 2, 32, 5, 0.1),     # ragged tail against 128-row tiles
    # window radius padded to an odd multiple of 64 (a tile's own keys span two key
    # chunks) and a last tile of fewer than 64 rows (the second one is out of range)
    (1, 2, 650, 150, 3, 8, 5, 0.1),
    (1, 3, 1034, 150, 5, 8, 3, 0.1),
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B%dH%dn%dr%dg%dR%dK%da%s" % c)
def test_forward_small(dl, case, dtype):
    import torch
    B, H, n, r, gn, R, hops, alpha = case
    g = dl.diffuser_build_graph(n, r, gn, rand_per_row=R, seed=0)
    o_ptr, o_col = oracle.token_graph(n, r, gn, R, seed=0)
    Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=n)
    out = dl.diffuser_forward(to_device(Q, dtype), to_device(K, dtype), to_device(V, dtype), g,
                              hops, alpha)
    torch.cuda.synchronize()
    ref = oracle.forward(oracle.widen(Q, dtype), oracle.widen(K, dtype), oracle.widen(V, dtype),
                         o_ptr, o_col, hops, alpha, nthreads=4)
    check_output(to_f64(out), ref, dtype)
    if hops == 0 or alpha == 1.0:
        np.testing.assert_array_equal(to_f64(out), oracle.widen(V, dtype))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("args", BLOCK_CASES[:4], ids=lambda a: "n%d_b%d" % (a["n"], a["block"]))
def test_forward_block_graph_small(dl, args, dtype):
    import torch
    g = build_graph(dl, args, "block")
    o_ptr, o_col = oracle_graph(args, "block")
    B, H, n = 2, 2, args["n"]
    Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=5)
    out = dl.diffuser_forward(to_device(Q, dtype), to_device(K, dtype), to_device(V, dtype), g,
                              5, 0.1)
    torch.cuda.synchronize()
    ref = oracle.forward(oracle.widen(Q, dtype), oracle.widen(K, dtype), oracle.widen(V, dtype),
                         o_ptr, o_col, 5, 0.1, nthreads=4)
    check_output(to_f64(out), ref, dtype)


@pytest.mark.parametrize("causal", [False, True], ids=["bidirectional", "causal"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_attention_weights_parity(dl, dtype, causal):
    import torch
    B, H, n = 1, 3, 600
    build = dl.diffuser_build_causal_graph if causal else dl.diffuser_build_graph
    g = build(n, 40, 4, rand_per_row=12, seed=0)
    o_ptr, o_col = oracle.token_graph(n, 40, 4, 12, seed=0, causal=causal)
    Q, K, _ = synthetic.qkv(B, H, n, 64, dtype, seed=2)
    A = dl.diffuser_attention_weights(to_device(Q, dtype), to_device(K, dtype), g)
    torch.cuda.synchronize()
    A = A.cpu().numpy().astype(np.float64)
    Qw, Kw = oracle.widen(Q, dtype), oracle.widen(K, dtype)
    for u in range(B * H):
        ref = oracle.attention_weights(Qw[0, u], Kw[0, u], o_ptr, o_col)
        np.testing.assert_allclose(A[u], ref, rtol=2e-5, atol=1e-8)


@pytest.mark.parametrize("causal", [False, True], ids=["bidirectional", "causal"])
@pytest.mark.parametrize("case", [(1, 2, 300, 8, 3, 5), (2, 3, 1000, 64, 8, 16),
                                  (1, 2, 777, 33, 0, 7), (1, 1, 4096, 256, 16, 32),
                                  (1, 2, 650, 150, 3, 8),
                                  # 16 global rows (two 16-row global-row images, used by
                                  # alternate tiles), 17 and 32 (one 32-row image); radii
                                  # whose tiles meet their own keys in their first chunk
                                  (1, 2, 1000, 32, 16, 16), (2, 1, 900, 40, 17, 8),
                                  (1, 1, 1200, 64, 32, 8)],
                         ids=lambda c: "B%dH%dn%dr%dg%dR%d" % c)
def test_band_path_matches_csr_path(dl, case, causal):
    # the tensor-core band path and the general CSR path on the same inputs
    import torch
    B, H, n, r, gn, R = case
    build = dl.diffuser_build_causal_graph if causal else dl.diffuser_build_graph
    g = build(n, r, gn, rand_per_row=R, seed=3)
    Q, K, V = synthetic.qkv(B, H, n, 64, "bf16", seed=11)
    Qd, Kd, Vd = (to_device(x, "bf16") for x in (Q, K, V))
    try:
        dl.diffuser_set_path(dl.DIFFUSER_PATH_CSR)
        ref = to_f64(dl.diffuser_forward(Qd, Kd, Vd, g, 5, 0.1))
    finally:
        dl.diffuser_set_path(dl.DIFFUSER_PATH_AUTO)
    out = to_f64(dl.diffuser_forward(Qd, Kd, Vd, g, 5, 0.1))
    torch.cuda.synchronize()
    assert dl.diffuser_graph_status(g) == 0
    o_ptr, o_col = oracle.token_graph(n, r, gn, R, seed=3, causal=causal)
    oref = oracle.forward(oracle.widen(Q, "bf16"), oracle.widen(K, "bf16"),
                          oracle.widen(V, "bf16"), o_ptr, o_col, 5, 0.1, nthreads=4)
    check_output(out, oref, "bf16")
    check_output(ref, oref, "bf16")
    # both round the same fp32-accurate values to bf16: at most one bf16 ulp apart
    assert np.abs(out - ref).max() <= 2 ** -7 * np.abs(oref).max()


def test_constant_v_is_preserved(dl):
    # A is row-stochastic, so a constant V is a fixed point of every hop
    import torch
    B, H, n = 2, 2, 1100
    g = dl.diffuser_build_graph(n, 100, 6, rand_per_row=10)
    Q, K, _ = synthetic.qkv(B, H, n, 64, "bf16", seed=3)
    V = torch.full((B, H, n, 64), 0.75, dtype=torch.bfloat16, device="cuda")
    out = dl.diffuser_forward(to_device(Q, "bf16"), to_device(K, "bf16"), V, g, 5, 0.1)
    torch.cuda.synchronize()
    assert float((out.float() - 0.75).abs().max()) <= 0.75 * 2 ** -8


def test_band_path_repeatable_under_load(dl):
    # Many tiles per SM over repeated calls: a constant V must come back exactly
    # (A is row-stochastic) on every unit, every call.  Guards the tensor-core
    # pipeline against stale shared-memory or TMEM stages.
    import torch
    B, H, n = 32, 8, 1024
    g = dl.diffuser_build_graph(n, 32, 8, rand_per_row=16)
    Q, K, _ = synthetic.qkv(B, H, n, 64, "bf16", seed=5)
    Qd, Kd = to_device(Q, "bf16"), to_device(K, "bf16")
    V = torch.full((B, H, n, 64), 0.5, dtype=torch.bfloat16, device="cuda")
    ws = dl.alloc_workspace(dl.diffuser_workspace_size(g, B, H, 64, dl.DIFFUSER_DTYPE_BF16))
    for hops in (1, 5, 5, 5, 5, 5):
        out = dl.diffuser_forward(Qd, Kd, V, g, hops, 0.1, workspace=ws)
        torch.cuda.synchronize()
        assert float((out.float() - 0.5).abs().max()) <= 0.5 * 2 ** -8
    assert dl.diffuser_graph_status(g) == 0


def test_replayed_forward_matches_direct(dl):
    # The same forward five times: the first runs its kernels directly, the
    # second is captured into a CUDA graph, the next ones replay it, and the
    # last (inside an open profile) launches directly again.  Every output must
    # be bit-identical, every call must count the same launches, and the
    # profile must see each kernel.
    import torch
    B, H, n = 2, 3, 1536
    g = dl.diffuser_build_graph(n, 64, 4, rand_per_row=8)
    Q, K, V = synthetic.qkv(B, H, n, 64, "bf16", seed=11)
    Qd, Kd, Vd = (to_device(x, "bf16") for x in (Q, K, V))
    ws = dl.alloc_workspace(dl.diffuser_workspace_size(g, B, H, 64, dl.DIFFUSER_DTYPE_BF16))
    out = torch.empty_like(Vd)
    ref, counts, prof = None, [], None
    for call in range(5):
        out.zero_()
        torch.cuda.synchronize()
        before, _ = dl.diffuser_launch_count()
        if call == 4:
            dl.diffuser_profile_begin()
        dl.diffuser_forward(Qd, Kd, Vd, g, 3, 0.1, out=out, workspace=ws)
        if call == 4:
            prof = dl.diffuser_profile_end()
        torch.cuda.synchronize()
        after, _ = dl.diffuser_launch_count()
        counts.append(after - before)
        if ref is None:
            ref = out.clone()
        else:
            assert torch.equal(out, ref), f"call {call} differs from the first"
    assert counts[0] > 0 and len(set(counts)) == 1, counts
    assert sum(v[1] for v in prof.values()) == counts[0]
    assert all(v[0] > 0 for v in prof.values() if v[1])
    assert dl.diffuser_graph_status(g) == 0


def test_band_dealing_table_and_snake_order_agree(dl):
    # The band hop kernel's tiles go to the CTAs through a deal table (the snake
    # order, then trades between the busiest and the least busy CTA), built on the
    # first forward with a given B*H outside stream capture; a forward issued while
    # the caller's stream is capturing deals them in snake order.  Each tile is
    # computed by one CTA in a fixed order either way (the global rows' shares are
    # added in tile order), so the two outputs agree bit for bit.  The text-like
    # shape (24 units of 32 tiles on 152 CTAs) is one where the two dealings differ.
    import torch
    g = dl.diffuser_build_graph(4096, 256, 16, rand_per_row=32)
    assert dl.diffuser_kernels_for(g, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_BAND
    # a plain forward with another B*H first: the one-time set-up happens outside
    # the capture below, and no table exists yet for B*H = 24
    Q1, K1, V1 = (to_device(x, "bf16") for x in synthetic.qkv(1, 1, 4096, 64, "bf16", seed=10))
    dl.diffuser_forward(Q1, K1, V1, g, 5, 0.1)
    torch.cuda.synchronize()
    B, H = 2, 12
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(B, H, 4096, 64, "bf16", seed=12))
    ws = dl.alloc_workspace(dl.diffuser_workspace_size(g, B, H, 64, dl.DIFFUSER_DTYPE_BF16))
    out_snake = torch.empty_like(V)
    side = torch.cuda.Stream()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=side):
        dl.diffuser_forward(Q, K, V, g, 5, 0.1, out=out_snake, workspace=ws)
    cg.replay()
    torch.cuda.synchronize()
    out_deal = dl.diffuser_forward(Q, K, V, g, 5, 0.1)
    torch.cuda.synchronize()
    assert dl.diffuser_graph_status(g) == 0
    assert torch.equal(out_snake, out_deal)


def test_bad_workspace_launches_nothing(dl):
    import torch
    g = dl.diffuser_build_graph(256, 8, 1, rand_per_row=2)
    Q = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    need = dl.diffuser_workspace_size(g, 1, 1, 64, dl.DIFFUSER_DTYPE_BF16)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    before, _ = dl.diffuser_launch_count()
    with pytest.raises(dl.DiffuserError) as e:
        dl.diffuser_forward(Q, Q.clone(), Q.clone(), g, 5, 0.1, workspace=small)
    assert e.value.status == 7
    with pytest.raises(dl.DiffuserError) as e:
        dl.diffuser_forward(Q, Q.clone(), Q.clone(), g, 5, 1.5)
    assert e.value.status == 1
    after, _ = dl.diffuser_launch_count()
    assert after == before


@pytest.mark.parametrize("pinned_out", [True, False], ids=["pinned-out", "pageable-out"])
def test_forward_host_buffers(dl, pinned_out):
    # the end-to-end entry point: host buffers in, host buffer out (a pinned,
    # mapped `out` is written in place by the last hop; a pageable one is copied back)
    import torch
    B, H, n = 1, 2, 513
    g = dl.diffuser_build_graph(n, 16, 2, rand_per_row=4)
    Q, K, V = synthetic.qkv(B, H, n, 64, "bf16", seed=8)
    Qh, Kh, Vh = (torch.from_numpy(x).view(torch.bfloat16).pin_memory() for x in (Q, K, V))
    out = torch.empty_like(Vh).pin_memory() if pinned_out else torch.empty(Vh.shape, dtype=Vh.dtype)
    ws = dl.alloc_workspace(dl.diffuser_host_workspace_size(g, B, H, 64, dl.DIFFUSER_DTYPE_BF16))
    dl.diffuser_forward_host(Qh, Kh, Vh, g, 5, 0.1, out, ws)
    torch.cuda.synchronize()
    ref_dev = dl.diffuser_forward(Qh.cuda(), Kh.cuda(), Vh.cuda(), g, 5, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_dev.cpu())


# ---------------------------------------------------------------- causal graph
def build_causal(dl, args):
    a = dict(args)
    gi = a.pop("globals_idx", None)
    return dl.diffuser_build_causal_graph(a["n"], a["r"], a["n_globals"], global_idx=gi,
                                          rand_per_row=a["rand_per_row"], seed=a["seed"])


@pytest.mark.parametrize("args", TOKEN_CASES)
def test_causal_graph_bit_exact(dl, args):
    g = build_causal(dl, args)
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    o_ptr, o_col = oracle.token_graph(**args, causal=True)
    np.testing.assert_array_equal(row_ptr, o_ptr)
    np.testing.assert_array_equal(col, o_col)


CAUSAL_SMALL = [  # (B, H, n, r, |G|, R, K, alpha)
    (2, 3, 300, 8, 3, 5, 5, 0.1),
    (1, 2, 1000, 64, 8, 16, 5, 0.1),
    (1, 1, 640, 640, 0, 0, 1, 0.0),      # full causal graph, one hop: dense causal attention
    (1, 2, 389, 256, 2, 32, 5, 0.1),     # the text workload's r, |G| and R on a ragged n
    (1, 2, 513, 20, 2, 4, 2, 1.0),       # alpha 1 returns V
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("case", CAUSAL_SMALL, ids=lambda c: "B%dH%dn%dr%dg%dR%dK%da%s" % c)
def test_causal_forward_small(dl, case, dtype):
    import torch
    B, H, n, r, gn, R, hops, alpha = case
    g = dl.diffuser_build_causal_graph(n, r, gn, rand_per_row=R, seed=0)
    o_ptr, o_col = oracle.token_graph(n, r, gn, R, seed=0, causal=True)
    Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=n + 1)
    out = dl.diffuser_forward(to_device(Q, dtype), to_device(K, dtype), to_device(V, dtype), g,
                              hops, alpha)
    torch.cuda.synchronize()
    ref = oracle.forward(oracle.widen(Q, dtype), oracle.widen(K, dtype), oracle.widen(V, dtype),
                         o_ptr, o_col, hops, alpha, nthreads=4)
    assert dl.diffuser_graph_status(g) == 0
    check_output(to_f64(out), ref, dtype)
    if alpha == 1.0:
        np.testing.assert_array_equal(to_f64(out), oracle.widen(V, dtype))


def test_causal_forward_never_reads_the_future(dl):
    # A lower-triangular: changing position p's V leaves every output row < p
    # bit-identical on the device; row 0 reads only itself, so it returns V_0
    import torch
    B, H, n, p = 1, 4, 1500, 700
    g = dl.diffuser_build_causal_graph(n, 64, 4, global_idx=[3, 650, 900, 1400],
                                       rand_per_row=8, seed=5)
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(B, H, n, 64, "bf16", seed=12))
    base = dl.diffuser_forward(Q, K, V, g, 5, 0.1)
    V2 = V.clone()
    V2[:, :, p] += 1.0
    pert = dl.diffuser_forward(Q, K, V2, g, 5, 0.1)
    torch.cuda.synchronize()
    assert dl.diffuser_graph_status(g) == 0
    assert torch.equal(base[:, :, :p], pert[:, :, :p])
    assert not torch.equal(base[:, :, p:], pert[:, :, p:])
    assert torch.equal(base[:, :, 0], V[:, :, 0])


def test_causal_text_workload_sampled_units(dl):
    # the text workload's sizes (B2 H12 n4096 r256 |G|16 R32) on the causal graph,
    # whole units sampled against the oracle
    import torch
    B, H, n, r, gn, R = 2, 12, 4096, 256, 16, 32
    dtype = "bf16"
    g = dl.diffuser_build_causal_graph(n, r, gn, rand_per_row=R, seed=1)
    o_ptr, o_col = oracle.token_graph(n, r, gn, R, seed=1, causal=True)
    assert g.nnz == o_ptr[-1]
    Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=4)
    out = dl.diffuser_forward(to_device(Q, dtype), to_device(K, dtype), to_device(V, dtype), g,
                              5, 0.1)
    torch.cuda.synchronize()
    got = to_f64(out).reshape(B * H, n, 64)
    Qw, Kw, Vw = (oracle.widen(x, dtype).reshape(B * H, n, 64) for x in (Q, K, V))
    units = _sample_units(B * H)
    ref = oracle.forward(Qw[units], Kw[units], Vw[units], o_ptr, o_col, 5, 0.1, nthreads=3)
    check_output(got[units], ref, dtype)


def test_causal_forward_host_buffers(dl):
    # host buffers through the end-to-end entry point take the same CSR path
    import torch
    B, H, n = 1, 2, 513
    g = dl.diffuser_build_causal_graph(n, 16, 2, rand_per_row=4)
    Q, K, V = synthetic.qkv(B, H, n, 64, "bf16", seed=9)
    Qh, Kh, Vh = (torch.from_numpy(x).view(torch.bfloat16).pin_memory() for x in (Q, K, V))
    out = torch.empty_like(Vh).pin_memory()
    ws = dl.alloc_workspace(dl.diffuser_host_workspace_size(g, B, H, 64, dl.DIFFUSER_DTYPE_BF16))
    dl.diffuser_forward_host(Qh, Kh, Vh, g, 5, 0.1, out, ws)
    torch.cuda.synchronize()
    ref_dev = dl.diffuser_forward(Qh.cuda(), Kh.cuda(), Vh.cuda(), g, 5, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_dev.cpu())


# ---------------------------------------------------------------- full-size workloads
def _sample_units(units: int):
    return sorted({0, units // 2, units - 1})


@pytest.mark.slow
@pytest.mark.parametrize("w", workloads.ALL, ids=lambda w: w.name)
def test_workload_full_size(dl, w):
    """Full-size forward (the benchmark's launch configuration); sampled units
    against the oracle, plus alpha=1 and constant-V properties on every unit."""
    import torch
    g = build_graph(dl, w.graph_args(), w.kind)
    o_ptr, o_col = oracle_graph(w.graph_args(), w.kind)
    Q, K, V = synthetic.qkv(w.B, w.H, w.n, w.d, w.dtype, seed=w.seed)
    Qd, Kd, Vd = (to_device(x, w.dtype) for x in (Q, K, V))
    ws = dl.alloc_workspace(dl.diffuser_workspace_size(g, w.B, w.H, w.d,
                                                       1 if w.dtype == "bf16" else 0))
    out = dl.diffuser_forward(Qd, Kd, Vd, g, w.hops, w.alpha, workspace=ws)
    torch.cuda.synchronize()
    got = to_f64(out).reshape(w.units, w.n, w.d)
    Qw = oracle.widen(Q, w.dtype).reshape(w.units, w.n, w.d)
    Kw = oracle.widen(K, w.dtype).reshape(w.units, w.n, w.d)
    Vw = oracle.widen(V, w.dtype).reshape(w.units, w.n, w.d)
    units = _sample_units(w.units)
    ref = oracle.forward(Qw[units], Kw[units], Vw[units], o_ptr, o_col, w.hops, w.alpha,
                         nthreads=len(units))
    check_output(got[units], ref, w.dtype)
    # properties on every unit: alpha = 1 gives V exactly; constant V is preserved
    out1 = dl.diffuser_forward(Qd, Kd, Vd, g, w.hops, 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, Vd)
    Vc = torch.full_like(Vd, 0.5)
    outc = dl.diffuser_forward(Qd, Kd, Vc, g, w.hops, w.alpha, workspace=ws)
    torch.cuda.synchronize()
    assert float((outc.float() - 0.5).abs().max()) <= 0.5 * 2 ** -8
