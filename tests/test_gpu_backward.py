"""GPU parity of diffuser_backward against the oracle's backward.

Tolerances: fp32 max|got - ref| <= 1e-4 * max|ref| per tensor; bf16 per-row
max|got - ref| / max|ref_row| <= 4e-3 (the bf16 rounding of the gradient is 2^-9).
"""
import numpy as np
import pytest

import oracle
from sparse_long_sequence_gb300 import synthetic
from tests.helpers import to_device, to_f64, row_relative_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_long_sequence_gb300 import binding
    return binding


def check_grad(got, ref, dtype):
    assert np.all(np.isfinite(got))
    if dtype == "fp32":
        err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
        assert err <= 1e-4, err
    else:
        assert row_relative_error(got, ref) <= 4e-3


CASES = [  # (B, H, n, r, g, R, hops, alpha, causal)
    (1, 2, 300, 8, 3, 5, 5, 0.1, False),
    (2, 1, 517, 40, 4, 12, 3, 0.2, False),
    (1, 2, 300, 8, 3, 5, 5, 0.1, True),
    (1, 1, 640, 640, 0, 0, 1, 0.0, False),
    (1, 2, 389, 256, 2, 32, 5, 0.1, True),
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("case", CASES)
def test_backward_small(dl, case, dtype):
    import torch
    B, H, n, r, gn, R, hops, alpha, causal = case
    build = dl.diffuser_build_causal_graph if causal else dl.diffuser_build_graph
    g = build(n, r, gn, rand_per_row=R, seed=0)
    o_ptr, o_col = oracle.token_graph(n, r, gn, R, seed=0, causal=causal)
    Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=n)
    dO, _, _ = synthetic.qkv(B, H, n, 64, dtype, seed=n + 7)
    dQ, dK, dV = dl.diffuser_backward(*(to_device(x, dtype) for x in (Q, K, V, dO)), g, hops, alpha)
    torch.cuda.synchronize()
    ref = oracle.backward(*(oracle.widen(x, dtype) for x in (Q, K, V, dO)), o_ptr, o_col, hops, alpha)
    for got, want in zip((dQ, dK, dV), ref):
        check_grad(to_f64(got), want, dtype)


@pytest.mark.parametrize("kind", ["bidirectional", "causal", "block"])
def test_backward_band_kernels_match_csr_kernels(dl, kind):
    # On a token graph with a plain window the backward takes the window's edges with
    # band kernels (64 x 64 tiles in shared memory) and the other edges with CSR
    # kernels; on a block graph of 64-token blocks the band kernels take every edge,
    # block by block.  With the CSR path forced, CSR kernels take every edge.  Both
    # sum in fp32, in fixed but different orders, so they agree to within fp32
    # rounding.  The window (r = 100) is wider than a tile; n = 700 and n = 1000
    # leave a ragged last tile (block).
    import torch
    if kind == "block":
        n = 1000
        g = dl.diffuser_build_block_graph(n=n, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=4)
    else:
        n = 700
        build = dl.diffuser_build_causal_graph if kind == "causal" else dl.diffuser_build_graph
        g = build(n, 100, 3, rand_per_row=9, seed=2)
    Q, K, V = (to_device(x, "fp32") for x in synthetic.qkv(1, 2, n, 64, "fp32", seed=21))
    dO = to_device(synthetic.qkv(1, 2, n, 64, "fp32", seed=22)[0], "fp32")
    band = dl.diffuser_backward(Q, K, V, dO, g, 5, 0.1)
    torch.cuda.synchronize()
    dl.diffuser_set_path(dl.DIFFUSER_PATH_CSR)
    try:
        csr = dl.diffuser_backward(Q, K, V, dO, g, 5, 0.1)
        torch.cuda.synchronize()
    finally:
        dl.diffuser_set_path(dl.DIFFUSER_PATH_AUTO)
    for x, y in zip(band, csr):
        x, y = to_f64(x), to_f64(y)
        assert np.abs(x - y).max() <= 1e-5 * np.abs(y).max()


def test_backward_block_graph(dl):
    import torch
    args = dict(n=1000, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=0)
    g = dl.diffuser_build_block_graph(**args)
    o_ptr, o_col = oracle.block_graph(**args)
    Q, K, V = synthetic.qkv(1, 2, 1000, 64, "fp32", seed=1)
    dO, _, _ = synthetic.qkv(1, 2, 1000, 64, "fp32", seed=2)
    got = dl.diffuser_backward(*(to_device(x, "fp32") for x in (Q, K, V, dO)), g, 5, 0.1)
    torch.cuda.synchronize()
    ref = oracle.backward(Q.astype(np.float64), K.astype(np.float64), V.astype(np.float64),
                          dO.astype(np.float64), o_ptr, o_col, 5, 0.1)
    for a, b in zip(got, ref):
        check_grad(to_f64(a), b, "fp32")


def test_backward_special_cases_and_repeatability(dl):
    import torch
    g = dl.diffuser_build_graph(300, 8, 2, rand_per_row=4)
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(1, 2, 300, 64, "bf16", seed=3))
    dO = to_device(synthetic.qkv(1, 2, 300, 64, "bf16", seed=4)[0], "bf16")
    for hops, alpha in ((0, 0.1), (4, 1.0)):
        dQ, dK, dV = dl.diffuser_backward(Q, K, V, dO, g, hops, alpha)
        torch.cuda.synchronize()
        assert torch.equal(dV, dO) and not dQ.any() and not dK.any()
    a = dl.diffuser_backward(Q, K, V, dO, g, 5, 0.1)
    b = dl.diffuser_backward(Q, K, V, dO, g, 5, 0.1)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_backward_full_text_sampled_unit(dl):
    """The text workload at full size (2 x 12 units, n = 4096, E = 2,271,946, K = 5),
    bf16: one sampled (batch, head) unit of every gradient against the oracle's
    backward on that unit alone (the units are independent)."""
    import torch
    from sparse_long_sequence_gb300 import workloads
    w = workloads.TEXT
    g = dl.diffuser_build_graph(w.n, w.r, w.n_globals, rand_per_row=w.rand_per_row, seed=w.seed)
    o_ptr, o_col = oracle.token_graph(w.n, w.r, w.n_globals, w.rand_per_row, seed=w.seed)
    Q, K, V = synthetic.qkv(w.B, w.H, w.n, w.d, w.dtype, seed=w.seed)
    dO = synthetic.qkv(w.B, w.H, w.n, w.d, w.dtype, seed=w.seed + 1)[0]
    grads = dl.diffuser_backward(*(to_device(x, w.dtype) for x in (Q, K, V, dO)), g, w.hops, w.alpha)
    torch.cuda.synchronize()
    b, h = 1, 7
    ref = oracle.backward(*(oracle.widen(x[b, h], w.dtype) for x in (Q, K, V, dO)), o_ptr, o_col,
                          w.hops, w.alpha)
    for got, want in zip(grads, ref):
        check_grad(to_f64(got[b, h]), want, w.dtype)
