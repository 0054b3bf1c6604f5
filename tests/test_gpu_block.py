"""The block-sparse tensor-core path (BigBird ITC block graphs of 64-token blocks,
bf16 I/O; "1.2.1 Static sparsity", sec 2 eq 13; "038 BigBird", sec 2) against the
oracle, against the general CSR path, and on its edge cases: ragged last block,
a tile whose second block row does not exist, an odd number of global blocks
(a tile mixing a global and a plain block row), wider windows, no random
blocks, hops 0 and 1, alpha 0 and 1."""
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


CASES = [  # graph arguments, B, H, hops, alpha
    (dict(n=1000, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=0), 2, 2, 5, 0.1),
    (dict(n=130, block=64, window_blocks=5, rand_blocks=3, global_blocks=0, seed=5), 1, 3, 5, 0.1),
    (dict(n=7, block=64, window_blocks=1, rand_blocks=0, global_blocks=1, seed=0), 2, 1, 3, 0.2),
    (dict(n=129, block=64, window_blocks=3, rand_blocks=1, global_blocks=1, seed=3), 1, 2, 5, 0.1),
    (dict(n=2048, block=64, window_blocks=3, rand_blocks=3, global_blocks=1, seed=7), 1, 2, 1, 0.0),
    (dict(n=1500, block=64, window_blocks=7, rand_blocks=0, global_blocks=3, seed=1), 2, 1, 4, 0.3),
    (dict(n=640, block=64, window_blocks=3, rand_blocks=8, global_blocks=2, seed=2 << 20), 3, 2, 5, 0.1),
]


def _ids(c):
    a = c[0]
    return "n%d_w%d_r%d_g%d_B%dH%dK%da%s" % (a["n"], a["window_blocks"], a["rand_blocks"],
                                             a["global_blocks"], c[1], c[2], c[3], c[4])


def test_block_path_selected(dl):
    g = dl.diffuser_build_block_graph(1000, 64, 3, 3, 2, seed=0)
    assert dl.diffuser_kernels_for(g, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_BLOCK
    assert dl.diffuser_kernels_for(g, dl.DIFFUSER_DTYPE_FP32) == dl.DIFFUSER_KERNELS_CSR
    g16 = dl.diffuser_build_block_graph(1000, 16, 3, 3, 2, seed=0)
    assert dl.diffuser_kernels_for(g16, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_CSR
    gt = dl.diffuser_build_graph(1000, 64, 4, rand_per_row=8)
    assert dl.diffuser_kernels_for(gt, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_BAND
    dl.diffuser_set_path(dl.DIFFUSER_PATH_CSR)
    try:
        assert dl.diffuser_kernels_for(g, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_CSR
    finally:
        dl.diffuser_set_path(dl.DIFFUSER_PATH_AUTO)


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_block_path_parity(dl, case):
    import torch
    args, B, H, hops, alpha = case
    g = dl.diffuser_build_block_graph(**args)
    assert dl.diffuser_kernels_for(g, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_BLOCK
    o_ptr, o_col = oracle.block_graph(**args)
    Q, K, V = synthetic.qkv(B, H, args["n"], 64, "bf16", seed=args["n"] + hops)
    Qd, Kd, Vd = (to_device(x, "bf16") for x in (Q, K, V))
    out = dl.diffuser_forward(Qd, Kd, Vd, g, hops, alpha)
    torch.cuda.synchronize()
    assert dl.diffuser_graph_status(g) == 0
    ref = oracle.forward(*(oracle.widen(x, "bf16") for x in (Q, K, V)), o_ptr, o_col, hops, alpha,
                         nthreads=4)
    got = to_f64(out)
    check_output(got, ref, "bf16")
    # the general CSR path on the same inputs: both round fp32-accurate values to bf16
    dl.diffuser_set_path(dl.DIFFUSER_PATH_CSR)
    try:
        csr = to_f64(dl.diffuser_forward(Qd, Kd, Vd, g, hops, alpha))
    finally:
        dl.diffuser_set_path(dl.DIFFUSER_PATH_AUTO)
    assert np.abs(got - csr).max() <= 2 ** -7 * np.abs(ref).max()


def test_block_path_special_cases(dl):
    import torch
    args = dict(n=1000, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=0)
    g = dl.diffuser_build_block_graph(**args)
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(2, 2, 1000, 64, "bf16", seed=4))
    for hops, alpha in ((0, 0.1), (5, 1.0)):
        out = dl.diffuser_forward(Q, K, V, g, hops, alpha)
        torch.cuda.synchronize()
        assert torch.equal(out, V)
    Vc = torch.full_like(V, 0.25)
    outc = dl.diffuser_forward(Q, K, Vc, g, 5, 0.1)          # rows of A sum to one
    torch.cuda.synchronize()
    assert float((outc.float() - 0.25).abs().max()) <= 0.25 * 2 ** -8
    a = dl.diffuser_forward(Q, K, V, g, 5, 0.1)
    b = dl.diffuser_forward(Q, K, V, g, 5, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(a, b)                                  # fixed summation order
    assert dl.diffuser_graph_status(g) == 0


def test_block_path_full_bigbird_workload_selected(dl):
    w = workloads.BIGBIRD
    g = dl.diffuser_build_block_graph(**w.graph_args())
    assert dl.diffuser_kernels_for(g, dl.DIFFUSER_DTYPE_BF16) == dl.DIFFUSER_KERNELS_BLOCK


@pytest.mark.parametrize("pinned_out", [True, False], ids=["pinned_out", "pageable_out"])
def test_block_path_host_buffers(dl, pinned_out):
    # the end-to-end entry point on the block path: Q and K upload side by side, V under
    # the score pass, a pinned mapped `out` written in place (a pageable one copied back);
    # three calls so that the pinned sequence is also replayed as a captured graph
    import torch
    args = dict(n=1000, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=0)
    g = dl.diffuser_build_block_graph(**args)
    Q, K, V = synthetic.qkv(2, 2, 1000, 64, "bf16", seed=9)
    Qh, Kh, Vh = (torch.from_numpy(x).view(torch.bfloat16).pin_memory() for x in (Q, K, V))
    out = torch.empty_like(Vh).pin_memory() if pinned_out else torch.empty(Vh.shape, dtype=Vh.dtype)
    ws = dl.alloc_workspace(dl.diffuser_host_workspace_size(g, 2, 2, 64, dl.DIFFUSER_DTYPE_BF16))
    ref_dev = dl.diffuser_forward(Qh.cuda(), Kh.cuda(), Vh.cuda(), g, 5, 0.1)
    torch.cuda.synchronize()
    for _ in range(3):
        out.zero_()
        dl.diffuser_forward_host(Qh, Kh, Vh, g, 5, 0.1, out, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_dev.cpu())
    assert dl.diffuser_graph_status(g) == 0


def test_block_dealing_table_and_snake_order_agree(dl):
    # The tiles of a launch go to the CTAs through a deal table (heaviest first to the
    # least-loaded CTA), built on the first forward with a given B*H outside stream
    # capture; a forward issued while the caller's stream is capturing deals them in
    # snake order instead.  Each tile is computed by one CTA in a fixed order either
    # way, so the two outputs agree bit for bit.
    import torch
    args = dict(n=4096, block=64, window_blocks=3, rand_blocks=3, global_blocks=2, seed=0)
    g = dl.diffuser_build_block_graph(**args)
    # a plain forward with another B*H first: the kernels' one-time set-up happens
    # outside the capture below, and no table exists yet for B*H = 12
    Q1, K1, V1 = (to_device(x, "bf16") for x in synthetic.qkv(1, 1, 4096, 64, "bf16", seed=10))
    dl.diffuser_forward(Q1, K1, V1, g, 5, 0.1)
    torch.cuda.synchronize()
    B, H = 3, 4        # 12 global block-row tiles of 32 chunks among 372 of 6: the dealings differ
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(B, H, 4096, 64, "bf16", seed=11))
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
