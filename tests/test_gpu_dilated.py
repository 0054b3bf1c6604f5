"""Dilated graph on the device: bit-exact CSR
against the oracle, and the forward on the CSR path."""
import numpy as np
import pytest

import oracle
from sparse_long_sequence_gb300 import synthetic
from tests.helpers import check_output, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_long_sequence_gb300 import binding
    return binding


CASES = [  # n, r, dilation, G, R, seed, causal
    (40, 2, 3, [], 0, 0, False), (1, 3, 2, [0], 5, 0, False), (300, 8, 3, [0, 1, 2], 5, 0, False),
    (777, 13, 5, [0, 100, 401, 776], 9, 2 ** 63 + 11, True), (4096, 64, 4, list(range(16)), 32, 1, False),
    (500, 7, 1, [3], 6, 2, False),
]


@pytest.mark.parametrize("case", CASES)
def test_dilated_graph_bit_exact(dl, case):
    n, r, dil, G, R, seed, causal = case
    g = dl.diffuser_build_dilated_graph(n, r, dil, len(G), global_idx=G or None, rand_per_row=R,
                                        seed=seed, causal=causal)
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    o_ptr, o_col = oracle.dilated_graph(n, r, dil, len(G), R, seed=seed, globals_idx=G or None,
                                        causal=causal)
    np.testing.assert_array_equal(row_ptr, o_ptr)
    np.testing.assert_array_equal(col, o_col)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_dilated_forward(dl, dtype):
    import torch
    n = 700
    g = dl.diffuser_build_dilated_graph(n, 16, 3, 4, rand_per_row=8, seed=2)
    o_ptr, o_col = oracle.dilated_graph(n, 16, 3, 4, 8, seed=2)
    Q, K, V = synthetic.qkv(1, 3, n, 64, dtype, seed=5)
    out = dl.diffuser_forward(*(to_device(x, dtype) for x in (Q, K, V)), g, 5, 0.1)
    torch.cuda.synchronize()
    ref = oracle.forward(*(oracle.widen(x, dtype) for x in (Q, K, V)), o_ptr, o_col, 5, 0.1, nthreads=3)
    check_output(to_f64(out), ref, dtype)
