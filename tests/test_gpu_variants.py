"""Graph variants on the device: the uniform-spaced extras ("w uni.", Diffuser
notes sec 4.5, Tab S.7) bit-exact against the oracle and through the forward,
and the forward with one graph per head (Diffuser notes sec 2.2) against the
oracle's per-head forward."""
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


UNIFORM_CASES = [  # n, r, G, R, causal
    (16, 1, [], 4, False), (300, 8, [0, 1, 2], 5, False), (777, 13, [0, 100, 401, 776], 9, True),
    (4096, 256, list(range(16)), 32, False), (1000, 40, [3], 1, False), (513, 0, [], 7, True),
]


@pytest.mark.parametrize("case", UNIFORM_CASES)
def test_uniform_graph_bit_exact(dl, case):
    n, r, G, R, causal = case
    g = dl.diffuser_build_uniform_graph(n, r, len(G), global_idx=G or None, positions_per_row=R,
                                        causal=causal)
    row_ptr, col = dl.diffuser_graph_copy_csr(g)
    o_ptr, o_col = oracle.uniform_graph(n, r, len(G), R, globals_idx=G or None, causal=causal)
    np.testing.assert_array_equal(row_ptr, o_ptr)
    np.testing.assert_array_equal(col, o_col)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_uniform_forward(dl, dtype, causal):
    import torch
    n, r, gn, R = 900, 40, 4, 16
    g = dl.diffuser_build_uniform_graph(n, r, gn, positions_per_row=R, causal=causal)
    o_ptr, o_col = oracle.uniform_graph(n, r, gn, R, causal=causal)
    Q, K, V = synthetic.qkv(2, 2, n, 64, dtype, seed=9)
    out = dl.diffuser_forward(*(to_device(x, dtype) for x in (Q, K, V)), g, 5, 0.1)
    torch.cuda.synchronize()
    ref = oracle.forward(*(oracle.widen(x, dtype) for x in (Q, K, V)), o_ptr, o_col, 5, 0.1,
                         nthreads=4)
    check_output(to_f64(out), ref, dtype)


def head_graphs(dl, n):
    """Three heads, three graphs: different seeds, a causal one and a uniform one."""
    return [
        (dl.diffuser_build_graph(n, 24, 3, rand_per_row=6, seed=1 << 20),
         oracle.token_graph(n, 24, 3, 6, seed=1 << 20)),
        (dl.diffuser_build_causal_graph(n, 24, 3, rand_per_row=6, seed=2 << 20),
         oracle.token_graph(n, 24, 3, 6, seed=2 << 20, causal=True)),
        (dl.diffuser_build_uniform_graph(n, 24, 3, positions_per_row=6),
         oracle.uniform_graph(n, 24, 3, 6)),
    ]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B", [1, 2])
def test_per_head_forward(dl, dtype, B):
    import torch
    n, H = 600, 3
    hg = head_graphs(dl, n)
    Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=11)
    Qd, Kd, Vd = (to_device(x, dtype) for x in (Q, K, V))
    out = dl.diffuser_forward_per_head(Qd, Kd, Vd, [g for g, _ in hg], 5, 0.1)
    torch.cuda.synchronize()
    ref = oracle.forward_per_head(*(oracle.widen(x, dtype) for x in (Q, K, V)),
                                  [o for _, o in hg], 5, 0.1, nthreads=4)
    check_output(to_f64(out), ref, dtype)
    # the same heads through the shared-graph entry point, one head at a time
    for h, (g, _) in enumerate(hg):
        one = dl.diffuser_forward(Qd[:, h:h + 1].contiguous(), Kd[:, h:h + 1].contiguous(),
                                  Vd[:, h:h + 1].contiguous(), g, 5, 0.1)
        torch.cuda.synchronize()
        assert torch.equal(one[:, 0], out[:, h])


def test_per_head_forward_special_cases(dl):
    import torch
    n = 300
    hg = head_graphs(dl, n)
    graphs = [g for g, _ in hg]
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(2, 3, n, 64, "bf16", seed=12))
    out = dl.diffuser_forward_per_head(Q, K, V, graphs, 0, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(out, V)                                     # hops = 0 returns V
    out = dl.diffuser_forward_per_head(Q, K, V, graphs, 3, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(out, V)                                     # alpha = 1 returns V
    other = dl.diffuser_build_graph(n + 1, 8, 0)
    with pytest.raises(dl.DiffuserError):                          # graphs must share n
        dl.diffuser_forward_per_head(Q, K, V, graphs[:2] + [other], 3, 0.1)
