"""The projections around the diffusion module on the tcgen05 GEMMs (Diffuser
notes sec 2.1 and sec 2.4, Fig S.3) against float64 products and the oracle's
module.

Tolerances, from the arithmetic:
  * each projection output element: |got - ref| <= 2^-8 |ref| + 2^-14 sum_c |x_c w_c|
    (its one bf16 rounding, at most half an ulp = 2^-8 of the value for 8
    significant bits, plus fp32 accumulation of K <= 1024 products, at most
    K 2^-24 <= 2^-14 of the sum of their magnitudes);
  * the module's output: per row, max |got - ref| / max |ref| <= 2^-7, against the
    oracle with bf16 interfaces (Q, K, V, Z, Y each rounded once): the output's
    own rounding (2^-8) plus the elements of Q, K, V and Z whose fp32 and float64
    values round to neighbouring bf16 values (one ulp each, a few percent of the
    elements, adding ~2^-7 sqrt(fraction) relative over the 64 H-term sums).
"""
import numpy as np
import pytest

import oracle
from sparse_long_sequence_gb300 import synthetic
from tests.helpers import row_relative_error, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dl():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_long_sequence_gb300 import binding
    return binding


def widen(bits):
    return oracle.widen(bits, "bf16")


def check_product(got, ref, absref):
    assert np.all(np.isfinite(got))
    excess = np.abs(got - ref) - (2 ** -8 * np.abs(ref) + 2 ** -14 * absref)
    assert excess.max() <= 0, f"worst excess {excess.max():.3e}"


SHAPES = [(2, 300, 256, 2), (1, 128, 768, 12), (3, 77, 200, 3), (1, 1000, 512, 8)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dn%dD%dH%d" % s)
def test_qkv_projection_elementwise(dl, shape):
    import torch
    B, n, D, H = shape
    X, Wqkv, _ = synthetic.layer_inputs(B, n, D, H, seed=n)
    Q, K, V = dl.diffuser_qkv_projection(to_device(X, "bf16"), to_device(Wqkv, "bf16"), H)
    torch.cuda.synchronize()
    x, w = widen(X), widen(Wqkv)                                   # [B][n][D], [3 H 64][D]
    ref = np.einsum("bnc,jc->bnj", x, w).reshape(B, n, 3, H, 64).transpose(2, 0, 3, 1, 4)
    absref = np.einsum("bnc,jc->bnj", np.abs(x), np.abs(w)).reshape(B, n, 3, H, 64).transpose(2, 0, 3, 1, 4)
    for s, got in enumerate((Q, K, V)):
        check_product(to_f64(got), ref[s], absref[s])


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dn%dD%dH%d" % s)
def test_output_projection_elementwise(dl, shape):
    import torch
    B, n, D, H = shape
    _, _, Wo = synthetic.layer_inputs(B, n, D, H, seed=n + 1)
    Z = synthetic.qkv(B, H, n, 64, "bf16", seed=n + 2)[0]
    Y = dl.diffuser_output_projection(to_device(Z, "bf16"), to_device(Wo, "bf16"))
    torch.cuda.synchronize()
    z, w = widen(Z), widen(Wo)
    heads = z.transpose(0, 2, 1, 3).reshape(B, n, H * 64)          # concatenation
    check_product(to_f64(Y), heads @ w.T, np.abs(heads) @ np.abs(w).T)


def oracle_module(X, Wqkv, Wo, H, row_ptr, col, hops, alpha):
    x, wqkv, wo = widen(X), widen(Wqkv), widen(Wo)
    D = x.shape[-1]
    per = wqkv.reshape(3, H, 64, D).transpose(0, 1, 3, 2)         # [3][H][D][64]
    return oracle.layer_forward(x, per[0], per[1], per[2], wo.T, row_ptr, col, hops, alpha,
                                bf16_interfaces=True)


@pytest.mark.parametrize("graph", ["token", "block", "causal"])
def test_layer_forward_against_oracle(dl, graph):
    import torch
    B, D, H, hops, alpha = 2, 256, 4, 5, 0.1
    if graph == "block":
        n = 1000
        g = dl.diffuser_build_block_graph(n, 64, 3, 3, 2, seed=0)
        o = oracle.block_graph(n, 64, 3, 3, 2, seed=0)
    else:
        n = 600
        build = dl.diffuser_build_causal_graph if graph == "causal" else dl.diffuser_build_graph
        g = build(n, 40, 4, rand_per_row=9, seed=0)
        o = oracle.token_graph(n, 40, 4, 9, seed=0, causal=graph == "causal")
    X, Wqkv, Wo = synthetic.layer_inputs(B, n, D, H, seed=7)
    Xd, Wqd, Wod = (to_device(t, "bf16") for t in (X, Wqkv, Wo))
    Y = dl.diffuser_layer_forward(Xd, Wqd, Wod, g, H, hops, alpha)
    torch.cuda.synchronize()
    assert dl.diffuser_graph_status(g) == 0
    ref = oracle_module(X, Wqkv, Wo, H, *o, hops, alpha)
    got = to_f64(Y)
    assert np.all(np.isfinite(got))
    err = row_relative_error(got, ref)
    assert err <= 2 ** -7, f"row-relative error {err:.3e}"
    # the same three stages called one by one give the same bits
    Q, K, V = dl.diffuser_qkv_projection(Xd, Wqd, H)
    Z = dl.diffuser_forward(Q, K, V, g, hops, alpha)
    Y2 = dl.diffuser_output_projection(Z, Wod)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2)


def test_projection_argument_checks(dl):
    import torch
    X = torch.zeros((1, 64, 100), dtype=torch.bfloat16, device="cuda")   # D = 100 is not a multiple of 8
    W = torch.zeros((3 * 64, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dl.DiffuserError):
        dl.diffuser_qkv_projection(X, W, 1)
    X = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((3 * 64, 128), dtype=torch.bfloat16, device="cuda")
    before, _ = dl.diffuser_launch_count()
    with pytest.raises(dl.DiffuserError):                              # an output overlapping the input
        dl.diffuser_qkv_projection(X, W, 1, Q=X.view(-1)[: 64 * 64].view(1, 1, 64, 64))
    assert dl.diffuser_launch_count()[0] == before
    assert dl.diffuser_projection_status() == 0
