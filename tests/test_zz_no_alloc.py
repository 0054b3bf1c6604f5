"""The no-allocation forward (diffuser_forward_no_alloc), for callers that
cannot allocate device memory while the forward runs (serving loops whose
memory is fixed at start-up, frameworks that forbid cudaMalloc on their hot
path).  Called through the C ABI directly, on two calls in a row with new
inputs (the shared scratch array keeps the previous call's contents).  Each
output is checked against the fp64 oracle with the parity tolerances, and
against the regular entry point's output on the same CSR kernels.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

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


def call_no_alloc(dl, Q, K, V, g, hops, alpha, out, dtype_code):
    import torch
    lib = dl.raw_library()
    B, H, n, d = Q.shape
    return lib.diffuser_forward_no_alloc(
        ctypes.c_void_p(Q.data_ptr()), ctypes.c_void_p(K.data_ptr()), ctypes.c_void_p(V.data_ptr()),
        dtype_code, B, H, d, g.handle, hops, ctypes.c_float(alpha), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_no_alloc_matches_forward_twice(dl, dtype):
    import torch
    B, H, n = 2, 2, 700
    g = dl.diffuser_build_graph(n, 40, 4, rand_per_row=9, seed=0)
    o_ptr, o_col = oracle.token_graph(n, 40, 4, 9, seed=0)
    code = dl.DIFFUSER_DTYPE_BF16 if dtype == "bf16" else dl.DIFFUSER_DTYPE_FP32
    for call in range(2):
        Q, K, V = synthetic.qkv(B, H, n, 64, dtype, seed=100 + call)
        Qd, Kd, Vd = (to_device(x, dtype) for x in (Q, K, V))
        out = torch.empty_like(Vd)
        status = call_no_alloc(dl, Qd, Kd, Vd, g, 5, 0.1, out, code)
        torch.cuda.synchronize()
        assert status == 0, dl.diffuser_status_string(status)
        got = to_f64(out)
        ref = oracle.forward(*(oracle.widen(x, dtype) for x in (Q, K, V)), o_ptr, o_col, 5, 0.1,
                             nthreads=4)
        check_output(got, ref, dtype)
        # the regular entry point on the same inputs and kernels, within the same tolerance
        dl.diffuser_set_path(dl.DIFFUSER_PATH_CSR)
        try:
            regular = to_f64(dl.diffuser_forward(Qd, Kd, Vd, g, 5, 0.1))
        finally:
            dl.diffuser_set_path(dl.DIFFUSER_PATH_AUTO)
        check_output(got, regular, dtype)


def test_no_alloc_rejects_oversized_problem(dl):
    import torch
    n = 4096
    g = dl.diffuser_build_graph(n, 256, 16, rand_per_row=32, seed=0)
    Q = torch.zeros((2, 12, n, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(Q)
    before, _ = dl.diffuser_launch_count()
    status = call_no_alloc(dl, Q, Q, Q, g, 5, 0.1, out, dl.DIFFUSER_DTYPE_BF16)
    assert status == 7      # DIFFUSER_ERR_WORKSPACE: larger than the fixed array
    assert dl.diffuser_launch_count()[0] == before
    assert dl.diffuser_no_alloc_scratch_bytes() == 32 << 20
