"""The device status word: a kernel whose bounded wait gives up records a code
in the graph's status word and its host mirror; after that every forward or
backward on the graph returns DIFFUSER_ERR_DEVICE without launching anything,
and the bench's completion check fails, until the word is reset.

No kernel is made to fail: the word is written from the host through the
library's test export (plain copies), exactly where a giving-up wait writes it.
"""
import numpy as np
import pytest

from sparse_long_sequence_gb300 import synthetic
from tests.helpers import to_device

pytestmark = pytest.mark.gpu

ERR_DEVICE = 6
TIMEOUT_CODE = 0x7100     # the code a bounded wait records when it gives up


@pytest.fixture(scope="module")
def dl():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_long_sequence_gb300 import binding
    return binding


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_status_word_stops_forwards_until_reset(dl, dtype):
    import torch
    g = dl.diffuser_build_graph(700, 40, 4, rand_per_row=9, seed=0)
    Q, K, V = (to_device(x, dtype) for x in synthetic.qkv(1, 2, 700, 64, dtype, seed=3))
    ref = dl.diffuser_forward(Q, K, V, g, 5, 0.1)
    torch.cuda.synchronize()
    assert dl.diffuser_graph_status(g) == 0

    dl.diffuser_graph_set_status(g, TIMEOUT_CODE)
    before, _ = dl.diffuser_launch_count()
    for call in (lambda: dl.diffuser_forward(Q, K, V, g, 5, 0.1),
                 lambda: dl.diffuser_backward(Q, K, V, V, g, 5, 0.1),
                 lambda: dl.diffuser_forward_no_alloc(Q, K, V, g, 5, 0.1, torch.empty_like(V))):
        with pytest.raises(dl.DiffuserError) as e:
            call()
        assert e.value.status == ERR_DEVICE
    assert dl.diffuser_launch_count()[0] == before, "a refused call launched kernels"

    # the bench's completion check sees it too
    import bench
    with pytest.raises(bench.BenchCheckFailed):
        bench.check_graph_status(dl, g, "a test")

    # reading with reset clears it; forwards run again and give the same bits
    assert dl.diffuser_graph_status(g, reset=True) == TIMEOUT_CODE
    assert dl.diffuser_graph_status(g) == 0
    again = dl.diffuser_forward(Q, K, V, g, 5, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(again, ref)


def test_status_word_is_per_graph(dl):
    import torch
    g1 = dl.diffuser_build_graph(300, 8, 2, rand_per_row=4, seed=0)
    g2 = dl.diffuser_build_graph(300, 8, 2, rand_per_row=4, seed=0)
    Q, K, V = (to_device(x, "bf16") for x in synthetic.qkv(1, 1, 300, 64, "bf16", seed=4))
    dl.diffuser_graph_set_status(g1, TIMEOUT_CODE)
    try:
        out = dl.diffuser_forward(Q, K, V, g2, 3, 0.1)     # the other graph is unaffected
        torch.cuda.synchronize()
        assert np.isfinite(out.float().cpu().numpy()).all()
        with pytest.raises(dl.DiffuserError):
            dl.diffuser_forward(Q, K, V, g1, 3, 0.1)
    finally:
        dl.diffuser_graph_status(g1, reset=True)
