"""Host model of the warp butterfly that the CSR score and backward kernels use
(`warp_transpose_sum32` in csrc/internal.h): every lane of a 32-lane warp holds
its share of 32 values; after the 5 exchange steps lane l must hold the sum over
the lanes of value l.  The model restates the kernel's steps (at step `off` a lane
keeps the half of its values whose index bit `off` matches its own lane bit, adds
its partner's copy of it) and checks them against the plain column sums, with
integers (exact) and with floats (the same additions in the same order every
time)."""
import numpy as np


def butterfly(v: np.ndarray) -> np.ndarray:
    """v[lane][k] -> out[lane], restating the kernel's exchange steps."""
    v = v.copy()
    off = 16
    while off >= 1:
        nxt = v.copy()
        for lane in range(32):
            partner = lane ^ off
            upper = (lane & off) != 0
            for k in range(off):
                send = v[partner][k + off] if not (partner & off) else v[partner][k]
                keep = v[lane][k] if not upper else v[lane][k + off]
                nxt[lane][k] = keep + send
        v = nxt
        off //= 2
    return v[:, 0]


def test_lane_l_gets_the_sum_of_value_l_exactly():
    rng = np.random.default_rng(0)
    v = rng.integers(-1000, 1000, size=(32, 32)).astype(np.int64)
    np.testing.assert_array_equal(butterfly(v), v.sum(axis=0))


def test_partner_sends_the_half_the_lane_keeps():
    # a single nonzero share travels to the lane of its value index and nowhere else
    for lane in (0, 5, 31):
        for k in (0, 17, 31):
            v = np.zeros((32, 32), dtype=np.int64)
            v[lane][k] = 1
            out = butterfly(v)
            assert out[k] == 1 and out.sum() == 1


def test_float_sums_are_repeatable_and_close():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((32, 32)).astype(np.float32)
    a, b = butterfly(v), butterfly(v)
    assert np.array_equal(a, b)
    np.testing.assert_allclose(a, v.astype(np.float64).sum(axis=0), rtol=1e-5, atol=1e-5)
