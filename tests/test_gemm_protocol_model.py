"""A host model of the projection GEMM's mbarrier protocol.

`proj_gemm_kernel` (csrc/layer_gemm.cu) runs one persistent CTA per SM over its
128 x 256 output tiles: the TMA warp fills a ring of K-step stages (full /
empty), the MMA warp accumulates each tile into one of two TMEM accumulators
(acc_full / acc_empty, the latter counting the 4 epilogue warps) and frees each
stage by a commit, and the epilogue warps read an accumulator while the next
tile accumulates into the other.  The roles' wait/arrive sequences are restated
here and played out (tests/barrier_model.py): every role must finish for any
tile and K-step count, and no wait may find its barrier two phases ahead.  It
checks the protocol as designed; keeping it in step with the kernel is a review
duty whenever either changes.
"""
import pytest

from tests.barrier_model import play

STAGES, EPI = 4, 4


def outcome(my, k_blocks, stages=STAGES, acc_empty_count=EPI, ring_backpressure=True):
    counts = {("full", s): 1 for s in range(stages)}
    counts.update({("empty", s): 1 for s in range(stages)})
    for b in range(2):
        counts[("accF", b)], counts[("accE", b)] = 1, acc_empty_count
    W = lambda bar, k: ("w", bar, k)
    A = lambda bar: ("a", bar)
    tma, mma = [], []
    g = 0
    for lt in range(my):
        for _ in range(k_blocks):
            s = g % stages
            if g >= stages and ring_backpressure:
                tma.append(W(("empty", s), g // stages - 1))
            tma.append(A(("full", s)))
            g += 1
    g = 0
    for lt in range(my):
        buf = lt & 1
        if lt >= 2:
            mma.append(W(("accE", buf), lt // 2 - 1))
        for _ in range(k_blocks):
            s = g % stages
            mma += [W(("full", s), g // stages), A(("empty", s))]
            g += 1
        mma.append(A(("accF", buf)))
    for s in range(stages):                 # drain before exit
        uses = (g - s + stages - 1) // stages
        if uses > 0:
            mma.append(W(("empty", s), uses - 1))
    epi = [[x for lt in range(my) for x in (W(("accF", lt & 1), lt // 2), A(("accE", lt & 1)))]
           for _ in range(EPI)]
    return play([tma, mma] + epi, counts)


@pytest.mark.parametrize("k_blocks", [1, 2, 3, 4, 5, 12, 13])
def test_gemm_protocol_completes(k_blocks):
    for my in range(0, 8):
        assert outcome(my, k_blocks) == "done", my
        assert outcome(my, k_blocks, stages=2) == "done", my


def test_model_detects_planted_mistakes():
    assert outcome(4, 12) == "done"
    assert outcome(4, 12, acc_empty_count=EPI + 1) == "stalled"         # a fifth epilogue warp awaited
    assert outcome(4, 12, ring_backpressure=False) == "overrun"         # stages refilled unread
