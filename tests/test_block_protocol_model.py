"""A host model of the block-sparse kernel's mbarrier protocol.

`block_kernel` (csrc/block_path.cu) runs one persistent CTA per SM over the
tiles dealt to it (two 64-token block rows each), a tile's allowed key blocks
taken in 128-key chunks through three pipeline slots.  Its roles:

  * the TMA warp loads the Q tile (two buffers) and each chunk's two K boxes;
    a slot's K stage is free again once its scores are written (full_S);
  * the Z warp (hops) loads each chunk's Z_k rows into the slot, counted as one
    arrival on full_P;
  * the score MMA warp writes S into the slot's TMEM buffer once the buffer is
    free (slot_free) and commits full_S, and empty_Q after a tile's last chunk;
  * the weights' MMA warp (hops) waits for key block 0's weights and the Z rows
    (full_P), then block 1's (full_P1), frees the slot and, after a tile's last
    chunk, hands the accumulator to the epilogue (acc_full / acc_empty);
  * 16 weight warps (4 lane quadrants x 4 key slices) read S: on the score pass
    they free the slot themselves and hand each row's maximum to their
    quadrant's epilogue warp at a tile's end; on the hops they write the weights
    (full_P, full_P1) and, on the first hop, hand over the row sums;
  * 4 epilogue warps take the hand-overs (xch_full / xch_empty, two buffers per
    quadrant) and, on the hops, the accumulator.

The roles' wait/arrive sequences are restated here step for step and played out
(tests/barrier_model.py): every role must finish for any list of tiles and chunk
counts, on the score pass, the first hop and the later hops, and no wait may
find its barrier two phases ahead.  It checks the protocol as designed; keeping
it in step with the kernel is a review duty whenever either changes.
"""
import random

import pytest

from tests.barrier_model import play

SLOTS, SOFT, SLICES, EPI = 3, 16, 4, 4


def roles_of(chunks, mode, slots=SLOTS, fp_count=SOFT + 1, acc_empty_count=EPI, k_backpressure=True):
    """The roles and barrier counts of one CTA whose tiles have `chunks[lt]`
    chunks each; mode is 'score', 'hop0' or 'hop'.  (k_backpressure=False drops
    the TMA warp's wait for a K stage to be consumed: a planted mistake.)"""
    hop, hop0 = mode != "score", mode == "hop0"
    counts = {}
    for s in range(2):
        counts[("fQ", s)] = counts[("eQ", s)] = 1
    for s in range(slots):
        counts[("fK", s)] = counts[("fS", s)] = 1
        counts[("fP", s)] = fp_count              # the weight warps + the Z copies' arrival
        counts[("fP1", s)] = SOFT
        counts[("free", s)] = 1 if hop else SOFT
    counts["accF"], counts["accE"] = 1, acc_empty_count
    for x in range(8):
        counts[("xf", x)], counts[("xe", x)] = SLICES, 1
    W = lambda bar, k: ("w", bar, k)
    A = lambda bar: ("a", bar)
    my = len(chunks)
    flat = [(lt, c == n - 1) for lt, n in enumerate(chunks) for c in range(n)]   # (tile, last chunk)
    total = len(flat)

    tma, zw, smma, pv = [], [], [], []
    g = 0
    for lt, n in enumerate(chunks):
        qb = lt & 1
        if lt >= 2:
            tma.append(W(("eQ", qb), lt // 2 - 1))
        tma.append(A(("fQ", qb)))
        for _ in range(n):
            b = g % slots
            if g >= slots and k_backpressure:
                tma.append(W(("fS", b), g // slots - 1))
            tma.append(A(("fK", b)))
            g += 1
    if hop:
        for g in range(total):
            b = g % slots
            if g >= slots:
                zw.append(W(("free", b), g // slots - 1))
            zw.append(A(("fP", b)))
    g = 0
    for lt, n in enumerate(chunks):
        qb = lt & 1
        smma.append(W(("fQ", qb), lt // 2))
        for c in range(n):
            b = g % slots
            smma.append(W(("fK", b), g // slots))
            if g >= slots:
                smma.append(W(("free", b), g // slots - 1))
            smma.append(A(("fS", b)))
            if c == n - 1:
                smma.append(A(("eQ", qb)))
            g += 1
    for s in range(slots):                          # drain before exit
        uses = (total - s + slots - 1) // slots
        if uses > 0:
            smma.append(W(("fS", s), uses - 1))
    for s in range(2):
        uses = (my - s + 1) // 2
        if uses > 0:
            smma.append(W(("eQ", s), uses - 1))
    if hop:
        g = 0
        for lt, n in enumerate(chunks):
            if lt >= 1:
                pv.append(W("accE", lt - 1))
            for c in range(n):
                sp = g % slots
                pv += [W(("fP", sp), g // slots), W(("fP1", sp), g // slots), A(("free", sp))]
                if c == n - 1:
                    pv.append(A("accF"))
                g += 1
        for s in range(slots):
            uses = (total - s + slots - 1) // slots
            if uses > 0:
                pv.append(W(("free", s), uses - 1))

    soft = []
    for w in range(SOFT):
        quad = (w + 4) & 3                          # warps 4..19: quadrant warp % 4
        seq = []

        def hand_over(lt):
            xb = quad * 2 + (lt & 1)
            if lt >= 2:
                seq.append(W(("xe", xb), lt // 2 - 1))
            seq.append(A(("xf", xb)))

        for g, (lt, last) in enumerate(flat):
            sb = g % slots
            seq.append(W(("fS", sb), g // slots))
            if not hop:
                seq.append(A(("free", sb)))
                if last:
                    hand_over(lt)
            else:
                seq += [A(("fP", sb)), A(("fP1", sb))]
                if hop0 and last:
                    hand_over(lt)
        soft.append(seq)
    epi = []
    for quad in range(EPI):
        seq = []
        for lt in range(my):
            xb = quad * 2 + (lt & 1)
            if not hop or hop0:
                seq += [W(("xf", xb), lt // 2), A(("xe", xb))]
            if hop:
                seq += [W("accF", lt), A("accE")]
        epi.append(seq)
    return [tma, zw, smma, pv] + soft + epi, counts


def outcome(chunks, mode, **kw):
    roles, counts = roles_of(chunks, mode, **kw)
    return play(roles, counts)


def completes(chunks, mode, **kw):
    return outcome(chunks, mode, **kw) == "done"


def tile_lists():
    rng = random.Random(7)
    lists = [[], [1], [6], [32], [6, 6], [32, 6, 6], [1, 1, 1, 1, 1], [6] * 7, [2, 32, 1, 6, 3]]
    lists += [[rng.randint(1, 32) for _ in range(rng.randint(1, 9))] for _ in range(12)]
    return lists


@pytest.mark.parametrize("mode", ["score", "hop0", "hop"])
def test_block_protocol_completes(mode):
    for chunks in tile_lists():
        assert completes(chunks, mode), chunks


@pytest.mark.parametrize("slots", [2, 4])
def test_block_protocol_completes_for_other_slot_counts(slots):
    for chunks in tile_lists()[:9]:
        for mode in ("score", "hop0", "hop"):
            assert completes(chunks, mode, slots=slots), (chunks, mode)


def test_model_detects_missing_arrivals():
    # not vacuous: full_P waiting for one arrival more than the weight warps and the
    # Z copies make, or the accumulator waiting for a fifth epilogue warp, stalls it
    chunks = [6, 32, 6]
    assert completes(chunks, "hop")
    assert not completes(chunks, "hop", fp_count=SOFT + 2)
    assert not completes(chunks, "hop", acc_empty_count=EPI + 1)
    assert completes(chunks, "score", fp_count=SOFT + 2)      # the score pass uses neither


def test_model_detects_a_producer_two_phases_ahead():
    # a TMA warp that refills a K stage without waiting for its scores lets full_K
    # complete two phases before the score MMA waits on it: the parity would alias
    assert outcome([6, 6], "score", k_backpressure=False) == "overrun"
    assert outcome([6, 6], "score") == "done"
