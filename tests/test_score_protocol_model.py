"""A host model of the window score kernel's mbarrier protocol.

`score_band_tc_kernel` (csrc/band_score.cu) runs one persistent CTA per SM over
the tiles blockIdx.x, blockIdx.x + gridDim.x, ...  Its roles hand the work to
one another through mbarriers and, between the two warps that share a TMEM lane
quadrant, named barriers:

  * warp 0 loads the Q tile (two buffers) and the 64-key K chunks (a ring);
  * warp 1 issues the score MMAs into a ring of TMEM score buffers, the
    out-of-window globals' scores at tile start and the global rows' scores on
    the tile's own two key chunks;
  * warp 2 stages the globals' q and k rows (two buffers);
  * eight row warps read each score buffer, release it, and at the tile's end
    (the transition) read the globals' scores; the two warps of quadrant 0 also
    read the global rows' scores.  With weight images (`kImages`) every chunk is
    read twice, the second pass between two pair barriers per chunk.

A mistake in the protocol shows up on the GPU as a wait that never ends, so the
roles' wait/arrive sequences are restated here step for step and played out with
the barriers' arrival counts and phases (tests/barrier_model.py): for any tile
count, chunk count, with and without globals and images, every role must finish,
and no wait may find its barrier two phases ahead (the parity would alias).  It
checks the protocol as designed; keeping it in step with the kernel is a review
duty whenever either changes.
"""
import pytest

from tests.barrier_model import play

K_STAGES, S_BUFS = 8, 5        # the kernel's K ring and TMEM score buffers
ROW_WARPS = 8                  # 4 lane quadrants x 2 column halves


def plan(n, r, causal):
    """(c0, nc, tiles): the chunk holding the tile's own first key, the 64-key
    chunks of a tile (even), and the 128-row tiles, as band_plan sets them."""
    r64 = (r + 63) // 64 * 64
    up = 0 if causal else r
    nc = (r64 + 128 + up + 63) // 64
    nc += nc & 1
    return r64 // 64, nc, (n + 127) // 128


def my_tiles(total, G, b):
    return (total - 1 - b) // G + 1 if b < total else 0


def simulate(my, nc, c0, has_g, images, k_stages=K_STAGES, s_bufs=S_BUFS, es_count=ROW_WARPS, egr_count=2):
    """Play the roles' waits and arrivals for one CTA with `my` tiles; True if
    every role finishes under every schedule tried, with no wait overtaken by
    two phases of its barrier."""
    per_tile = 2 * nc if images else nc
    counts = {}
    for s in range(2):
        counts[("fQ", s)] = counts[("eQ", s)] = counts[("fG", s)] = counts[("eG", s)] = 1
    for s in range(k_stages):
        counts[("fK", s)] = counts[("eK", s)] = 1
    for b in range(s_bufs):
        counts[("fS", b)] = 1
        counts[("eS", b)] = es_count        # lane 0 of each row warp
    counts["fGR"] = 1
    counts["eGR"] = egr_count               # the two warps of quadrant 0 (64 threads in the kernel)
    for q in range(4):
        counts[("pair", q)] = 2             # the named barrier of a quadrant's two warps
    W = lambda bar, k: ("w", bar, k)
    A = lambda bar: ("a", bar)

    tma, mma, gld = [], [], []
    for lt in range(my):
        qb = lt & 1
        if lt >= 2:
            tma.append(W(("eQ", qb), lt // 2 - 1))
        tma.append(A(("fQ", qb)))
        for it in range(per_tile):
            gi = lt * per_tile + it
            s = gi % k_stages
            if gi >= k_stages:
                tma.append(W(("eK", s), gi // k_stages - 1))
            tma.append(A(("fK", s)))
    for lt in range(my):
        qb = lt & 1
        mma.append(W(("fQ", qb), lt // 2))
        if has_g:
            mma.append(W(("fG", qb), lt // 2))
        for it in range(per_tile):
            gi = lt * per_tile + it
            s, b = gi % k_stages, gi % s_bufs
            mma.append(W(("fK", s), gi // k_stages))
            if gi >= s_bufs:
                mma.append(W(("eS", b), gi // s_bufs - 1))
            h = it - c0
            if has_g and h in (0, 1):
                if h == 0 and lt >= 1:
                    mma.append(W("eGR", lt - 1))
                if h == 1:
                    mma += [A("fGR"), A(("eG", qb))]
            mma += [A(("eK", s)), A(("fS", b))]
        mma.append(A(("eQ", qb)))
    total = my * per_tile                   # drain the commit arrivals before exit
    for s in range(k_stages):
        uses = (total - s + k_stages - 1) // k_stages
        if uses > 0:
            mma.append(W(("eK", s), uses - 1))
    for s in range(2):
        uses = (my - s + 1) // 2
        if uses > 0:
            mma.append(W(("eQ", s), uses - 1))
            if has_g:
                mma.append(W(("eG", s), uses - 1))
    if has_g:
        for lt in range(my):
            qb = lt & 1
            if lt >= 2:
                gld.append(W(("eG", qb), lt // 2 - 1))
            gld.append(A(("fG", qb)))

    rows = []
    for rw in range(ROW_WARPS):
        quad = (rw + 4) & 3                 # warps 4..11: quadrant warp % 4
        seq, syncs = [], [0]

        def pair():
            seq.extend([A(("pair", quad)), W(("pair", quad), syncs[0])])
            syncs[0] += 1

        def transition(lt):
            pair()
            if has_g and quad == 0:
                seq.extend([W("fGR", lt), A("eGR")])
            pair()

        for lt in range(my):
            for it in range(per_tile):
                gi = lt * per_tile + it
                b = gi % s_bufs
                if images and it == nc:
                    transition(lt)
                seq.extend([W(("fS", b), gi // s_bufs), A(("eS", b))])
                if it >= nc:                # second pass: stage, then hand the chunk's image to the copy
                    pair()
                    pair()
            if not images:
                transition(lt)
            pair()                          # the row sums' exchange at the tile's end
            pair()
        rows.append(seq)

    return play([tma, mma, gld] + rows, counts) == "done"


CASES = [(4096, 256, False), (4096, 256, True), (1024, 32, False), (1024, 32, True), (16384, 256, False),
         (300, 8, False), (200, 300, False), (640, 640, True), (129, 64, False)]


@pytest.mark.parametrize("n,r,causal", CASES)
def test_every_tile_dealt_once(n, r, causal):
    _, _, tiles = plan(n, r, causal)
    for units in (1, 3, 24):
        total = units * tiles
        for G in (152, 7, 1):
            dealt = sorted(b + lt * G for b in range(min(G, total)) for lt in range(my_tiles(total, G, b)))
            assert dealt == list(range(total))


@pytest.mark.parametrize("images", [False, True], ids=["maxima", "images"])
@pytest.mark.parametrize("n,r,causal", CASES)
def test_score_protocol_completes(n, r, causal, images):
    c0, nc, _ = plan(n, r, causal)
    assert c0 + 1 < nc                      # every tile meets its own two key chunks
    for my in (0, 1, 2, 3, 5, 6, 14):
        for has_g in (False, True):
            assert simulate(my, nc, c0, has_g, images), (my, has_g)


@pytest.mark.parametrize("k_stages,s_bufs", [(8, 2), (8, 3), (10, 5), (12, 5), (4, 5)])
def test_score_protocol_completes_for_other_ring_depths(k_stages, s_bufs):
    for n, r, causal in CASES[:4]:
        c0, nc, _ = plan(n, r, causal)
        for my in (1, 2, 5):
            for images in (False, True):
                assert simulate(my, nc, c0, True, images, k_stages=k_stages, s_bufs=s_bufs)


def test_model_detects_missing_arrivals():
    # not vacuous: a score buffer that waits for a ninth row warp, or a global-row
    # hand-off that waits for a third warp, stalls the CTA
    c0, nc, _ = plan(4096, 256, False)
    assert simulate(3, nc, c0, True, False)
    assert not simulate(3, nc, c0, True, False, es_count=ROW_WARPS + 1)
    assert not simulate(3, nc, c0, True, False, egr_count=3)
    assert simulate(3, nc, c0, False, False, egr_count=3)      # no globals: the hand-off is unused
