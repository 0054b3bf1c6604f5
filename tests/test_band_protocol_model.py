"""A host model of the band hop kernel's tile order and mbarrier protocol.

The kernel's CTAs walk per-tile ranges of 128-key chunks [c_lo, c_hi] in a
table order, and six roles (Q/K loads, Z_k loads, score MMAs, weight MMAs,
softmax warps, epilogue) hand every chunk and tile to one another through
mbarriers.  A mistake in either shows up on the GPU as a wait that never ends,
so both are restated here in Python, step for step with `chunk_range`,
`tile_position`, `cta_tile_count` and `cta_tile` in csrc/band_hop.cu and the
roles' wait/arrive sequences, and checked on the CPU:

  * every (unit, tile) is dealt to exactly one CTA, and each tile's chunk range
    covers every key of each of its rows' windows (bidirectional [i - r, i + r]
    or causal [i - r, i]);
  * the roles' waits and arrivals, played out with the barriers' arrival counts
    and phases (tests/barrier_model.py), run to completion (no deadlock) for any
    tile list, with and without globals, on the first hop (row-sum hand-off) and
    later ones, and no wait finds its barrier two phases ahead (where the
    parity would alias).

It checks the protocol as designed; keeping it in step with the kernel is a
review duty whenever either changes.
"""
import pytest

from tests.barrier_model import play

CK, TR = 128, 128          # keys per chunk, rows per tile


def plan(n, r, causal):
    r64 = (r + 63) // 64 * 64
    up = 0 if causal else r
    chunks64 = (r64 + TR + up + 63) // 64
    chunks64 += chunks64 & 1
    return r64, chunks64 // 2, (n + TR - 1) // TR


def chunk_range(n, r64, nc, i0):
    below = r64 - i0 - (CK - 1)
    c_lo = (below + CK - 1) // CK if below > 0 else 0
    last = (n - (i0 - r64) - 1) // CK
    return c_lo, min(last, nc - 1)


def interior(n, r64, nc, tiles):
    tl = (r64 - (CK - 1) + CK - 1) // CK if r64 > CK - 1 else 0
    rnum = n + r64 - 1 - CK * (nc - 1)
    tr = min(rnum // CK if rnum >= 0 else -1, tiles - 1)
    return tl, tr


def tile_position(n, r64, nc, tiles, p):
    tl, tr = interior(n, r64, nc, tiles)
    if tl > tr:
        return p
    ni = tr - tl + 1
    if p < ni:
        return tl + p

    def count(t):
        lo, hi = chunk_range(n, r64, nc, t * TR)
        return hi - lo
    li, ri, q = tl - 1, tr + 1, p - ni
    while True:
        has_l, has_r = li >= 0, ri < tiles
        take_l = has_l and (not has_r or count(li) >= count(ri))
        t = li if take_l else ri
        if q == 0 or (not has_l and not has_r):
            return t
        if take_l:
            li -= 1
        else:
            ri += 1
        q -= 1


def cta_tiles(n, r, causal, units, G, b):
    """(u, t, c_lo, c_hi) of CTA b's tiles in its order, as cta_tile deals them."""
    r64, nc, tiles = plan(n, r, causal)
    T = units * tiles
    R, rem = T // G, T % G
    my = R + ((1 if b < rem else 0) if R % 2 == 0 else (1 if b >= G - rem else 0))
    tl, tr = interior(n, r64, nc, tiles)
    ni = tr - tl + 1 if tl <= tr else 0
    out = []
    for lt in range(my):
        k = lt * G + ((G - 1 - b) if lt & 1 else b)
        if k < units * ni:
            u, t = k // ni, tl + k % ni
        else:
            k2 = k - units * ni
            u, t = k2 % units, tile_position(n, r64, nc, tiles, ni + k2 // units)
        lo, hi = chunk_range(n, r64, nc, t * TR)
        out.append((u, t, lo, hi))
    return out


def simulate(tiles, c0, r64, has_g, hop0, slots=2, fp_arrivals=2):
    """Play the roles' waits and arrivals; True if every role finishes under every
    schedule tried, with no wait overtaken by two phases of its barrier."""
    counts = {}
    for s in range(2):
        counts[("fQ", s)] = counts[("eQ", s)] = 1
        counts[("xf", s)] = counts[("xe", s)] = 1
    for s in range(slots):
        counts[("fK", s)] = counts[("fS", s)] = counts[("pd", s)] = 1
        counts[("fP", s)] = fp_arrivals             # the weight warps + the Z_k copy
    for nm in ("accF", "accE", "gE", "fG", "eG", "eGC"):
        counts[nm] = 1
    counts["fGC"] = 2
    W = lambda bar, k: ("w", bar, k)   # wait for phase completion number k
    A = lambda bar: ("a", bar)         # arrive once
    kq, zp, si, pv, ep, sw = [], [], [], [], [], []
    g = 0
    for lt, (_, _, lo, hi) in enumerate(tiles):
        qb = lt & 1
        glob_last = c0 + 1 if (r64 % CK != 0 and c0 + 1 <= hi) else c0
        if lt >= 2:
            kq.append(W(("eQ", qb), lt // 2 - 1))
        kq.append(A(("fQ", qb)))
        if has_g:
            if lt >= 1:
                zp.append(W("eG", lt - 1))
            zp.append(A("fG"))
        si.append(W(("fQ", qb), lt // 2))
        if lt >= 1:
            pv.append(W("accE", lt - 1))
        if has_g:
            pv.append(W("fGC", lt))
            pv.append(A("eGC"))
        for c in range(lo, hi + 1):
            b = g % slots
            if g >= slots:
                kq.append(W(("fS", b), g // slots - 1))
                zp.append(W(("pd", b), g // slots - 1))
            kq.append(A(("fK", b)))
            zp.append(A(("fP", b)))
            si.append(W(("fK", b), g // slots))
            if g >= slots:
                si.append(W(("pd", b), g // slots - 1))
            si.append(A(("fS", b)))
            if c == hi:
                si.append(A(("eQ", qb)))
            pv.append(W(("fP", b), g // slots))
            if has_g and c == c0:
                pv.append(W("fG", lt))
                if lt >= 1:
                    pv.append(W("gE", lt - 1))
            if has_g and c == glob_last:
                pv.append(A("eG"))
            pv.append(A(("pd", b)))
            if c == hi:
                pv.append(A("accF"))
            sw.append(W(("fS", b), g // slots))
            sw.append(A(("fP", b)))
            if c == hi and hop0:
                if lt >= 2:
                    sw.append(W(("xe", lt & 1), lt // 2 - 1))
                sw.append(A(("xf", lt & 1)))
            g += 1
    for s in range(slots):                          # drain before exit
        uses = (g - s + slots - 1) // slots
        if uses > 0:
            pv.append(W(("pd", s), uses - 1))
            si.append(W(("fS", s), uses - 1))
    my = len(tiles)
    if has_g and my > 0:
        pv.append(W("eG", my - 1))
        pv.append(W("eGC", my - 1))
        ep += [A("fGC"), A("fGC")]
    for lt in range(my):
        if has_g and lt + 1 < my:
            ep += [W("eGC", lt), A("fGC"), A("fGC")]
        if hop0:
            ep += [W(("xf", lt & 1), lt // 2), A(("xe", lt & 1))]
        ep += [W("accF", lt), A("accE")]
        if has_g:
            ep.append(A("gE"))
    return play([kq, zp, si, pv, ep, sw], counts) == "done"


CASES = [(4096, 256, 24), (1024, 32, 32), (513, 16, 2), (300, 8, 3), (200, 300, 3), (129, 64, 5),
         (1000, 200, 7), (650, 150, 3), (1034, 150, 2), (389, 256, 2), (640, 640, 1), (130, 8, 2)]


@pytest.mark.parametrize("causal", [False, True], ids=["bidirectional", "causal"])
@pytest.mark.parametrize("n,r,units", CASES)
def test_tiles_dealt_once_and_windows_covered(n, r, units, causal):
    r64, nc, tiles = plan(n, r, causal)
    for G in (152, 7, 1):
        G = min(G, units * tiles)
        seen = set()
        for b in range(G):
            for u, t, lo, hi in cta_tiles(n, r, causal, units, G, b):
                assert (u, t) not in seen
                seen.add((u, t))
                assert lo <= r64 // CK <= hi          # the tile's own first key is in range
                for i in range(t * TR, min(n, t * TR + TR)):
                    klo, khi = max(0, i - r), min(n - 1, i if causal else i + r)
                    assert t * TR - r64 + CK * lo <= klo
                    assert khi <= t * TR - r64 + CK * hi + CK - 1
        assert len(seen) == units * tiles


@pytest.mark.parametrize("causal", [False, True], ids=["bidirectional", "causal"])
@pytest.mark.parametrize("n,r,units", CASES)
def test_barrier_protocol_completes(n, r, units, causal):
    r64, nc, tiles = plan(n, r, causal)
    for G in (152, 3, 1):
        G = min(G, units * tiles)
        for b in range(G):
            tl = cta_tiles(n, r, causal, units, G, b)
            for has_g in (False, True):
                for hop0 in (False, True):
                    assert simulate(tl, r64 // CK, r64, has_g, hop0), (G, b, has_g, hop0)


def test_model_detects_a_missing_arrival():
    # the model is not vacuous: a barrier that expects one arrival more than the
    # roles make (full_P counting a third arrival) stalls it
    r64, nc, tiles = plan(300, 8, False)
    tl = cta_tiles(300, 8, False, 1, 1, 0)
    assert simulate(tl, r64 // CK, r64, True, True)
    assert not simulate(tl, r64 // CK, r64, True, True, fp_arrivals=3)


# ---------------------------------------------------------------- the gather's row split
def quarter_rows(q, nq, n, units, x_ptr, row_cost=2):
    """causal_row_range in csrc/band_hop.cu: rows [R0, R1) of quarter q, found by the
    quarter's 8 lanes probing 8 points a round (both boundaries together)."""
    per_unit = row_cost * n + x_ptr[n]
    total = units * per_unit

    def first_row(t):
        u, rem = divmod(t, per_unit)
        lo, hi = 0, n
        while lo < hi:
            probes = [lo + (hi - lo) * (l + 1) // 9 for l in range(8)]
            k = sum(1 for p in probes if row_cost * p + x_ptr[p] < rem)   # probes below
            new_lo = lo + (hi - lo) * k // 9 + 1 if k > 0 else lo
            new_hi = lo + (hi - lo) * (k + 1) // 9 if k < 8 else hi
            lo, hi = new_lo, new_hi
        return u * n + lo
    return first_row(q * total // nq), first_row((q + 1) * total // nq)


@pytest.mark.parametrize("n,units,nq", [(4096, 24, 14592), (389, 2, 64), (1, 3, 32), (1000, 7, 448)])
def test_causal_gather_split_covers_rows_once_in_balanced_ranges(n, units, nq):
    import random
    rng = random.Random(n)
    counts = [rng.randint(0, 32 * (i + 1) // n) for i in range(n)]   # late rows keep more draws
    x_ptr = [0]
    for c in counts:
        x_ptr.append(x_ptr[-1] + c)
    bounds = [quarter_rows(q, nq, n, units, x_ptr) for q in range(nq)]
    assert bounds[0][0] == 0 and bounds[-1][1] == units * n
    for (a0, a1), (b0, _) in zip(bounds, bounds[1:]):
        assert a0 <= a1 == b0
    ideal = units * (2 * n + x_ptr[n]) / nq
    worst = max(sum(2 + counts[R % n] for R in range(r0, r1)) for r0, r1 in bounds)
    assert worst <= ideal + 2 + max(counts)
