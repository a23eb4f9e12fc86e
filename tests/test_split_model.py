"""The balanced kernel's work split, restated on the host and checked for
the invariants its piece bookkeeping relies on.

The kernel (balanced_kernel.cuh: real_at, vpos0, flush, merge) splits the
(KV head j, sequence b, tile t) units evenly over "virtual" units in which
every segment (b, j) with tiles is preceded by kCut extra units: unit x of
segment number s (in j, b order) sits at position x + kCut * (s + 1), and
warp w takes the units whose positions fall in [w * U, (w + 1) * U).  For
every segment, the warps holding its units must be exactly wf..wl computed
from the first and last positions, and "the piece in warp wf is that warp's
first piece" must match the ranges; kCut = 0 is the plain even split."""
import random

import pytest


def split(tiles, Hk, workers, k_cut, k_min=4):
    B = len(tiles)
    pre, nz = [0], [0]
    for t in tiles:
        pre.append(pre[-1] + t)
        nz.append(nz[-1] + (t > 0))
    TB, NZ = pre[B], nz[B]
    T = Hk * TB
    VTB = TB + k_cut * NZ
    VT = Hk * VTB
    U = max(k_min, -(-VT // workers))

    def real_at(v):  # the first unit at or after position v
        if v >= VT:
            return T
        j, r = divmod(v, VTB)
        lo, hi = 0, B - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if pre[mid] + k_cut * nz[mid] <= r:
                lo = mid
            else:
                hi = mid - 1
        assert tiles[lo] > 0
        off = r - (pre[lo] + k_cut * nz[lo])
        x0 = j * TB + pre[lo]
        return x0 if off < k_cut else x0 + off - k_cut

    starts = [real_at(w * U) for w in range(workers + 1)]
    return pre, nz, TB, NZ, T, U, starts


def check(tiles, Hk, workers, k_cut):
    pre, nz, TB, NZ, T, U, starts = split(tiles, Hk, workers, k_cut)
    assert starts[0] == 0 and starts[-1] == T
    assert all(a <= b for a, b in zip(starts, starts[1:]))  # contiguous, disjoint ranges
    owner = {}
    for w in range(workers):
        for x in range(starts[w], starts[w + 1]):
            owner[x] = w
    assert len(owner) == T  # every unit has exactly one warp
    for j in range(Hk):
        for b, nt in enumerate(tiles):
            if nt == 0:
                continue
            x0 = j * TB + pre[b]
            v0 = x0 + k_cut * (j * NZ + nz[b] + 1)  # vpos0(b, j)
            wf, wl = v0 // U, (v0 + nt - 1) // U
            assert sorted({owner[x] for x in range(x0, x0 + nt)}) == list(range(wf, wl + 1))
            starts_here = x0 == 0 or wf * U > v0 - k_cut - 1
            assert starts_here == (starts[wf] == x0)
    return U, starts


@pytest.mark.parametrize("k_cut", [0, 2, 3, 4])
def test_split_invariants_on_random_batches(k_cut):
    rng = random.Random(100 + k_cut)
    for _ in range(1000):
        B = rng.randint(1, 40)
        tiles = [rng.choice([0, 0, 1, 2, 3, rng.randint(1, 200)]) for _ in range(B)]
        check(tiles, rng.choice([1, 2, 8]), rng.choice([1, 3, 8, 64, 304, 1216]), k_cut)


def test_plain_split_is_even():
    tiles = [7, 0, 33, 12, 5]
    U, starts = check(tiles, 2, 10, 0)
    T = 2 * sum(tiles)
    assert starts == [min(T, w * U) for w in range(11)]


def test_extra_units_take_the_place_of_tiles():
    # every warp but the last covers U positions: its tiles plus the extra
    # units (k_cut before each segment) that fall in its positions
    k_cut = 2
    tiles = [100, 0, 37, 1, 1, 250, 64]
    Hk = 2
    pre, nz, TB, NZ, T, U, starts = split(tiles, Hk, 20, k_cut)
    check(tiles, Hk, 20, k_cut)
    extra = []
    for j in range(Hk):
        for b, nt in enumerate(tiles):
            if nt:
                vs = j * TB + pre[b] + k_cut * (j * NZ + nz[b])  # first extra unit
                extra += [vs + i for i in range(k_cut)]
    for w in range(19):
        n_extra = sum(w * U <= v < (w + 1) * U for v in extra)
        assert starts[w + 1] - starts[w] + n_extra == U
