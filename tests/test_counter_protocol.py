"""Model check of the split kernels' arrival-counter protocol (host only).

The n pieces of a cut segment each add 1 to the segment's 32-bit counter.
The arrival that sees n - 1 merges and later subtracts n (a reduction whose
result nobody waits for).  An arrival that sees a value >= n (unsigned)
flags PKV_ERRBIT_WORKSPACE and later exchanges the counter to a poison value.
The subtraction and the exchange are separate atomics that other
arrivals may overtake, so the model runs every interleaving of the arrivals
with those deferred operations and checks what include/pagedkv.h states:
a zeroed counter merges once, with every piece in, and is left zero; a stale
start that is negative or >= n is flagged in every interleaving and leaves a
counter the next launch flags again; a stale start in [1, n) merges early and
is flagged in some interleavings but not all."""
import pytest

MASK = 0xFFFFFFFF
POISON = 1 << 30


def outcomes(n, start):
    """Every (flagged, merges, final) reachable from counter value `start`;
    merges is a tuple with, per merge, how many pieces had arrived."""
    seen = set()

    def run(counter, arrived, pending, flagged, merges):
        if arrived == n and not pending:
            seen.add((flagged, merges, counter))
            return
        if arrived < n:  # the next piece's atomic add
            old = counter
            c2 = (counter + 1) & MASK
            p2, f2, m2 = pending, flagged, merges
            if old > n - 1:
                f2 = True
                p2 = p2 + (("exch",),)
            elif old == n - 1:
                m2 = m2 + (arrived + 1,)
                p2 = p2 + (("sub",),)
            run(c2, arrived + 1, p2, f2, m2)
        for i, op in enumerate(pending):  # or a deferred atomic lands first
            rest = pending[:i] + pending[i + 1:]
            if op[0] == "sub":
                c2 = (counter - n) & MASK
            else:
                c2 = POISON
            run(c2, arrived, rest, flagged, merges)

    run(start & MASK, 0, (), False, ())
    return seen


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_zeroed_counter_merges_once_complete_and_returns_to_zero(n):
    for flagged, merges, final in outcomes(n, 0):
        assert not flagged
        assert merges == (n,)
        assert final == 0


@pytest.mark.parametrize("n", [2, 3, 5])
@pytest.mark.parametrize("kind", ["minus_one", "minus_n", "n", "n_plus_3", "poison",
                                  "float_one", "pointer_like"])
def test_stale_start_outside_the_piece_range_is_always_flagged(n, kind):
    start = {"minus_one": -1, "minus_n": -n, "n": n, "n_plus_3": n + 3, "poison": POISON,
             "float_one": 0x3F800000, "pointer_like": 0x7F3A10000000 & MASK}[kind]
    finals = set()
    for flagged, merges, final in outcomes(n, start):
        assert flagged
        assert merges == ()  # no arrival sees n - 1: nothing is merged early
        assert final >= n
        finals.add(final)
    for f in finals:  # the next launch on the same counters is flagged again
        assert all(flagged for flagged, _, _ in outcomes(n, f))


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_small_stale_start_merges_early_and_is_caught_only_sometimes(n):
    for c in range(1, n):
        res = outcomes(n, c)
        for flagged, merges, final in res:
            assert merges and merges[0] == n - c < n  # the merge misses c pieces
        flags = {flagged for flagged, _, _ in res}
        assert flags == {True, False}, (n, c)
        # caught whenever a late piece lands before the subtraction
        caught_final = [final for flagged, _, final in res if flagged]
        assert all(f >= n for f in caught_final)
