"""The window's slot rotation (more slots than one window holds): the oracle's
rule against hand-worked rotations, and the library's host function against
the oracle (no GPU)."""
import numpy as np
import pytest

from oracle import head as oh
from slot_decode_window_gb300 import binding as B
from slot_decode_window_gb300 import build as BLD


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.load()


def test_six_mtp_slots_rotate_four_per_window():
    rows = [2] * 6
    w1, s = oh.window_slots(rows, 0)
    w2, s = oh.window_slots(rows, s)
    w3, s = oh.window_slots(rows, s)
    assert (w1, w2, w3, s) == ([0, 1, 2, 3], [4, 5, 0, 1], [2, 3, 4, 5], 0)


def test_mixed_rows_and_idle_slots():
    # slot 2 idle; 2 + 1 + 2 + 2 + 1 = 8 rows fit in one window
    assert oh.window_slots([2, 1, 0, 2, 2, 1], 0) == ([0, 1, 3, 4, 5], 0)
    # a 2-row slot that would make 9 rows waits for the next window
    assert oh.window_slots([2, 2, 2, 1, 2], 1) == ([1, 2, 3, 4], 0)
    # no MTP: eight single-row slots per window
    assert oh.window_slots([1] * 10, 8) == ([8, 9, 0, 1, 2, 3, 4, 5], 6)


def test_every_slot_is_served_equally_over_a_cycle():
    rng = np.random.default_rng(0)
    for n in range(1, 20):
        rows = [2] * n
        served = np.zeros(n, int)
        s = 0
        for _ in range(4 * n):
            w, s = oh.window_slots(rows, s)
            assert sum(rows[i] for i in w) <= 8 and len(set(w)) == len(w)
            served[w] += 1
        assert served.max() - served.min() <= 1


def test_library_matches_the_oracle(lib):
    rng = np.random.default_rng(1)
    for _ in range(300):
        n = int(rng.integers(1, 13))
        rows = [int(r) for r in rng.integers(0, 3, size=n)]
        start = int(rng.integers(0, n))
        mr = int(rng.integers(2, 9))
        st, w, nxt = B.strata_window_slots(rows, start, mr)
        assert st == B.STRATA_OK
        assert (w, nxt) == oh.window_slots(rows, start, mr)


@pytest.mark.parametrize("rows,start,mr", [([2, 2], 2, 8), ([2, 2], -1, 8), ([9, 1], 0, 8), ([2, -1], 0, 8),
                                           ([1], 0, 0), ([1], 0, 9), ([], 0, 8)])
def test_library_rejects_bad_arguments(lib, rows, start, mr):
    st, w, nxt = B.strata_window_slots(rows, start, mr)
    assert st == B.STRATA_EINVAL
