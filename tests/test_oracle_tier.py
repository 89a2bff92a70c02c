"""Pins of the adaptive-tier oracle (no GPU): a hand-worked sequence of
windows and rounds, the tie order, the min-gain bar, and invariants."""
import numpy as np

from oracle import tier as ot


def test_hand_worked_rounds():
    # E = 4, a tier of 2 holding {0, 1}; a round every 2 windows, at most 2
    # swaps, decay 0.5, min gain 1.5.
    st = ot.tier_init(4, 2)
    kw = dict(adapt_every=2, adapt_swaps=2, decay=0.5, min_gain=1.5)
    assert ot.tier_window(st, [1, 0, 3, 0], **kw) == []          # c = 1 0 3 0, no round yet
    # c = 1 0 5 1; in: 2 (5), 3 (1); out: 1 (0), 0 (1).  (2, 1): 5 > 0, 5 >= 0 -> swap;
    # (3, 0): 1 > 1 fails -> the round ends.  Then c = 0.5 0 2.5 0.5.
    assert ot.tier_window(st, [0, 0, 2, 1], **kw) == [(2, 1)]
    assert list(np.nonzero(st.resident)[0]) == [0, 2]
    np.testing.assert_array_equal(st.counters, np.float32([0.5, 0, 2.5, 0.5]))
    assert ot.tier_window(st, [0, 4, 0, 0], **kw) == []          # c = 0.5 4 2.5 0.5
    # c = 0.5 6 2.5 1.5; in: 1 (6), 3 (1.5); out: 0 (0.5), 2 (2.5).  (1, 0) swaps;
    # (3, 2): 1.5 > 2.5 fails.  Then c = 0.25 3 1.25 0.75.
    assert ot.tier_window(st, [0, 2, 0, 1], **kw) == [(1, 0)]
    assert list(np.nonzero(st.resident)[0]) == [1, 2]
    np.testing.assert_array_equal(st.counters, np.float32([0.25, 3, 1.25, 0.75]))
    assert st.windows == 4 and st.rounds == 2


def test_gain_bar_is_inclusive_and_needs_a_strict_gain():
    kw = dict(adapt_every=1, adapt_swaps=1, decay=1.0, min_gain=1.5)
    st = ot.tier_init(2, 1)                      # tier {0}
    assert ot.tier_window(st, [2, 3], **kw) == [(1, 0)]        # 3 >= 1.5 * 2 exactly: swaps
    st = ot.tier_init(2, 1)
    assert ot.tier_window(st, [2, 2.9990234375], **kw) == []   # just under the bar
    st = ot.tier_init(2, 1)
    assert ot.tier_window(st, [0, 0], **kw) == []              # 0 >= 1.5 * 0, but no gain
    st = ot.tier_init(2, 1)
    assert ot.tier_window(st, [0, 1], **kw) == [(1, 0)]        # anything beats a zero count


def test_ties_go_to_the_lower_expert_on_both_sides():
    st = ot.tier_init(6, 3, initial=[3, 4, 5])
    swaps = ot.tier_window(st, [5, 5, 5, 1, 1, 1], adapt_every=1, adapt_swaps=2, decay=1.0, min_gain=1.5)
    assert swaps == [(0, 3), (1, 4)]


def test_invariants_over_random_windows():
    rng = np.random.default_rng(0)
    E, cap = 32, 12
    for gain, swaps_max in ((1.5, 4), (1.0, 32), (1e30, 8)):
        st = ot.tier_init(E, cap)
        for w in range(40):
            counts = rng.multinomial(64, rng.dirichlet(np.full(E, 0.3)))
            before = st.resident.copy()
            c = (st.counters + counts.astype(np.float32)).astype(np.float32)  # the counts a round sees
            sw = ot.tier_window(st, counts, adapt_every=3, adapt_swaps=swaps_max, decay=0.5, min_gain=gain)
            assert int(st.resident.sum()) == cap
            assert len(sw) <= swaps_max
            for a, b in sw:
                assert not before[a] and before[b] and st.resident[a] and not st.resident[b]
                assert c[a] > c[b] and c[a] >= np.float32(gain) * c[b]
                if gain == 1e30:
                    assert c[b] == 0  # only an expert with no count yields to such a bar


def test_one_round_with_no_decay_and_no_bar_takes_the_top_counts():
    """decay 1, gain 1 and enough swaps: after one round the tier holds the
    capacity experts with the largest counts (ties to the lower expert)."""
    rng = np.random.default_rng(1)
    E, cap = 20, 7
    counts = rng.integers(0, 50, size=E)
    st = ot.tier_init(E, cap)
    ot.tier_window(st, counts, adapt_every=1, adapt_swaps=E, decay=1.0, min_gain=1.0)
    top = sorted(range(E), key=lambda e: (-counts[e], e))[:cap]
    # experts tied with the cut may stay either side; the counts held must be the top ones
    held = sorted(counts[np.nonzero(st.resident)[0]])
    assert held == sorted(counts[top])
