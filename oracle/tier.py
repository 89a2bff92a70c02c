"""Oracle of the adaptive expert tier's bookkeeping -- TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import
this module; the CUDA library never calls it.

What the Strata pages fix ("BATCHING.md", section "Several requests at once
(batch slots)", the adaptive expert tier paragraphs): batch windows count the
experts they route to; every ``--adapt-every`` windows (default 4) a round
swaps the most-routed experts that are not in the fast tier into it in place of
the least-routed resident ones; ``--adapt-swaps`` bounds the swaps of a round
and ``--adapt-decay`` ages the counts; ``--adapt-min-gain F`` (default 1.5)
makes a swap clear a bar: the routing count of the expert coming in against
the one going out.

The pages leave the rest open; the readings taken here:

* a window adds its per-expert entry counts to fp32 counters (``c += n``);
* a round runs after the counts of every ``adapt_every``-th window are added;
* candidates in: experts outside the tier by counter, descending, ties to the
  lower expert; candidates out: tier experts by counter, ascending, ties to the
  lower expert; the i-th pair swaps when ``i < adapt_swaps``,
  ``c_in > c_out`` and ``c_in >= min_gain * c_out`` (the first pair that fails
  ends the round: later pairs have a smaller ``c_in`` and a larger ``c_out``);
* after the round every counter is multiplied by ``decay``;
* arithmetic in fp32 (``numpy.float32``), one rounding per operation, in this
  order, so that the decisions a device makes in fp32 are reproduced exactly.

Plain Python loops; each function cites the step it follows.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass
class TierState:
    counters: np.ndarray          # float32 [E]
    resident: np.ndarray          # bool [E]
    windows: int = 0
    rounds: int = 0
    last_swaps: List[Tuple[int, int]] = dataclasses.field(default_factory=list)  # (in, out) of the last round


def tier_init(n_experts: int, capacity: int, initial: Optional[Sequence[int]] = None) -> TierState:
    """Counters at zero; the tier holds ``initial`` (default experts 0..capacity-1)."""
    res = np.zeros(n_experts, dtype=bool)
    for e in (range(capacity) if initial is None else initial):
        res[int(e)] = True
    assert int(res.sum()) == capacity
    return TierState(np.zeros(n_experts, dtype=np.float32), res)


def tier_round(st: TierState, adapt_swaps: int, decay: float, min_gain: float) -> List[Tuple[int, int]]:
    """One round: pair the best experts outside the tier with the worst inside it, swap
    the pairs that clear the bar, then age every counter."""
    E = st.counters.size
    c = st.counters
    outside = [e for e in range(E) if not st.resident[e]]
    inside = [e for e in range(E) if st.resident[e]]
    outside.sort(key=lambda e: (-float(c[e]), e))
    inside.sort(key=lambda e: (float(c[e]), e))
    gain = np.float32(min_gain)
    swaps = []
    for i in range(min(adapt_swaps, len(outside), len(inside))):
        a, b = outside[i], inside[i]
        bar = np.float32(gain * c[b])
        if c[a] > c[b] and c[a] >= bar:
            swaps.append((a, b))
        else:
            break
    for a, b in swaps:
        st.resident[a] = True
        st.resident[b] = False
    d = np.float32(decay)
    for e in range(E):
        st.counters[e] = np.float32(st.counters[e] * d)
    st.rounds += 1
    st.last_swaps = swaps
    return swaps


def tier_window(st: TierState, counts: Sequence[int], adapt_every: int, adapt_swaps: int, decay: float,
                min_gain: float) -> List[Tuple[int, int]]:
    """One window: add its per-expert counts; every adapt_every-th window, a round."""
    for e, n in enumerate(counts):
        st.counters[e] = np.float32(st.counters[e] + np.float32(n))
    st.windows += 1
    if adapt_every > 0 and st.windows % adapt_every == 0:
        return tier_round(st, adapt_swaps, decay, min_gain)
    return []
