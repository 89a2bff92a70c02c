"""Oracle of the window's output head, token draw and proposal check -- TEST
INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import
this module; the CUDA library never calls it.

What the Strata pages fix:

* "BATCHING.md", section "Several requests at once (batch slots)", opening
  paragraph: the head is among the weights a verify window reads once for all
  of its rows;
* same page, section "Exactness", sampled requests: every row draws its token
  with the solo window's counter-based draw, Philox(seed, position);
* same page, ``--batch-mtp`` paragraph: a window carries two rows per slot,
  the slot's token and its MTP proposal, and the window verifies the
  proposal (66-67 % accepted in the pages' table).

The readings taken where the pages are silent:

* head input: RMSNorm of the row (``x / sqrt(mean(x^2) + 1e-6)``, unit gain),
  the plain pre-norm reading applied to the head as to every block;
* head weight: ``[V][d]`` in the library's block format; logits in fp64 here;
* greedy rows (temperature <= 0): the argmax, ties to the lower token;
* sampled rows: one uniform ``u`` per row from Philox4x64-10 (Salmon et al.,
  "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with key
  ``(seed, 0)`` and counter ``(position, 0, 0, 0)``: ``u`` = the top 24 bits
  of the first output word times 2^-24; the token is the first ``v`` whose
  cumulative softmax(logits / temperature) probability exceeds ``u``
  (inverse-CDF sampling; the greedy token should rounding leave ``u`` at or
  above the total);
* the proposal check: a slot's rows are consecutive; its first row was fed
  the slot's last token (marked ``fed = -1``), each later row was fed a
  proposal; the slot emits its first row's token, and then, for as long as the
  previous row's token equals the proposal a row was fed, that row's token too.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np

from .moe_window import OQMat, dequant, rmsnorm

# Philox4x64 round multipliers and key increments (Salmon et al. 2011)
_M0, _M1 = 0xD2E7470EE14C6C93, 0xCA5A826395121157
_W0, _W1 = 0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B
_MASK = (1 << 64) - 1


def philox4x64(counter: Sequence[int], key: Sequence[int], rounds: int = 10) -> List[int]:
    """Philox4x64-R on a 4-word counter and a 2-word key (plain Python integers).

    Each round multiplies words 0 and 2 by the two constants (128-bit
    products), then the new block is (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
    hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key is bumped by the Weyl
    constants before every round but the first.
    """
    c = [int(v) & _MASK for v in counter]
    k = [int(v) & _MASK for v in key]
    for r in range(rounds):
        if r:
            k = [(k[0] + _W0) & _MASK, (k[1] + _W1) & _MASK]
        p0 = _M0 * c[0]
        p1 = _M1 * c[2]
        c = [(p1 >> 64) ^ c[1] ^ k[0], p1 & _MASK, (p0 >> 64) ^ c[3] ^ k[1], p0 & _MASK]
    return c


def row_uniform(seed: int, position: int) -> float:
    """The row's uniform: top 24 bits of Philox4x64-10(key (seed, 0), counter (position, 0, 0, 0))[0] x 2^-24."""
    w = philox4x64([position, 0, 0, 0], [seed, 0])[0]
    return (w >> 40) * 2.0 ** -24


def head_logits(x: np.ndarray, head: OQMat) -> np.ndarray:
    """logits = W_head rmsnorm(x), fp64."""
    return dequant(head) @ rmsnorm(x)


def draw_token(logits: np.ndarray, temperature: float, seed: int, position: int) -> int:
    """Greedy argmax (temperature <= 0; ties to the lower token) or the
    inverse-CDF draw of softmax(logits / temperature) at the row's uniform."""
    if temperature <= 0:
        return int(np.argmax(logits))          # first maximum: the lower token
    z = logits / temperature
    p = np.exp(z - z.max())
    cdf = np.cumsum(p / p.sum())
    u = row_uniform(seed, position)
    v = int(np.searchsorted(cdf, u, side="right"))
    if v >= logits.size:                       # rounding left u at or above the total
        v = int(np.argmax(logits))
    return v


def verify_slots(tokens: Sequence[int], fed: Sequence[int]) -> List[int]:
    """Tokens each slot emits, at its first row (0 at proposal rows).

    A row with fed[t] = -1 starts a slot; the slot emits tokens[start], then
    tokens[t] for each next proposal row t while tokens[t - 1] == fed[t].
    """
    T = len(tokens)
    n = [0] * T
    t = 0
    while t < T:
        assert fed[t] == -1, "a window starts with a slot's first row"
        start, emit = t, 1
        t += 1
        ok = True
        while t < T and fed[t] != -1:
            if ok and tokens[t - 1] == fed[t]:
                emit += 1
            else:
                ok = False
            t += 1
        n[start] = emit
    return n


def window_slots(rows_per_slot: Sequence[int], start: int, max_rows: int = 8):
    """Slots of the next window when more slots are open than one window holds.

    The pages ("BATCHING.md", --batch-mtp paragraph): a window carries each
    active slot's rows (its token, plus its proposal with --batch-mtp), at most
    8 rows, and more slots rotate through.  Reading: starting at slot
    ``start``, slots are taken in cyclic order, each once, while their rows
    still fit; a slot with no rows is skipped; the next window starts at the
    slot after the last one taken.  Returns (slots in window order, next start).
    """
    n = len(rows_per_slot)
    taken, used = [], 0
    last = start - 1
    for i in range(n):
        s = (start + i) % n
        r = int(rows_per_slot[s])
        if r <= 0:
            continue
        if used + r > max_rows:
            break
        taken.append(s)
        used += r
        last = s
    return taken, (last + 1) % n if n else 0
