"""Pins of the head / token-draw / proposal-check oracle (no GPU)."""
import math

import numpy as np
import pytest

import oracle
from oracle import head as oh


@pytest.mark.parametrize("key,counter", [
    ((0, 0), (1, 0, 0, 0)), ((0x1234, 0x5678), (1, 0, 0, 0)), ((2 ** 64 - 1, 7), (5, 9, 0, 3)),
    ((123456789, 0), (1000, 0, 0, 0)), ((42, 0), (2 ** 40, 2 ** 63, 1, 2 ** 64 - 1)),
])
def test_philox_matches_numpys_philox_bit_generator(key, counter):
    """numpy's Philox (4x64, 10 rounds) increments its counter before each
    block: a generator set to counter c - 1 yields the block of counter c."""
    prev = list(counter)
    prev[0] -= 1  # every counter above has word 0 >= 1
    bg = np.random.Philox(counter=np.array(prev, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
    assert [int(v) for v in bg.random_raw(4)] == oh.philox4x64(counter, key)


def test_row_uniform_is_the_top_24_bits():
    w = oh.philox4x64([17, 0, 0, 0], [99, 0])[0]
    u = oh.row_uniform(99, 17)
    assert u == (w >> 40) / 2 ** 24 and 0.0 <= u < 1.0


def test_greedy_is_argmax_with_ties_to_the_lower_token():
    assert oh.draw_token(np.array([0.1, 2.0, -1.0, 2.0]), 0.0, 5, 5) == 1
    assert oh.draw_token(np.array([3.0, 2.0]), -1.0, 5, 5) == 0


def test_two_token_draw_follows_the_uniform():
    """logits (0, ln 3) at temperature 1: p = (1/4, 3/4), so the token is 0
    exactly when the row's uniform is below 1/4."""
    logits = np.array([0.0, math.log(3.0)])
    seen = set()
    for pos in range(1, 200):
        u = oh.row_uniform(7, pos)
        tok = oh.draw_token(logits, 1.0, 7, pos)
        assert tok == (0 if u < 0.25 else 1)
        seen.add(tok)
    assert seen == {0, 1}


def test_draw_frequencies_match_the_softmax():
    rng = np.random.default_rng(0)
    logits = rng.normal(0, 1.0, size=6)
    tau = 0.7
    p = np.exp(logits / tau - (logits / tau).max())
    p /= p.sum()
    n = 6000
    counts = np.bincount([oh.draw_token(logits, tau, 11, pos) for pos in range(1, n + 1)], minlength=6)
    # each frequency within 5 binomial standard deviations
    assert np.all(np.abs(counts / n - p) <= 5 * np.sqrt(p * (1 - p) / n))


def test_tiny_temperature_draw_is_greedy():
    logits = np.array([0.3, 1.2, 1.1, -4.0])
    for pos in range(1, 50):
        assert oh.draw_token(logits, 1e-4, 3, pos) == 1


def test_head_logits_match_scalar_loops():
    rng = np.random.default_rng(2)
    V, d = 16, 64
    codes = rng.integers(0, 256, size=(1, V, d // 2), dtype=np.uint8)
    s = np.float16(rng.uniform(0.001, 0.02, size=(1, V, d // 32))).view(np.uint16)
    m = np.float16(rng.uniform(-0.1, 0.0, size=(1, V, d // 32))).view(np.uint16)
    W = oracle.OQMat(codes, s, m, V, d, 4, 32)
    x = rng.standard_normal(d)
    ms = sum(a * a for a in x) / d
    a = [v / (ms + 1e-6) ** 0.5 for v in x]

    def w(r, c):
        q = (int(codes[0, r, c // 2]) >> (4 * (c % 2))) & 15
        return float(np.uint16(s[0, r, c // 32]).view(np.float16)) * q + float(np.uint16(m[0, r, c // 32]).view(np.float16))
    expect = [sum(w(r, c) * a[c] for c in range(d)) for r in range(V)]
    np.testing.assert_allclose(oh.head_logits(x, W), expect, rtol=1e-12, atol=1e-12)


def test_verify_slots_hand_worked():
    # slot A: rows 0-1, proposal 5 matches row 0's token 5 -> 2 tokens
    # slot B: rows 2-3, proposal 8 against row 2's token 9 -> 1 token
    # slot C: row 4 alone -> 1 token
    # slot D: rows 5-7 (two proposals): 1 == 1, then 4 != 3 -> 2 tokens
    tokens = [5, 7, 9, 8, 2, 1, 3, 6]
    fed = [-1, 5, -1, 8, -1, -1, 1, 4]
    assert oh.verify_slots(tokens, fed) == [2, 0, 1, 0, 1, 2, 0, 0]
    # a later match after a mismatch does not count
    assert oh.verify_slots([1, 2, 3], [-1, 9, 2]) == [1, 0, 0]
