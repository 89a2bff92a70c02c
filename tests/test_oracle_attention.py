"""Pins of the KV-cache attention oracle (no GPU)."""
import math

import numpy as np

import oracle
from oracle import attention as oa
from tests.test_oracle_stack import _layer_weights


def _caches(rng, slots=3, kvh=2, ctx=6, hd=8):
    kc = oa.fp16_round(rng.standard_normal((slots, kvh, ctx, hd)))
    vc = oa.fp16_round(rng.standard_normal((slots, kvh, ctx, hd)))
    return kc, vc


def test_first_position_is_the_length_one_reading():
    """At position 0 a row attends to its own entry only: query head h outputs
    (the fp16 rounding of) v of its kv head, the length-one reading."""
    rng = np.random.default_rng(0)
    kc, vc = _caches(rng)
    k, v, q = rng.standard_normal(16), rng.standard_normal(16), rng.standard_normal(32)
    oa.append_kv(kc, vc, k, v, slot=1, pos=0)
    att = oa.attention_row(q, kc, vc, slot=1, pos=0, heads=4)
    np.testing.assert_array_equal(att, oracle.dense_attention_len1(oa.fp16_round(v), 4, 2, 8))


def test_zero_query_averages_the_values():
    rng = np.random.default_rng(1)
    kc, vc = _caches(rng)
    att = oa.attention_row(np.zeros(32), kc, vc, slot=2, pos=4, heads=4)
    for h in range(4):
        np.testing.assert_allclose(att[8 * h:8 * h + 8], vc[2, h // 2, :5, :].mean(axis=0), rtol=1e-14, atol=1e-15)


def test_scalar_loops():
    rng = np.random.default_rng(2)
    kc, vc = _caches(rng)
    q = rng.standard_normal(32)
    pos, slot = 3, 0
    att = oa.attention_row(q, kc, vc, slot, pos, heads=4)
    for h in range(4):
        g = h // 2
        s = [sum(q[8 * h + i] * kc[slot, g, j, i] for i in range(8)) / math.sqrt(8) for j in range(pos + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for i in range(8):
            want = sum(e[j] / z * vc[slot, g, j, i] for j in range(pos + 1))
            assert abs(att[8 * h + i] - want) <= 1e-13


def test_positions_beyond_the_row_and_other_slots_do_not_matter():
    rng = np.random.default_rng(3)
    kc, vc = _caches(rng)
    q = rng.standard_normal(32)
    a1 = oa.attention_row(q, kc, vc, 1, 2, heads=4)
    kc[1, :, 3:, :] = 7.0
    vc[1, :, 3:, :] = -7.0
    kc[0], vc[2] = 0.0, 5.0
    np.testing.assert_array_equal(a1, oa.attention_row(q, kc, vc, 1, 2, heads=4))


def test_a_window_equals_its_rows_one_after_another():
    """A window holding a slot's token row (position p) and proposal row (p + 1)
    and another slot's row gives, bit for bit, what running the rows one at a
    time in that order gives (each row's entry is written before later rows
    attend)."""
    rng = np.random.default_rng(4)
    dense, moe = _layer_weights(rng)
    X = rng.standard_normal((3, 32))
    slots, positions = [0, 0, 1], [3, 4, 2]
    kc, vc = _caches(rng, slots=2, kvh=2, ctx=6, hd=8)
    kc2, vc2 = kc.copy(), vc.copy()
    out, q, k, sel, _ = oa.decoder_layer_window(X, dense, moe, kc, vc, slots, positions)
    for t in range(3):
        o1, q1, k1, s1, _ = oa.decoder_layer_window(X[t:t + 1], dense, moe, kc2, vc2, slots[t:t + 1],
                                                    positions[t:t + 1])
        np.testing.assert_array_equal(out[t], o1[0])
        assert list(sel[t]) == list(s1[0])
    np.testing.assert_array_equal(kc, kc2)
    np.testing.assert_array_equal(vc, vc2)


def test_layer_at_position_zero_matches_the_length_one_layer_with_rounded_v():
    """A fresh slot (position 0): the layer equals the length-one decoder layer
    whose v is rounded to fp16, computed here by hand from the oracle's pieces."""
    rng = np.random.default_rng(5)
    dense, moe = _layer_weights(rng)
    x = rng.standard_normal(32)
    kc, vc = _caches(rng, slots=1, kvh=2, ctx=2, hd=8)
    out, _, _, _, _ = oa.decoder_layer_window(x[None], dense, moe, kc, vc, [0], [0])
    a = oracle.rmsnorm(x)
    v = oa.fp16_round(oracle.dequant(dense.v) @ a)
    x1 = x + oracle.dequant(dense.o) @ oracle.dense_attention_len1(v, dense.heads, dense.kv_heads, dense.head_dim)
    y, _, _ = oracle.moe_row(oracle.rmsnorm(x1), moe)
    np.testing.assert_allclose(out[0], x1 + y, rtol=1e-13, atol=1e-13)
