"""Pins of the oracle's decoder-stack pieces (no GPU)."""
import numpy as np

import oracle
from tests.helpers import small_spec


def test_rmsnorm_closed_form():
    for c in (3.0, -0.5, 1e-4):
        x = np.full(16, c)
        np.testing.assert_allclose(oracle.rmsnorm(x), np.full(16, c / np.sqrt(c * c + 1e-6)), rtol=1e-15)
    x = np.array([3.0, 4.0])
    np.testing.assert_allclose(oracle.rmsnorm(x), x / np.sqrt(12.5 + 1e-6), rtol=1e-15)


def test_attention_len1_broadcasts_kv_heads():
    v = np.arange(4 * 3, dtype=np.float64)  # 4 kv heads of dim 3
    att = oracle.dense_attention_len1(v, 8, 4, 3)
    for h in range(8):
        np.testing.assert_array_equal(att[3 * h:3 * h + 3], v[3 * (h // 2):3 * (h // 2) + 3])


def _zero_qmat(rows, cols, bits=4, block=32, n=1):
    z = np.zeros((n, rows, cols // block), np.uint16)
    return oracle.OQMat(np.zeros((n, rows, cols * bits // 8), np.uint8), z, z.copy(), rows, cols, bits, block)


def test_zero_layer_is_identity_and_routes_to_first_experts():
    d, F, E, k, H, Hkv, Dh = 64, 32, 4, 2, 4, 2, 16
    dense = oracle.ODenseLayer(_zero_qmat(H * Dh, d), _zero_qmat(Hkv * Dh, d), _zero_qmat(Hkv * Dh, d),
                               _zero_qmat(d, H * Dh), H, Hkv, Dh)
    moe = oracle.OMoELayer(E, k, np.zeros((E, d), np.float32), None, _zero_qmat(F, d, n=E),
                           _zero_qmat(F, d, n=E), _zero_qmat(d, F, n=E))
    x = np.random.default_rng(0).standard_normal(d)
    out, q, kk, (sel, g) = oracle.decoder_layer_row(x, dense, moe)
    np.testing.assert_array_equal(out, x)
    assert list(sel) == [0, 1] and np.allclose(g, 0.25)


def test_dense_only_layer_matches_scalar_loops():
    """With a zero MoE, x_out = x + Wo * broadcast(Wv * rmsnorm(x)), checked with scalar loops."""
    rng = np.random.default_rng(1)
    d, H, Hkv, Dh = 32, 4, 2, 8

    def rand_qmat(rows, cols):
        codes = rng.integers(0, 256, size=(1, rows, cols // 2), dtype=np.uint8)
        s = np.float16(rng.uniform(0.001, 0.01, size=(1, rows, cols // 32))).view(np.uint16)
        m = np.float16(rng.uniform(-0.05, 0.0, size=(1, rows, cols // 32))).view(np.uint16)
        return oracle.OQMat(codes, s, m, rows, cols, 4, 32)

    dq, dk, dv, do = rand_qmat(H * Dh, d), rand_qmat(Hkv * Dh, d), rand_qmat(Hkv * Dh, d), rand_qmat(d, H * Dh)
    dense = oracle.ODenseLayer(dq, dk, dv, do, H, Hkv, Dh)
    moe = oracle.OMoELayer(2, 1, np.zeros((2, d), np.float32), None, _zero_qmat(32, d, n=2),
                           _zero_qmat(32, d, n=2), _zero_qmat(d, 32, n=2))
    x = rng.standard_normal(d)
    out, _, _, _ = oracle.decoder_layer_row(x, dense, moe)

    def w(m, r, c):
        byte = int(m.codes[0, r, c // 2])
        q = (byte >> (4 * (c % 2))) & 15
        s = float(np.uint16(m.scale[0, r, c // 32]).view(np.float16))
        mn = float(np.uint16(m.min[0, r, c // 32]).view(np.float16))
        return s * q + mn

    ms = sum(v * v for v in x) / d
    a = [v / (ms + 1e-6) ** 0.5 for v in x]
    v = [sum(w(dv, r, c) * a[c] for c in range(d)) for r in range(Hkv * Dh)]
    att = [v[(h // (H // Hkv)) * Dh + i] for h in range(H) for i in range(Dh)]
    expect = [x[i] + sum(w(do, i, c) * att[c] for c in range(H * Dh)) for i in range(d)]
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-13)
