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


# ---------------------------------------------------------------------------
# a decoder layer with both halves non-zero, and two layers chained, against
# scalar loops written out here (pre-norm attention of one position, then
# pre-norm MoE with its residual)


def _rand_qmat(rng, rows, cols, n=1):
    codes = rng.integers(0, 256, size=(n, rows, cols // 2), dtype=np.uint8)
    s = np.float16(rng.uniform(0.002, 0.02, size=(n, rows, cols // 32))).view(np.uint16)
    m = np.float16(rng.uniform(-0.12, -0.02, size=(n, rows, cols // 32))).view(np.uint16)
    return oracle.OQMat(codes, s, m, rows, cols, 4, 32)


def _w(m, i, r, c):
    """Element (r, c) of matrix i of a 4-bit/32 stack, decoded one byte at a time."""
    byte = int(m.codes[i, r, c // 2])
    q = (byte >> (4 * (c % 2))) & 15
    s = float(np.uint16(m.scale[i, r, c // 32]).view(np.float16))
    mn = float(np.uint16(m.min[i, r, c // 32]).view(np.float16))
    return s * q + mn


def _layer_weights(rng, d=32, H=4, Hkv=2, Dh=8, E=3, k=2, F=32, Fs=32):
    dense = oracle.ODenseLayer(_rand_qmat(rng, H * Dh, d), _rand_qmat(rng, Hkv * Dh, d),
                               _rand_qmat(rng, Hkv * Dh, d), _rand_qmat(rng, d, H * Dh), H, Hkv, Dh)
    rw = rng.normal(0.0, 0.3, size=(E, d)).astype(np.float32)
    rb = rng.normal(0.0, 0.1, size=E).astype(np.float32)
    moe = oracle.OMoELayer(E, k, rw, rb, _rand_qmat(rng, F, d, E), _rand_qmat(rng, F, d, E),
                           _rand_qmat(rng, d, F, E), _rand_qmat(rng, Fs, d), _rand_qmat(rng, Fs, d),
                           _rand_qmat(rng, d, Fs))
    return dense, moe


def _scalar_layer(x, dense, moe):
    """One decoder layer on one row, every sum a Python loop."""
    import math
    d = len(x)
    H, Hkv, Dh = dense.heads, dense.kv_heads, dense.head_dim

    def norm(v):
        ms = sum(a * a for a in v) / len(v)
        return [a / math.sqrt(ms + 1e-6) for a in v]

    def matvec(m, i, rows, cols, v):
        return [sum(_w(m, i, r, c) * v[c] for c in range(cols)) for r in range(rows)]

    def ffn(g, u, dn, i, rows, v):
        gu = matvec(g, i, rows, d, v)
        uu = matvec(u, i, rows, d, v)
        h = [gu[f] / (1.0 + math.exp(-gu[f])) * uu[f] for f in range(rows)]
        return matvec(dn, i, d, rows, h)

    a = norm(list(x))
    v = matvec(dense.v, 0, Hkv * Dh, d, a)
    att = [v[(h // (H // Hkv)) * Dh + i] for h in range(H) for i in range(Dh)]
    o = matvec(dense.o, 0, d, H * Dh, att)
    x1 = [x[i] + o[i] for i in range(d)]
    b = norm(x1)
    E, k = moe.n_experts, moe.top_k
    logit = [sum(float(moe.router_w[e, j]) * b[j] for j in range(d)) + float(moe.router_b[e]) for e in range(E)]
    order = sorted(range(E), key=lambda e: (-logit[e], e))[:k]
    top = max(logit)
    z = sum(math.exp(l - top) for l in logit)
    out = [x1[i] for i in range(d)]
    s = ffn(moe.shared_gate, moe.shared_up, moe.shared_down, 0, moe.shared_gate.rows, b)
    y = [s[i] for i in range(d)]
    for e in order:
        g = math.exp(logit[e] - top) / z
        oe = ffn(moe.gate, moe.up, moe.down, e, moe.gate.rows, b)
        y = [y[i] + g * oe[i] for i in range(d)]
    return [out[i] + y[i] for i in range(d)], order


def test_decoder_layer_with_moe_matches_scalar_loops():
    """x_out = x1 + shared(b) + sum_j g_j expert_j(b), b = rmsnorm(x1), x1 = x + Wo att:
    the router and the experts see rmsnorm(x1) and the residual is x1."""
    rng = np.random.default_rng(7)
    dense, moe = _layer_weights(rng)
    for _ in range(3):
        x = rng.standard_normal(32) * 2.0
        out, _, _, (sel, _) = oracle.decoder_layer_row(x, dense, moe)
        expect, order = _scalar_layer(x, dense, moe)
        assert list(sel) == order
        np.testing.assert_allclose(out, expect, rtol=1e-11, atol=1e-12)


def test_two_layer_stack_chains_the_layers():
    """stack_row carries each layer's output into the next layer."""
    rng = np.random.default_rng(8)
    l1, l2 = _layer_weights(rng), _layer_weights(rng)
    x = rng.standard_normal(32)
    out, routing = oracle.stack_row(x, [l1[0], l2[0]], [l1[1], l2[1]])
    h1, o1 = _scalar_layer(x, *l1)
    h2, o2 = _scalar_layer(h1, *l2)
    assert [list(r[0]) for r in routing] == [o1, o2]
    np.testing.assert_allclose(out, h2, rtol=1e-11, atol=1e-12)
