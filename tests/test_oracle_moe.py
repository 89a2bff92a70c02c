"""Pins of the oracle's window step: brute force, textbook special cases,
closed forms and the invariants of the definition (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import omoe, small_spec


def _brute_dequant(m: oracle.OQMat, idx: int) -> np.ndarray:
    """Pure-Python element-by-element decoding of one matrix (independent of oracle.dequant)."""
    out = np.empty((m.rows, m.cols))
    for r in range(m.rows):
        row = int.from_bytes(bytes(m.codes[idx, r]), "little")
        sc = np.frombuffer(m.scale[idx, r].astype(np.uint16).tobytes(), np.float16)
        mn = np.frombuffer(m.min[idx, r].astype(np.uint16).tobytes(), np.float16)
        for c in range(m.cols):
            q = (row >> (c * m.bits)) & ((1 << m.bits) - 1)
            out[r, c] = float(sc[c // m.block]) * q + float(mn[c // m.block])
    return out


def _brute_window(x, ol: oracle.OMoELayer):
    """Every expert densely on every row, then a one-hot gate mask (einsum form)."""
    E = ol.n_experts
    Wg = np.stack([_brute_dequant(ol.gate, e) for e in range(E)])
    Wu = np.stack([_brute_dequant(ol.up, e) for e in range(E)])
    Wd = np.stack([_brute_dequant(ol.down, e) for e in range(E)])
    x = x.astype(np.float64)
    g_all = np.einsum("efd,td->tef", Wg, x)
    u_all = np.einsum("efd,td->tef", Wu, x)
    h_all = g_all * torch.sigmoid(torch.from_numpy(g_all)).numpy() * u_all
    o_all = np.einsum("edf,tef->ted", Wd, h_all)
    logits = x @ ol.router_w.astype(np.float64).T
    if ol.router_b is not None:
        logits = logits + ol.router_b
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    mask = np.zeros_like(p)
    for t in range(x.shape[0]):
        top = sorted(range(E), key=lambda e: (-logits[t, e], e))[: ol.top_k]
        mask[t, top] = 1.0
    w = p * mask
    if ol.renorm:
        w = w / w.sum(axis=1, keepdims=True)
    y = np.einsum("te,ted->td", w, o_all)
    if ol.shared_gate is not None:
        sg, su, sd = (_brute_dequant(m, 0) for m in (ol.shared_gate, ol.shared_up, ol.shared_down))
        hs = (x @ sg.T) * torch.sigmoid(torch.from_numpy(x @ sg.T)).numpy() * (x @ su.T)
        y = y + hs @ sd.T
    return y


@pytest.mark.parametrize("spec", [small_spec(), small_spec(bits=2, block=16, renorm_topk=1),
                                  small_spec(shared_ffn=0, top_k=3)])
def test_window_matches_brute_force(spec):
    layer = wlm.make_moe_layer(spec, seed=5)
    ol = omoe(layer)
    x = np.random.default_rng(0).standard_normal((4, spec.hidden)).astype(np.float32)
    res = oracle.moe_window(x, ol)
    np.testing.assert_allclose(res["y"], _brute_window(x, ol), rtol=1e-10, atol=1e-13)


def test_single_expert_is_textbook_swiglu():
    """E = k = 1, no shared expert: a dense SwiGLU MLP (torch float64 on brute-decoded weights)."""
    spec = small_spec(n_experts=1, top_k=1, shared_ffn=0)
    ol = omoe(wlm.make_moe_layer(spec, seed=8))
    x = np.random.default_rng(1).standard_normal((3, spec.hidden)).astype(np.float32)
    Wg, Wu, Wd = (torch.from_numpy(_brute_dequant(m, 0)) for m in (ol.gate, ol.up, ol.down))
    xt = torch.from_numpy(x.astype(np.float64))
    ref = torch.nn.functional.linear(torch.nn.functional.silu(torch.nn.functional.linear(xt, Wg))
                                     * torch.nn.functional.linear(xt, Wu), Wd)
    res = oracle.moe_window(x, ol)
    np.testing.assert_allclose(res["y"], ref.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(res["topk_w"], np.ones((3, 1)))


def _row_constant_qmat(codes_per_row, scale, mn, cols, bits=4, block=32):
    rows = len(codes_per_row)
    per_byte = 8 // bits
    byte = lambda q: sum(q << (bits * i) for i in range(per_byte))
    codes = np.array([[byte(q)] * (cols * bits // 8) for q in codes_per_row], np.uint8)[None]
    s = np.full((1, rows, cols // block), np.float16(scale).view(np.uint16), np.uint16)
    m = np.full((1, rows, cols // block), np.float16(mn).view(np.uint16), np.uint16)
    return oracle.OQMat(codes, s, m, rows, cols, bits, block)


def test_row_constant_weights_closed_form():
    """W[f][j] = a_f etc.: y_i = c_i * sum_f silu(a_f S) * b_f S with S = sum_j x_j."""
    d, F = 64, 32
    qa = [i % 16 for i in range(F)]
    qb = [(3 * i + 1) % 16 for i in range(F)]
    qc = [(5 * i + 2) % 16 for i in range(d)]
    gate = _row_constant_qmat(qa, 0.0625, -0.5, d)
    up = _row_constant_qmat(qb, 0.03125, -0.25, d)
    down = _row_constant_qmat(qc, 0.125, -1.0, F)
    ol = oracle.OMoELayer(1, 1, np.zeros((1, d), np.float32), None, gate, up, down)
    x = np.random.default_rng(2).standard_normal((2, d)).astype(np.float32)
    res = oracle.moe_window(x, ol)
    for t in range(2):
        S = float(np.sum(x[t].astype(np.float64)))
        h = 0.0
        for f in range(F):
            a, b = 0.0625 * qa[f] - 0.5, 0.03125 * qb[f] - 0.25
            z = a * S
            h += z / (1.0 + np.exp(-z)) * (b * S)
        expect = np.array([(0.125 * qc[i] - 1.0) * h for i in range(d)])
        np.testing.assert_allclose(res["y"][t], expect, rtol=1e-12, atol=1e-12)


def _layer_and_x(T=6, seed=0, **kw):
    spec = small_spec(**kw)
    ol = omoe(wlm.make_moe_layer(spec, seed=seed))
    x = np.random.default_rng(seed + 100).standard_normal((T, spec.hidden)).astype(np.float32)
    return ol, x


def test_window_equals_single_row_windows():
    """A T-row window equals T one-row windows, bit for bit ("Exactness")."""
    ol, x = _layer_and_x()
    full = oracle.moe_window(x, ol)
    for t in range(x.shape[0]):
        one = oracle.moe_window(x[t:t + 1], ol)
        np.testing.assert_array_equal(full["y"][t], one["y"][0])
        np.testing.assert_array_equal(full["topk_idx"][t], one["topk_idx"][0])
        np.testing.assert_array_equal(full["topk_w"][t], one["topk_w"][0])


def test_rows_unaffected_by_other_rows():
    """Changing rows routed elsewhere leaves an expert's rows bitwise unchanged."""
    ol, x = _layer_and_x(T=6, seed=3, n_experts=8)
    base = oracle.moe_window(x, ol)
    x2 = x.copy()
    rng = np.random.default_rng(9)
    changed = [1, 4]
    for t in changed:
        x2[t] = rng.standard_normal(x.shape[1])
    alt = oracle.moe_window(x2, ol)
    for t in range(6):
        if t not in changed:
            np.testing.assert_array_equal(alt["y"][t], base["y"][t])
            np.testing.assert_array_equal(alt["topk_idx"][t], base["topk_idx"][t])
    # groups: entries of unchanged rows keep their relative order within each expert
    for res in (base, alt):
        for e in range(ol.n_experts):
            ents = res["entries"][res["offsets"][e]:res["offsets"][e + 1]]
            assert list(ents) == sorted(ents)


def test_row_permutation_equivariance():
    ol, x = _layer_and_x(T=5, seed=4)
    perm = np.array([3, 0, 4, 1, 2])
    a = oracle.moe_window(x, ol)
    b = oracle.moe_window(x[perm], ol)
    np.testing.assert_array_equal(b["y"], a["y"][perm])
    np.testing.assert_array_equal(b["counts"], a["counts"])
    k = ol.top_k
    # entry t*k+j of the permuted window is entry perm[t]*k+j of the original
    for e in range(ol.n_experts):
        ea = set(a["entries"][a["offsets"][e]:a["offsets"][e + 1]])
        eb = b["entries"][b["offsets"][e]:b["offsets"][e + 1]]
        assert set(perm[t // k] * k + t % k for t in eb) == ea


def test_zeroed_shared_expert_removes_exactly_its_output():
    ol, x = _layer_and_x(T=3, seed=6)
    with_shared = oracle.moe_window(x, ol)
    z = lambda m: oracle.OQMat(m.codes, np.zeros_like(m.scale), np.zeros_like(m.min), m.rows, m.cols, m.bits, m.block)
    ol0 = oracle.OMoELayer(ol.n_experts, ol.top_k, ol.router_w, ol.router_b, ol.gate, ol.up, ol.down,
                           z(ol.shared_gate), z(ol.shared_up), z(ol.shared_down), ol.renorm)
    without = oracle.moe_window(x, ol0)
    for t in range(3):
        np.testing.assert_array_equal(oracle.shared_ffn(x[t], ol0), np.zeros(x.shape[1]))
        np.testing.assert_allclose(with_shared["y"][t] - without["y"][t], oracle.shared_ffn(x[t], ol),
                                   rtol=1e-12, atol=1e-15)


def test_group_rows_invariants():
    rng = np.random.default_rng(7)
    for T, k, E in [(1, 1, 1), (8, 8, 128), (8, 8, 16), (3, 2, 5)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        counts, offsets, entries, distinct = oracle.group_rows(idx, E)
        assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
        assert np.all(np.diff(offsets) >= 0)
        assert sorted(entries) == list(range(T * k))
        keys = [(idx[en // k, en % k], en) for en in entries]
        assert keys == sorted(keys)
        assert list(distinct) == sorted(set(idx.ravel()))
