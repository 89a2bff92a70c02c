"""The seeded input generator: determinism, shapes, margins, row recipes (no GPU)."""
import numpy as np
import torch

import oracle
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import MARGIN, margin_accept, omoe


def test_deterministic_and_seed_sensitive():
    spec = wlm.WORKLOADS["tiny"].moe
    a = wlm.make_moe_layer(spec, seed=0, cfg_id=1)
    b = wlm.make_moe_layer(spec, seed=0, cfg_id=1)
    c = wlm.make_moe_layer(spec, seed=1, cfg_id=1)
    assert torch.equal(a.gate.codes, b.gate.codes) and torch.equal(a.router_w, b.router_w)
    assert not torch.equal(a.gate.codes, c.gate.codes)
    assert not torch.equal(a.gate.codes[0], a.gate.codes[1])


def test_shapes_of_tiny():
    wl = wlm.WORKLOADS["tiny"]
    L = wlm.make_moe_layer(wl.moe, cfg_id=wl.cfg_id)
    s = wl.moe
    assert L.gate.codes.shape == (s.n_experts, s.ffn, s.hidden // 2)
    assert L.down.scale.shape == (s.n_experts, s.hidden, s.ffn // 32)
    assert L.shared_down.codes.shape == (1, s.hidden, s.shared_ffn // 2)
    assert L.expert_bytes == 3 * s.ffn * s.hidden * 5 // 8


def test_weights_are_normal_002():
    w = wlm._normal((256, 256), wlm.WEIGHT_STD, 5, "cpu")
    assert abs(float(w.std()) - 0.02) < 0.001 and abs(float(w.mean())) < 0.001


def test_windows_respect_margin():
    wl = wlm.WORKLOADS["tiny"]
    ol = omoe(wlm.make_moe_layer(wl.moe, cfg_id=wl.cfg_id))
    x = wlm.make_window(wl, 8, seed=0, window=3, accept_row=margin_accept(ol))
    for r in x:
        assert oracle.topk_margin(r, ol.router_w, ol.router_b, ol.top_k) >= MARGIN
    assert x.dtype == np.float32 and x.shape == (8, wl.moe.hidden)


def test_mtp_pairs_recipe():
    wl = wlm.Workload("pairs", 9, wlm.MoESpec(512, 8, 2, 64, 64, 4, 32), (8,), mtp_pairs=True)
    x = wlm.make_window(wl, 8)
    noise = x[1::2] - x[0::2]
    assert abs(float(noise.std()) - 0.1) < 0.01
    assert abs(float(x[0::2].std()) - 1.0) < 0.05


def test_zipf_bias_is_log_zipf_permutation():
    b = wlm.zipf_bias(160, 1.1, 7)
    ranks = np.exp(-b.astype(np.float64) / 1.1)
    np.testing.assert_allclose(np.sort(ranks), np.arange(1, 161), rtol=1e-5)
