"""GPU parity of the adaptive tier's bookkeeping against the fp32 oracle in
oracle/tier.py, through the C ABI: after every window the device's counters
are bitwise the oracle's, and the tier's experts, the last round's swaps and
the window/round counts are equal.  The per-window expert counts fed to the
oracle come from the fp64 oracle's own routing of the same rows (routing is
bit-exact against it, as the parity tests check)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import tier as ot
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import margin_accept, omoe, small_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    return binding


def _oracle_counts(x, ol):
    idx = np.stack([oracle.router(x[t], ol.router_w, ol.router_b, ol.top_k, ol.renorm)[2] for t in range(x.shape[0])])
    return oracle.group_rows(idx, ol.n_experts)[0]


def _compare(B, tier, st, E):
    rc, got = B.strata_tier_read(tier, E)
    assert rc == B.STRATA_OK
    np.testing.assert_array_equal(got["counters"], st.counters)
    np.testing.assert_array_equal(got["resident"].astype(bool), st.resident)
    assert got["windows"] == st.windows and got["rounds"] == st.rounds
    assert list(zip(got["swap_in"].tolist(), got["swap_out"].tolist())) == st.last_swaps


@pytest.mark.parametrize("name,spec,kw", [
    ("small", small_spec(hidden=256, n_experts=16, top_k=3, ffn=128, shared_ffn=128),
     dict(capacity=5, adapt_every=2, adapt_swaps=3, decay=0.5, min_gain=1.5)),
    ("mid", None, dict(capacity=40, adapt_every=4, adapt_swaps=8, decay=0.75, min_gain=1.5)),
])
def test_tier_matches_oracle_window_by_window(B, name, spec, kw):
    if spec is None:
        wl = wlm.WORKLOADS[name]
        spec, cfg = wl.moe, wl.cfg_id
    else:
        wl, cfg = wlm.Workload("custom", 77, spec, (1,)), 77
    layer = wlm.make_moe_layer(spec, seed=2, cfg_id=cfg, device="cuda")
    ol = omoe(layer)
    win = B.Window(layer, max_rows=8)
    E = spec.n_experts
    st_c, tier = B.strata_tier_create(B.strata_tier_desc(E, **kw))
    assert st_c == B.STRATA_OK
    try:
        assert B.strata_window_set_tier(win.handle, tier) == B.STRATA_OK
        st = ot.tier_init(E, kw["capacity"])
        rng = np.random.default_rng(5)
        for w in range(14):
            T = int(rng.integers(1, 9))
            x = wlm.make_window(wl, T, seed=2, window=100 + w, accept_row=margin_accept(ol))
            xt = torch.from_numpy(x).cuda()
            y = torch.empty_like(xt)
            # the three entry points all update the tier
            if w % 3 == 0:
                win.forward(xt, y)
            elif w % 3 == 1:
                assert B.strata_moe_window_forward_noalloc(win.handle, xt.data_ptr(), T, y.data_ptr()) == B.STRATA_OK
            else:
                win.forward_graph(xt, y)
            assert B.strata_window_sync(win.handle) == B.STRATA_OK
            ot.tier_window(st, _oracle_counts(x, ol), kw["adapt_every"], kw["adapt_swaps"], kw["decay"],
                           kw["min_gain"])
            _compare(B, tier, st, E)
        assert st.rounds >= 3
        # detached: windows no longer touch it
        assert B.strata_window_set_tier(win.handle, None) == B.STRATA_OK
        win.forward(torch.from_numpy(wlm.make_window(wl, 4, seed=2, window=999)).cuda())
        win.sync()
        _compare(B, tier, st, E)
    finally:
        win.close()
        B.strata_tier_destroy(tier)


def test_tier_rejects_a_handle_of_another_expert_count(B):
    spec = small_spec(hidden=256, n_experts=8, top_k=2, ffn=128, shared_ffn=0)
    layer = wlm.make_moe_layer(spec, seed=0, cfg_id=77, device="cuda")
    win = B.Window(layer, max_rows=8)
    st, tier = B.strata_tier_create(B.strata_tier_desc(9, 3, 1, 1, 0.5, 1.5))
    try:
        assert st == B.STRATA_OK
        assert B.strata_window_set_tier(win.handle, tier) == B.STRATA_EINVAL
    finally:
        B.strata_tier_destroy(tier)
        win.close()
