"""GPU parity of the window step against the fp64 oracle, through the C ABI.

Routing (selected experts, counts, offsets, grouped entries, distinct experts)
must match bit for bit; inputs keep every row's top-k logit margin >= 1e-3 so
fp32 and fp64 logits order the experts alike.  Outputs must satisfy
max|y - y_oracle| <= 2e-3 * RMS(y_oracle) over the compared rows.
"""
import numpy as np
import pytest
import torch

import oracle
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import margin_accept, omoe, small_spec

pytestmark = pytest.mark.gpu

TOL = 2e-3
_cache = {}
_pool = {}


@pytest.fixture(scope="module", autouse=True)
def lib():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    yield
    if "p" in _pool:
        _pool.pop("p").shutdown()


def _oracle_pool():
    """A spawn-started process pool for the full-size oracle checks (made on first use)."""
    if "p" not in _pool:
        from tests import oracle_lean
        _pool["p"] = oracle_lean.spawn_pool()
    return _pool["p"]


def _setup(name=None, spec=None, seed=0, max_rows=8):
    key = (name, spec, seed, max_rows)
    if key not in _cache:
        from slot_decode_window_gb300.binding import Window
        if name is not None:
            wl = wlm.WORKLOADS[name]
            spec, cfg_id = wl.moe, wl.cfg_id
        else:
            wl, cfg_id = wlm.Workload("custom", 77, spec, (1,)), 77
        layer = wlm.make_moe_layer(spec, seed=seed, cfg_id=cfg_id, device="cuda")
        ol = omoe(layer)
        win = Window(layer, max_rows=max_rows)
        _cache.clear()  # keep one big layer resident at a time
        _cache[key] = (wl, layer, ol, win)
    return _cache[key]


def _run(win, x):
    xt = torch.from_numpy(x).cuda()
    y, rt = win.forward(xt, routing=True)
    win.sync()
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64), {k: v.cpu().numpy() for k, v in rt.items()}


def _check(win, ol, x, rows=None, lean=False):
    """Routing bit-exact and y within tolerance on ``rows`` (all rows when None).
    ``lean``: the oracle's expert-by-expert evaluation (bitwise the same
    results, for full-size layers whose experts do not all fit a cache)."""
    y, rt = _run(win, x)
    if lean:
        from tests import oracle_lean
        ref = oracle_lean.moe_window(x, ol, pool=_oracle_pool())
    else:
        ref = oracle.moe_window(x, ol, rows=rows)
    np.testing.assert_array_equal(rt["topk_idx"], ref["topk_idx"])
    np.testing.assert_array_equal(rt["counts"], ref["counts"])
    np.testing.assert_array_equal(rt["offsets"], ref["offsets"])
    np.testing.assert_array_equal(rt["entries"], ref["entries"])
    nd = int(rt["n_distinct"][0])
    assert nd == ref["n_distinct"]
    np.testing.assert_array_equal(rt["distinct"][:nd], ref["distinct"])
    np.testing.assert_allclose(rt["topk_w"], ref["topk_w"], rtol=2e-5, atol=1e-7)
    sel = list(range(x.shape[0])) if rows is None else list(rows)
    yr = ref["y"][sel]
    err = np.abs(y[sel] - yr).max()
    rms = np.sqrt(np.mean(yr * yr))
    assert np.isfinite(y[sel]).all()
    assert err <= TOL * rms, f"max err {err:.3e} > {TOL} * rms {rms:.3e}"
    return y, err / rms


def _window(wl, ol, T, window=0, seed=0):
    return wlm.make_window(wl, T, seed=seed, window=window, accept_row=margin_accept(ol))


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_tiny(T):
    wl, layer, ol, win = _setup("tiny")
    for w in range(3):
        _check(win, ol, _window(wl, ol, T, window=w))


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_mid_full_rows(T):
    wl, layer, ol, win = _setup("mid")
    _check(win, ol, _window(wl, ol, T, window=T))


def test_zipf_mtp_pairs_all_rows():
    """The Zipf-biased layer at its full size: 4 slots x (token, MTP proposal), every row."""
    wl, layer, ol, win = _setup("zipf")
    x = _window(wl, ol, 8)
    _check(win, ol, x, lean=True)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_lowbit_all_rows(T):
    """The 2-bit d=4096 layer with 256 experts at every window size it is run at, every row."""
    wl, layer, ol, win = _setup("lowbit")
    _check(win, ol, _window(wl, ol, T, window=T), lean=True)


@pytest.mark.parametrize("spec", [
    small_spec(hidden=256, ffn=128, shared_ffn=0, n_experts=4, top_k=4),           # k = E, no shared expert
    small_spec(hidden=256, ffn=192, shared_ffn=64, n_experts=16, top_k=1),         # k = 1, widths differ
    small_spec(hidden=256, ffn=128, shared_ffn=128, n_experts=1, top_k=1),         # a single expert
    small_spec(hidden=384, ffn=256, shared_ffn=128, n_experts=12, top_k=3, renorm_topk=1),
    small_spec(hidden=512, ffn=256, shared_ffn=384, n_experts=10, top_k=4, bits=2, block=16),
])
@pytest.mark.parametrize("T", [1, 4, 7])
def test_edge_shapes(spec, T):
    wl, layer, ol, win = _setup(spec=spec, seed=3)
    _check(win, ol, _window(wl, ol, T, window=T))


def test_all_rows_one_expert_and_max_group():
    """Every row routes to the same experts (groups of 8 rows: the unpaired path)."""
    spec = small_spec(hidden=256, ffn=128, shared_ffn=128, n_experts=8, top_k=2)
    wl, layer, ol, win = _setup(spec=spec, seed=4)
    base = _window(wl, ol, 1)[0]
    rng = np.random.default_rng(0)
    rows = [base]
    while len(rows) < 8:
        r = (base + rng.normal(0, 1e-3, base.shape)).astype(np.float32)
        if margin_accept(ol)(r):
            rows.append(r)
    x = np.stack(rows)
    y, _ = _check(win, ol, x)
    ref = oracle.moe_window(x, ol)
    assert ref["n_distinct"] == 2


def test_repeat_is_bitwise_deterministic():
    wl, layer, ol, win = _setup("mid")
    x = _window(wl, ol, 8, window=11)
    y1, _ = _run(win, x)
    y2, _ = _run(win, x)
    np.testing.assert_array_equal(y1, y2)


def test_window_rows_equal_single_rows_within_tolerance():
    """A row computed inside an 8-row window matches the same row alone."""
    wl, layer, ol, win = _setup("mid")
    x = _window(wl, ol, 8, window=12)
    y8, _ = _run(win, x)
    for t in (0, 7):
        y1, _ = _run(win, x[t:t + 1])
        rms = np.sqrt(np.mean(y1 * y1))
        assert np.abs(y8[t] - y1[0]).max() <= TOL * rms


def test_forward_argument_errors_on_device_handle():
    from slot_decode_window_gb300 import binding as B
    wl, layer, ol, win = _setup("tiny", max_rows=4)
    x = torch.zeros(8, wl.moe.hidden, device="cuda")
    y = torch.zeros_like(x)
    assert B.strata_moe_window_forward(win.handle, x.data_ptr(), 5, y.data_ptr()) == B.STRATA_EINVAL
    assert B.strata_moe_window_forward(win.handle, x.data_ptr(), 0, y.data_ptr()) == B.STRATA_EINVAL
    assert B.strata_moe_window_forward(win.handle, x.data_ptr(), 2, x[1].data_ptr()) == B.STRATA_EINVAL
    st, info = B.strata_window_query(win.handle)
    assert st == B.STRATA_OK and info.n_sm > 0 and info.stages >= 2 and info.smem_bytes > 0
    assert info.expert_bytes == layer.expert_bytes and info.shared_bytes == layer.shared_bytes
    assert B.strata_window_sync(win.handle) == B.STRATA_OK


# A 2-bit layer large enough for the warp-streamed window path (every warp
# gets at least one 128-column k-step of each task: d, F and the shared width
# of at least 8 k-steps), small enough for full oracle checks; shared routing
# (few experts) mixes one- and many-row groups in the same window.
WIDE2 = small_spec(hidden=1024, n_experts=12, top_k=4, ffn=1024, shared_ffn=1024, bits=2, block=16)


@pytest.mark.parametrize("T", [1, 3, 6, 8])
def test_two_bit_streamed_path(T):
    wl, layer, ol, win = _setup(spec=WIDE2)
    assert win.info().stages == 1  # the warp-streamed configuration holds no stage ring
    _check(win, ol, _window(wl, ol, T, window=T))


def test_two_bit_streamed_path_entry_points_agree():
    from slot_decode_window_gb300 import binding as B
    wl, layer, ol, win = _setup(spec=WIDE2)
    for T in (2, 8):
        x = torch.from_numpy(_window(wl, ol, T, window=50 + T)).cuda()
        y0 = win.forward(x)
        yg = torch.empty_like(x)
        win.forward_graph(x, yg)
        yn = torch.full_like(x, float("nan"))
        assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), T, yn.data_ptr()) == B.STRATA_OK
        win.sync()
        assert torch.equal(y0, yg)
        assert torch.equal(y0, yn)


# A 4-bit layer at the smallest width where every warp of the warp-streamed
# path gets a 64-column k-step of each task.  At this width the ring is long,
# so the handle would take the ring path; STRATA_WINDOW_DIRECT=1 at creation
# forces the warp-streamed one (which 4-bit layers take when their activations
# leave a short ring, as at d = 4096).
WIDE4 = small_spec(hidden=512, n_experts=12, top_k=4, ffn=512, shared_ffn=512)


def _forced_direct(spec, seed=5):
    import os
    os.environ["STRATA_WINDOW_DIRECT"] = "1"
    try:
        return _setup(spec=spec, seed=seed)
    finally:
        del os.environ["STRATA_WINDOW_DIRECT"]


@pytest.mark.parametrize("T", [1, 3, 6, 8])
def test_four_bit_streamed_path(T):
    wl, layer, ol, win = _forced_direct(WIDE4)
    assert win.info().stages == 1
    _check(win, ol, _window(wl, ol, T, window=T))


def test_four_bit_paths_agree_and_wide_layer_streams():
    """The forced warp-streamed handle and a ring handle of the same layer agree
    within the tolerance; a d = 4096 4-bit layer takes the streamed path."""
    from slot_decode_window_gb300.binding import Window
    wl, layer, ol, win = _forced_direct(WIDE4)
    ring = Window(layer, max_rows=8)
    try:
        assert ring.info().stages >= 2
        x = torch.from_numpy(_window(wl, ol, 8, window=21)).cuda()
        yd, yr = win.forward(x), ring.forward(x)
        win.sync()
        ring.sync()
        rms = float(torch.sqrt(torch.mean(yr.double() ** 2)))
        assert float((yd - yr).abs().max()) <= TOL * rms
    finally:
        ring.close()
    wz, _, _, winz = _setup("zipf")
    assert winz.info().stages == 1
