"""GPU parity of the decoder stack with attention over each slot's KV cache
against the fp64 oracle in oracle/attention.py, through the C ABI.

Each window holds token / proposal row pairs of some slots (positions p and
p + 1) and single rows of others.  The caches hold fp16 history below the
window's positions and NaN everywhere the window must not read (positions past
each slot's last window row, and slots with no row), so any stray read shows
up as a non-finite output.  Routing must match the oracle bit for bit at every
layer on rows whose fp64 router margin stays >= 1e-3; y, q and k within
2e-3 x RMS; the entries the window appends within that tolerance plus fp16
rounding of the oracle's.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import MARGIN, odense, omoe, omoe_lazy

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def B():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    return binding


def _caches(wl, n_layers, n_slots, max_ctx, history, seed=0):
    """fp16 caches: N(0, 1) history below each slot's first window position, NaN elsewhere."""
    rng = np.random.default_rng(seed)
    shape = (n_layers, n_slots, wl.kv_heads, max_ctx, wl.head_dim)
    k = np.full(shape, np.nan, dtype=np.float16)
    v = np.full(shape, np.nan, dtype=np.float16)
    for s, h in history.items():
        k[:, s, :, :h, :] = rng.standard_normal((n_layers, wl.kv_heads, h, wl.head_dim)).astype(np.float16)
        v[:, s, :, :h, :] = rng.standard_normal((n_layers, wl.kv_heads, h, wl.head_dim)).astype(np.float16)
    return k, v


def _run(B, wl, n_layers, slots, positions, max_ctx, n_slots, lazy=False, seed=0):
    moe = [wlm.make_moe_layer(wl.moe, seed=seed, cfg_id=wl.cfg_id, layer=l, device="cuda") for l in range(n_layers)]
    dense = [wlm.make_dense_layer(wl, seed=seed, layer=l, device="cuda") for l in range(n_layers)]
    T = len(slots)
    history = {}
    for s, p in zip(slots, positions):
        history[s] = min(history.get(s, p), p)
    k, v = _caches(wl, n_layers, n_slots, max_ctx, history, seed)
    x = wlm.make_window(wl, T, seed=seed, window=300)
    kd, vd = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    stk = B.Stack(wl, moe, dense, max_rows=8)
    try:
        stk.set_kv(kd, vd, n_slots, max_ctx)
        sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
        ps = torch.tensor(positions, dtype=torch.int32, device="cuda")
        y, res = stk.forward(torch.from_numpy(x).cuda(), outputs=True, slot=sl, position=ps)
        stk.sync()
        y = y.cpu().numpy().astype(np.float64)
        kg, vg = kd.cpu().numpy(), vd.cpu().numpy()
        out = {n: t.cpu().numpy() for n, t in res.items()}
    finally:
        stk.close()
    # the oracle on fp64 copies of the same caches
    dense_o = [odense(dl, wl) for dl in dense]
    moe_o = [(omoe_lazy if lazy else omoe)(m) for m in moe]
    kcs = [k[l].astype(np.float64) for l in range(n_layers)]
    vcs = [v[l].astype(np.float64) for l in range(n_layers)]
    yo, Q, K, S, margin = oa.stack_window(x, dense_o, moe_o, kcs, vcs, slots, positions)
    return x, y, out, kg, vg, (yo, Q, K, S, margin, kcs, vcs)


def _compare(wl, n_layers, slots, positions, y, out, kg, vg, ref):
    yo, Q, K, S, margin, kcs, vcs = ref
    assert np.isfinite(y).all(), "a row read a cache entry it must not"
    rows = [t for t in range(len(slots)) if margin[t] >= MARGIN]
    assert rows, "no row kept a 1e-3 margin"
    idx = out["topk_idx"]
    for l in range(n_layers):
        for t in rows:
            np.testing.assert_array_equal(idx[l, t], S[l][t], err_msg=f"layer {l} row {t}")
    ref_y = yo[rows]
    rms = np.sqrt(np.mean(ref_y * ref_y))
    assert np.abs(y[rows] - ref_y).max() <= TOL * rms
    for name, g, r in (("q", out["q"], Q), ("k", out["k"], K)):
        for l in range(n_layers):
            rl = np.stack([r[l][t] for t in rows])
            e = np.abs(g[l][rows].astype(np.float64) - rl).max()
            assert e <= TOL * np.sqrt(np.mean(rl * rl)), f"{name} layer {l}"
    # the window's appended entries: the row's k and v (within the tolerance)
    # rounded to fp16 (within half an fp16 step more)
    for l in range(n_layers):
        for t in rows:
            s, p = slots[t], positions[t]
            for got, want in ((kg, kcs), (vg, vcs)):
                a = got[l, s, :, p, :].astype(np.float64)
                b = want[l][s, :, p, :]
                bound = TOL * np.sqrt(np.mean(b * b)) + 2.0 ** -10 * np.abs(b)
                assert np.all(np.abs(a - b) <= bound), f"appended entry: layer {l} row {t}"


SMALL = wlm.Workload("stack_kv_small", 95, wlm.MoESpec(256, 8, 2, 128, 128, 4, 32), (1,), n_layers=3,
                     heads=4, kv_heads=2, head_dim=64)


@pytest.mark.parametrize("slots,positions", [
    ([0, 0, 1, 2, 2], [17, 18, 5, 130, 131]),          # two token/proposal pairs and a single row
    ([3], [0]),                                        # a fresh slot: its own entry only
    ([1, 1, 0, 0, 2, 2, 3, 3], [63, 64, 0, 1, 190, 191, 64, 65]),  # 4 pairs, chunk edges
])
def test_small_stack_with_caches(B, slots, positions):
    x, y, out, kg, vg, ref = _run(B, SMALL, 3, slots, positions, max_ctx=200, n_slots=4)
    _compare(SMALL, 3, slots, positions, y, out, kg, vg, ref)


def test_stack48_shapes_three_layers_with_caches(B):
    """The 48-layer stack's layer shapes (d 2048, 32 / 4 heads of 128, 128
    experts top-8), three layers, a T = 8 window of 4 slots x (token, proposal)
    at positions up to ~1000."""
    base = wlm.WORKLOADS["stack48"]
    wl = wlm.Workload("stack48", base.cfg_id, base.moe, (8,), n_layers=3)
    slots = [0, 0, 1, 1, 2, 2, 3, 3]
    positions = [900, 901, 37, 38, 511, 512, 1000, 1001]
    x, y, out, kg, vg, ref = _run(B, wl, 3, slots, positions, max_ctx=1024, n_slots=5, lazy=True)
    _compare(wl, 3, slots, positions, y, out, kg, vg, ref)


def test_a_row_out_of_range_reports_edevice(B):
    moe = [wlm.make_moe_layer(SMALL.moe, seed=0, cfg_id=SMALL.cfg_id, layer=l, device="cuda") for l in range(1)]
    dense = [wlm.make_dense_layer(SMALL, seed=0, layer=l, device="cuda") for l in range(1)]
    wl = wlm.Workload("stack_kv_small1", 95, SMALL.moe, (1,), n_layers=1, heads=4, kv_heads=2, head_dim=64)
    stk = B.Stack(wl, moe, dense, max_rows=8)
    try:
        k = torch.zeros(1, 2, 2, 16, 64, dtype=torch.float16, device="cuda")
        v = torch.zeros_like(k)
        stk.set_kv(k, v, 2, 16)
        x = torch.from_numpy(wlm.make_window(wl, 2, seed=0, window=1)).cuda()
        y = torch.zeros_like(x)
        sl = torch.tensor([0, 5], dtype=torch.int32, device="cuda")   # slot 5 of 2
        ps = torch.tensor([3, 3], dtype=torch.int32, device="cuda")
        assert B.strata_stack_forward_kv(stk.handle, x.data_ptr(), 2, y.data_ptr(), sl.data_ptr(),
                                         ps.data_ptr()) == B.STRATA_OK
        assert B.strata_stack_sync(stk.handle) == B.STRATA_EDEVICE
        assert bool(torch.isfinite(y).all())
        # without caches set, the call is refused before any launch
        stk.set_kv(None, None, 0, 0)
        assert B.strata_stack_forward_kv(stk.handle, x.data_ptr(), 2, y.data_ptr(), sl.data_ptr(),
                                         ps.data_ptr()) == B.STRATA_EINVAL
    finally:
        stk.close()
