"""The window's failure paths on the GPU, made on the host side only.

Nothing here faults, traps or hangs a GPU.  Errors come from host-made
inputs (a row of NaNs), from the test hook that fails a launch before any
CUDA call (STRATA_FAULT=launch), and from a grid barrier told to wait for an
arrival that never comes, with the device's wait limit shortened to about a
millisecond (STRATA_TEST_BARRIER_EXTRA, STRATA_WAIT_CYCLES, both read when
a handle is created): every CTA then gives up after the limit, records the
error and returns, and the next strata_window_sync reports EDEVICE.
"""
import os
import time

import numpy as np
import pytest
import torch

import oracle
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import margin_accept, omoe, small_spec

pytestmark = pytest.mark.gpu

TOL = 2e-3
# the 2-bit layer of the warp-streamed path (as in test_parity_gpu.py)
WIDE2 = small_spec(hidden=1024, n_experts=12, top_k=4, ffn=1024, shared_ffn=1024, bits=2, block=16)


@pytest.fixture(scope="module")
def B():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    return binding


def _layer(spec=None, name=None, seed=0):
    if name is not None:
        wl = wlm.WORKLOADS[name]
        spec, cfg_id = wl.moe, wl.cfg_id
    else:
        wl, cfg_id = wlm.Workload("custom", 77, spec, (1,)), 77
    layer = wlm.make_moe_layer(spec, seed=seed, cfg_id=cfg_id, device="cuda")
    return wl, layer, omoe(layer)


def _window_with_env(B, layer, env):
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return B.Window(layer, max_rows=8)
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def _rows_within_tolerance(y, ref, rows):
    yr = ref["y"][rows]
    rms = np.sqrt(np.mean(yr * yr))
    assert np.abs(y[rows] - yr).max() <= TOL * rms


@pytest.mark.parametrize("which", ["mid", "wide2"])
def test_nan_row_reports_edevice_and_spares_the_other_rows(B, which):
    """A row of NaNs gives non-finite router logits: the window still runs to
    the end, the next sync reports EDEVICE, the other rows are unaffected, and
    the handle serves the next window normally."""
    wl, layer, ol = _layer(name="mid") if which == "mid" else _layer(spec=WIDE2)
    win = B.Window(layer, max_rows=8)
    try:
        x = wlm.make_window(wl, 6, seed=0, window=7, accept_row=margin_accept(ol))
        xn = x.copy()
        xn[2] = np.nan
        y = torch.full((6, x.shape[1]), 0.0, device="cuda")
        xt = torch.from_numpy(xn).cuda()
        assert B.strata_moe_window_forward(win.handle, xt.data_ptr(), 6, y.data_ptr()) == B.STRATA_OK
        assert B.strata_window_sync(win.handle) == B.STRATA_EDEVICE
        assert B.strata_window_sync(win.handle) == B.STRATA_OK  # the error was reported once and cleared
        yn = y.cpu().numpy().astype(np.float64)
        ref = oracle.moe_window(x, ol, rows=[0, 1, 3, 4, 5])
        _rows_within_tolerance(yn, ref, [0, 1, 3, 4, 5])
        # the next window on the same handle is clean and matches the oracle
        y2 = win.forward(torch.from_numpy(x).cuda())
        assert B.strata_window_sync(win.handle) == B.STRATA_OK
        _rows_within_tolerance(y2.cpu().numpy().astype(np.float64), oracle.moe_window(x, ol), list(range(6)))
    finally:
        win.close()


@pytest.mark.parametrize("which", ["tiny", "wide2"])
def test_grid_barrier_wait_runs_out_and_reports_edevice(B, which):
    """A barrier that waits for one arrival too many gives up after the short
    limit (~1 ms at GB300 clocks): the call returns, sync reports EDEVICE, and
    the context stays usable (a normal handle afterwards matches the oracle)."""
    wl, layer, ol = _layer(name="tiny") if which == "tiny" else _layer(spec=WIDE2)
    bad = _window_with_env(B, layer, {"STRATA_WAIT_CYCLES": "2000000", "STRATA_TEST_BARRIER_EXTRA": "1"})
    x = wlm.make_window(wl, 4, seed=0, window=3, accept_row=margin_accept(ol))
    xt = torch.from_numpy(x).cuda()
    y = torch.zeros_like(xt)
    try:
        t0 = time.perf_counter()
        assert B.strata_moe_window_forward(bad.handle, xt.data_ptr(), 4, y.data_ptr()) == B.STRATA_OK
        assert B.strata_window_sync(bad.handle) == B.STRATA_EDEVICE
        assert time.perf_counter() - t0 < 10.0
        # every later window on this handle gives up the same way
        assert B.strata_moe_window_forward(bad.handle, xt.data_ptr(), 4, y.data_ptr()) == B.STRATA_OK
        assert B.strata_window_sync(bad.handle) == B.STRATA_EDEVICE
    finally:
        bad.close()
    good = B.Window(layer, max_rows=8)
    try:
        yg = good.forward(xt)
        assert B.strata_window_sync(good.handle) == B.STRATA_OK
        _rows_within_tolerance(yg.cpu().numpy().astype(np.float64), oracle.moe_window(x, ol), list(range(4)))
    finally:
        good.close()


def test_stack_barrier_wait_runs_out_and_reports_edevice(B):
    from slot_decode_window_gb300.binding import Stack
    wl = wlm.Workload("stack_small_fail", 93, wlm.MoESpec(256, 8, 2, 128, 128, 4, 32), (1,), n_layers=2,
                      heads=4, kv_heads=2, head_dim=64)
    moe = [wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, layer=l, device="cuda") for l in range(2)]
    dense = [wlm.make_dense_layer(wl, seed=0, layer=l, device="cuda") for l in range(2)]
    env = {"STRATA_WAIT_CYCLES": "2000000", "STRATA_TEST_BARRIER_EXTRA": "1"}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        stk = Stack(wl, moe, dense, max_rows=8)
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v
    try:
        x = torch.from_numpy(wlm.make_window(wl, 3, seed=0, window=1)).cuda()
        y = torch.zeros_like(x)
        assert B.strata_stack_forward(stk.handle, x.data_ptr(), 3, y.data_ptr()) == B.STRATA_OK
        assert B.strata_stack_sync(stk.handle) == B.STRATA_EDEVICE
    finally:
        stk.close()


def test_launch_fault_hook_returns_ecuda_and_launches_nothing(B):
    wl, layer, ol = _layer(name="tiny")
    win = B.Window(layer, max_rows=8)
    try:
        x = torch.from_numpy(wlm.make_window(wl, 2, seed=0, window=1)).cuda()
        y = torch.full_like(x, 7.0)
        os.environ["STRATA_FAULT"] = "launch"
        try:
            st = B.strata_moe_window_forward(win.handle, x.data_ptr(), 2, y.data_ptr())
        finally:
            del os.environ["STRATA_FAULT"]
        assert st == B.STRATA_ECUDA
        assert B.strata_window_sync(win.handle) == B.STRATA_OK
        assert bool((y == 7.0).all())
    finally:
        win.close()
