"""The window entry point that allocates nothing (its scratch is one static
device array) against the regular entry point, through the C ABI.  The file
name keeps it last in collection; it also passes when run alone."""
import numpy as np
import pytest
import torch

from slot_decode_window_gb300 import workloads as wlm

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def B():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    return binding


def test_noalloc_matches_forward_on_two_calls_in_a_row(B):
    wl = wlm.WORKLOADS["mid"]
    layer = wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, device="cuda")
    win = B.Window(layer, max_rows=8)
    for w, T in enumerate((8, 3)):
        x = torch.from_numpy(wlm.make_window(wl, T, seed=0, window=40 + w)).cuda()
        y_ref = torch.empty_like(x)
        y_na = torch.full_like(x, float("nan"))
        assert B.strata_moe_window_forward(win.handle, x.data_ptr(), T, y_ref.data_ptr()) == B.STRATA_OK
        assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), T, y_na.data_ptr()) == B.STRATA_OK
        assert B.strata_window_sync(win.handle) == B.STRATA_OK
        torch.cuda.synchronize()
        ref = y_ref.cpu().numpy().astype(np.float64)
        got = y_na.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        rms = np.sqrt(np.mean(ref * ref))
        assert np.abs(got - ref).max() <= TOL * rms
    win.close()


def test_noalloc_rejects_a_shape_beyond_its_scratch(B):
    # d = F = 8192: the down outputs (64 entries x 8192 x 4 B) and the h
    # fragments (64 x 2 x 8192 x 2 B) together exceed the 4 MiB array
    spec = wlm.MoESpec(8192, 1, 1, 8192, 0, 4, 32)
    layer = wlm.make_moe_layer(spec, seed=0, cfg_id=78, device="cuda")
    win = B.Window(layer, max_rows=4)
    assert win.info().workspace_bytes > B.NOALLOC_SCRATCH_BYTES
    x = torch.zeros(1, 8192, device="cuda")
    y = torch.zeros_like(x)
    assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), 1, y.data_ptr()) == B.STRATA_EUNSUPPORTED
    assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), 0, y.data_ptr()) == B.STRATA_EINVAL
    win.close()
