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


def test_noalloc_alternates_between_two_layer_shapes(B):
    """Calls on two handles of different width and bit width take turns on the
    one shared array; each matches its own handle's regular forward (bit for
    bit: the same kernel runs on the same inputs), so what one shape leaves in
    the array never leaks into the other's window."""
    from tests.helpers import small_spec
    wide2 = small_spec(hidden=1024, n_experts=12, top_k=4, ffn=1024, shared_ffn=1024, bits=2, block=16)
    wl_a = wlm.WORKLOADS["mid"]
    wl_b = wlm.Workload("custom", 77, wide2, (1,))
    win_a = B.Window(wlm.make_moe_layer(wl_a.moe, seed=0, cfg_id=wl_a.cfg_id, device="cuda"), max_rows=8)
    win_b = B.Window(wlm.make_moe_layer(wide2, seed=0, cfg_id=77, device="cuda"), max_rows=8)
    try:
        for i, (wl, win, T) in enumerate(((wl_a, win_a, 8), (wl_b, win_b, 5), (wl_a, win_a, 2), (wl_b, win_b, 8))):
            x = torch.from_numpy(wlm.make_window(wl, T, seed=0, window=60 + i)).cuda()
            y_ref = torch.empty_like(x)
            y_na = torch.full_like(x, float("nan"))
            assert B.strata_moe_window_forward(win.handle, x.data_ptr(), T, y_ref.data_ptr()) == B.STRATA_OK
            assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), T, y_na.data_ptr()) == B.STRATA_OK
            assert B.strata_window_sync(win.handle) == B.STRATA_OK
            assert torch.equal(y_ref, y_na), f"call {i}"
    finally:
        win_a.close()
        win_b.close()


def test_noalloc_rejects_a_shape_beyond_its_scratch(B):
    # d = F = 8192: the down outputs (64 entries x 8192 x 4 B) and the h
    # fragments (64 x 2 x 8192 x 2 B) alone fill the 4 MiB array, and the
    # window needs x fragments, partial logits and counters besides
    spec = wlm.MoESpec(8192, 1, 1, 8192, 0, 4, 32)
    layer = wlm.make_moe_layer(spec, seed=0, cfg_id=78, device="cuda")
    win = B.Window(layer, max_rows=4)
    assert 64 * 8192 * 4 + 64 * 2 * 8192 * 2 >= B.NOALLOC_SCRATCH_BYTES
    x = torch.zeros(1, 8192, device="cuda")
    y = torch.zeros_like(x)
    assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), 1, y.data_ptr()) == B.STRATA_EUNSUPPORTED
    assert B.strata_moe_window_forward_noalloc(win.handle, x.data_ptr(), 0, y.data_ptr()) == B.STRATA_EINVAL
    win.close()
