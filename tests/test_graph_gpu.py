"""The window's bounded CUDA-graph cache, through the C ABI: graph replays
give the plain forward's bits for every T, a cache hit reuses the captured
graph with the new contents of x, and more keys than the cache holds evict
and recapture correctly."""
import numpy as np
import pytest
import torch

from slot_decode_window_gb300 import workloads as wlm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    wl = wlm.WORKLOADS["mid"]
    layer = wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, device="cuda")
    win = binding.Window(layer, max_rows=8)
    yield binding, wl, win
    win.close()


def test_graph_matches_forward_for_every_T(setup):
    B, wl, win = setup
    for T in range(1, 9):
        x = torch.from_numpy(wlm.make_window(wl, T, seed=0, window=100 + T)).cuda()
        y_ref = win.forward(x)
        y_g = torch.full_like(x, float("nan"))
        win.forward_graph(x, y_g)
        win.sync()
        assert torch.equal(y_ref, y_g), f"T={T}"


def test_cache_hit_reads_the_new_x(setup):
    B, wl, win = setup
    x = torch.empty(8, wl.moe.hidden, device="cuda")
    y = torch.empty_like(x)
    for w in range(3):  # same (T, x, y) key: one capture, three replays
        x.copy_(torch.from_numpy(wlm.make_window(wl, 8, seed=0, window=200 + w)))
        win.forward_graph(x, y)
        ref = win.forward(x)
        win.sync()
        assert torch.equal(ref, y)


def test_more_keys_than_the_cache_holds(setup):
    B, wl, win = setup
    x = torch.from_numpy(wlm.make_window(wl, 4, seed=0, window=300)).cuda()
    ref = win.forward(x)
    ys = [torch.full_like(x, float("nan")) for _ in range(20)]  # 20 keys > 16 cached graphs
    for y in ys:
        win.forward_graph(x, y)
    win.forward_graph(x, ys[0])  # evicted earlier: captured again
    win.sync()
    for y in ys:
        assert torch.equal(ref, y)
    with pytest.raises(B.StrataError):
        win.forward_graph(x[:0].reshape(0, wl.moe.hidden), ys[0][:0].reshape(0, wl.moe.hidden))
