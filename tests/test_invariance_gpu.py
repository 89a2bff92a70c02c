"""A row's output does not depend on the window it is in, bit for bit.

The Strata docs ("BATCHING.md", section "Exactness") state that a batch row's
arithmetic is the single-token window's, and warn that rounding which depends
on how many rows share an expert breaks that.  Here every row of windows of
T = 1..8 rows (including windows where the same row appears several times, so
that its experts' groups are as large as they get) must be torch.equal to the
same row run alone, on the ring path (4-bit d = 2048), the warp-streamed path
for 4-bit (d = 4096) and 2-bit layers, and a small layer.
"""
import numpy as np
import pytest
import torch

from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import small_spec

pytestmark = pytest.mark.gpu

WIDE2 = small_spec(hidden=1024, n_experts=12, top_k=4, ffn=1024, shared_ffn=1024, bits=2, block=16)


@pytest.fixture(scope="module")
def B():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    return binding


def _win(B, name=None, spec=None):
    if name is not None:
        wl = wlm.WORKLOADS[name]
        spec, cfg = wl.moe, wl.cfg_id
    else:
        wl, cfg = wlm.Workload("custom", 77, spec, (1,)), 77
    layer = wlm.make_moe_layer(spec, seed=0, cfg_id=cfg, device="cuda")
    return wl, B.Window(layer, max_rows=8)


def _alone(win, rows):
    out = []
    for r in rows:
        out.append(win.forward(r.unsqueeze(0).contiguous())[0].clone())
    win.sync()
    return out


@pytest.mark.parametrize("which", ["mid", "zipf", "lowbit", "tiny", "wide2"])
def test_rows_are_bitwise_their_single_row_windows(B, which):
    wl, win = _win(B, name=which) if which != "wide2" else _win(B, spec=WIDE2)
    try:
        d = wl.moe.hidden
        pool = torch.from_numpy(np.stack([wlm.hidden_row(0, wl.cfg_id, 700, t, 0, d) for t in range(8)])).cuda()
        alone = _alone(win, pool)
        rng = np.random.default_rng(1)
        windows = [list(range(T)) for T in range(1, 9)]                       # rows 0..T-1
        windows += [list(rng.permutation(8)[:T]) for T in (3, 5, 8)]          # other orders
        windows += [[2] * 8, [5, 5, 5, 1, 1, 5, 5, 1], [0, 7, 0, 7]]         # repeated rows: big groups
        for idx in windows:
            x = pool[idx].contiguous()
            y = win.forward(x)
            win.sync()
            for pos, r in enumerate(idx):
                assert torch.equal(y[pos], alone[r]), f"{which}: window {idx}, row {r} at {pos}"
    finally:
        win.close()
