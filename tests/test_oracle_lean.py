"""The expert-by-expert evaluation in tests/oracle_lean.py is bitwise the
oracle's per-row evaluation (no GPU)."""
import numpy as np
import pytest

import oracle
from slot_decode_window_gb300 import workloads as wlm
from tests import oracle_lean
from tests.helpers import odense, omoe, small_spec, stack_trajectory


@pytest.mark.parametrize("spec", [
    small_spec(),
    small_spec(hidden=128, n_experts=5, top_k=3, ffn=64, shared_ffn=0, renorm_topk=1),
    small_spec(hidden=256, n_experts=7, top_k=2, ffn=128, shared_ffn=128, bits=2, block=16),
])
def test_lean_window_equals_oracle_window(spec):
    layer = wlm.make_moe_layer(spec, seed=1, cfg_id=90)
    ol = omoe(layer)
    wl = wlm.Workload("custom", 90, spec, (1,))
    x = wlm.make_window(wl, 6, seed=1, window=2)
    ref = oracle.moe_window(x, ol)
    got = oracle_lean.moe_window(x, ol)
    for k in ("y", "topk_idx", "topk_w", "counts", "offsets", "entries", "distinct"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    assert got["n_distinct"] == ref["n_distinct"]


def test_lean_stack_equals_oracle_trajectories_with_a_spawn_pool():
    wl = wlm.Workload("stack_lean", 94, wlm.MoESpec(128, 6, 2, 64, 64, 4, 32), (1,), n_layers=2,
                      heads=4, kv_heads=2, head_dim=32)
    moe = [omoe(wlm.make_moe_layer(wl.moe, seed=0, cfg_id=wl.cfg_id, layer=l)) for l in range(2)]
    dense = [odense(wlm.make_dense_layer(wl, seed=0, layer=l, device="cpu"), wl) for l in range(2)]
    x = wlm.make_window(wl, 3, seed=0, window=4)
    with oracle_lean.spawn_pool(2) as pool:
        got = oracle_lean.stack_rows(x, dense, moe, pool=pool)
    for t in range(3):
        ref = stack_trajectory(x[t], dense, moe)
        np.testing.assert_array_equal(got[t][0], ref[0])
        for a, b in zip(got[t][1] + got[t][2] + got[t][3], ref[1] + ref[2] + ref[3]):
            np.testing.assert_array_equal(a, b)
        assert got[t][4] == ref[4]
