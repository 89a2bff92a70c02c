"""C-ABI contract checks that need no GPU: the library builds and loads, it
exports every function the header declares, and argument errors are caught
on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from slot_decode_window_gb300 import binding as B
from slot_decode_window_gb300 import build as BLD

HEADER = os.path.join(BLD.INCLUDE, "strata_window.h")


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:strata_status|const char\*)\s+(strata_\w+)\s*\(", text, re.M)))


def test_header_declares_the_calls():
    assert set(_declared()) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    syms = set(re.findall(r"\bT\s+(\w+)", out))
    for name in _declared():
        assert name in syms, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    assert B.status_str(B.STRATA_OK) == "ok"
    assert "invalid" in B.status_str(B.STRATA_EINVAL)
    assert B.status_str(99) == "unknown status"


def _desc(**kw):
    base = dict(hidden=256, n_experts=8, top_k=2, ffn=128, shared_ffn=128, bits=4, block=32, max_rows=8, renorm_topk=0)
    base.update(kw)
    return B.strata_moe_desc(**base)


def _weights(fake=0x1000):
    q = B.strata_qmat(fake, fake, fake)
    return B.strata_moe_weights(fake, None, q, q, q, q, q, q)


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=0), B.STRATA_EINVAL),
    (dict(top_k=9, n_experts=8), B.STRATA_EINVAL),
    (dict(max_rows=9), B.STRATA_EINVAL),
    (dict(max_rows=0), B.STRATA_EINVAL),
    (dict(renorm_topk=2), B.STRATA_EINVAL),
    (dict(bits=3), B.STRATA_EUNSUPPORTED),
    (dict(bits=4, block=16), B.STRATA_EUNSUPPORTED),
    (dict(hidden=96), B.STRATA_EUNSUPPORTED),
    (dict(bits=2, block=16, hidden=192), B.STRATA_EUNSUPPORTED),
    (dict(n_experts=300, top_k=2), B.STRATA_EUNSUPPORTED),
    (dict(n_experts=16, top_k=12), B.STRATA_EUNSUPPORTED),
])
def test_create_rejects_bad_desc_on_host(lib, kw, status):
    st, h = B.strata_window_create(_desc(**kw), _weights())
    assert st == status and h is None


def test_create_rejects_null_pointers(lib):
    w = _weights()
    w.router_w = None
    assert B.strata_window_create(_desc(), w)[0] == B.STRATA_EINVAL
    w = _weights()
    w.shared_down = B.strata_qmat(0x1000, None, 0x1000)
    assert B.strata_window_create(_desc(), w)[0] == B.STRATA_EINVAL
    # no shared expert: the shared pointers are ignored, so the host checks pass;
    # with the allocation fault hook on, create stops before touching the GPU
    assert lib.strata_window_create(None, ctypes.byref(_weights()), None, ctypes.byref(ctypes.c_void_p())) == B.STRATA_EINVAL
    assert lib.strata_window_create(ctypes.byref(_desc()), ctypes.byref(_weights()), None, None) == B.STRATA_EINVAL


def test_fault_hook_alloc_gives_enomem(lib, monkeypatch):
    monkeypatch.setenv("STRATA_FAULT", "alloc")
    st, h = B.strata_window_create(_desc(shared_ffn=0), _weights())
    assert st == B.STRATA_ENOMEM and h is None


def test_calls_on_null_handle(lib):
    assert B.strata_moe_window_forward(None, 0x1000, 1, 0x2000) == B.STRATA_EINVAL
    assert B.strata_window_sync(None) == B.STRATA_EINVAL
    assert B.strata_window_query(None)[0] == B.STRATA_EINVAL
    assert B.strata_window_destroy(None) == B.STRATA_OK


def test_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = B.strata_window_create(_desc(), _weights())
    assert st == B.STRATA_ECUDA and h is None


# ---- the window-kernel plan a handle would choose (host only) ----

def _plan(spec, monkeypatch=None, env=(), max_rows=8, smem_limit=0):
    if monkeypatch is not None:
        for name in ("STRATA_WINDOW_RING", "STRATA_WINDOW_DIRECT"):
            monkeypatch.delenv(name, raising=False)
        for name in env:
            monkeypatch.setenv(name, "1")
    return B.strata_window_plan(B.desc_of(spec, max_rows), smem_limit)


def test_plan_keeps_the_ring_for_the_d2048_layer(lib, monkeypatch):
    """The d = 2048 4-bit layer keeps a three-stage ring of 40 KB stages."""
    from slot_decode_window_gb300 import workloads as wlm
    st, info = _plan(wlm.WORKLOADS["mid"].moe, monkeypatch)
    assert st == B.STRATA_OK
    assert (info.stages, info.stage_bytes) == (3, 40960)
    assert info.smem_bytes <= 232448 - 12288
    assert info.n_sm == 0 and info.packed_bytes == 0  # fields a plan does not fill


@pytest.mark.parametrize("name", ["zipf", "lowbit"])
def test_plan_streams_the_d4096_layers(lib, monkeypatch, name):
    """Both 4096-wide layers (4-bit with a ring under three 32 KB stages, and
    2-bit) take the warp-streamed path: no ring, per-warp FIFOs."""
    from slot_decode_window_gb300 import workloads as wlm
    spec = wlm.WORKLOADS[name].moe
    st, info = _plan(spec, monkeypatch)
    assert st == B.STRATA_OK and info.stages == 1
    item = 576 if spec.bits == 4 else 768  # one k-step chunk: codes + scale records
    assert info.stage_bytes == 16 * 4 * item
    st, ring = _plan(spec, monkeypatch, env=("STRATA_WINDOW_RING",))
    assert st == B.STRATA_OK and ring.stages >= 2
    assert ring.stages * ring.stage_bytes < 96 * 1024  # the short ring the rule avoids
    assert info.smem_bytes <= ring.smem_bytes


def test_plan_overrides_and_shape_rule(lib, monkeypatch):
    """STRATA_WINDOW_DIRECT forces the streamed path only where every warp gets
    a k-step of each task; the tiny layer (d = 256: 4 k-steps) stays on the ring."""
    from slot_decode_window_gb300 import workloads as wlm
    wide4 = wlm.MoESpec(512, 12, 4, 512, 512, 4, 32)
    assert _plan(wide4, monkeypatch)[1].stages >= 2
    assert _plan(wide4, monkeypatch, env=("STRATA_WINDOW_DIRECT",))[1].stages == 1
    tiny = wlm.WORKLOADS["tiny"].moe
    assert _plan(tiny, monkeypatch, env=("STRATA_WINDOW_DIRECT",))[1].stages >= 2
    wide2 = wlm.MoESpec(1024, 12, 4, 1024, 1024, 2, 16)
    assert _plan(wide2, monkeypatch)[1].stages == 1
    # both overrides: the ring wins
    assert _plan(wide2, monkeypatch, env=("STRATA_WINDOW_DIRECT", "STRATA_WINDOW_RING"))[1].stages >= 2


def test_plan_limits_and_errors(lib, monkeypatch):
    from slot_decode_window_gb300 import workloads as wlm
    mid = wlm.WORKLOADS["mid"].moe
    for limit in (150_000, 180_000, 220_160):
        st, info = _plan(mid, monkeypatch, smem_limit=limit)
        assert st == B.STRATA_OK and info.smem_bytes <= limit
        # a ring of three or more 32 KB stages, else the warp-streamed path
        assert info.stages == 1 or (info.stages >= 2 and info.stages * info.stage_bytes >= 96 * 1024)
    assert _plan(mid, monkeypatch, smem_limit=150_000)[1].stages == 1  # the ring would be short here
    assert _plan(mid, monkeypatch, smem_limit=220_160)[1].stages == 3
    assert _plan(mid, monkeypatch, smem_limit=60_000)[0] == B.STRATA_EUNSUPPORTED
    assert _plan(mid, monkeypatch, smem_limit=-1)[0] == B.STRATA_EINVAL
    assert B.strata_window_plan(_desc(hidden=0))[0] == B.STRATA_EINVAL
    assert B.strata_window_plan(_desc(bits=3))[0] == B.STRATA_EUNSUPPORTED
    assert lib.strata_window_plan(None, 0, ctypes.byref(B.strata_window_info())) == B.STRATA_EINVAL
    assert lib.strata_window_plan(ctypes.byref(_desc()), 0, None) == B.STRATA_EINVAL


@pytest.mark.parametrize("ffn,shared_ffn", [(256, 0), (1024, 256), (1024, 448)])
def test_plan_keeps_the_ring_when_a_warp_would_get_no_k_step(lib, monkeypatch, ffn, shared_ffn):
    """A d = 4096 4-bit layer leaves a short ring, but the warp-streamed path
    needs at least 8 64-column k-steps in every task (each warp of a sub-tile
    must get one): an expert or shared width under 512 keeps the ring."""
    from slot_decode_window_gb300 import workloads as wlm
    spec = wlm.MoESpec(4096, 16, 2, ffn, shared_ffn, 4, 32)
    st, info = _plan(spec, monkeypatch)
    assert st == B.STRATA_OK and info.stages >= 2
    st, forced = _plan(spec, monkeypatch, env=("STRATA_WINDOW_DIRECT",))
    assert st == B.STRATA_OK and forced.stages >= 2
    wide = wlm.MoESpec(4096, 16, 2, 1024, 512, 4, 32)
    assert _plan(wide, monkeypatch)[1].stages == 1


@pytest.mark.parametrize("kw", [
    dict(n_experts=0), dict(n_experts=300), dict(capacity=0), dict(capacity=17), dict(adapt_every=0),
    dict(adapt_swaps=-1), dict(adapt_swaps=17), dict(decay=0.0), dict(decay=1.5), dict(min_gain=0.5),
    dict(min_gain=float("inf")), dict(min_gain=float("nan")),
])
def test_tier_create_rejects_bad_desc_on_host(lib, kw):
    base = dict(n_experts=16, capacity=4, adapt_every=4, adapt_swaps=2, decay=0.5, min_gain=1.5)
    base.update(kw)
    st, t = B.strata_tier_create(B.strata_tier_desc(**base))
    assert st == B.STRATA_EINVAL and t is None


@pytest.mark.parametrize("initial", [[0, 1, 1, 2], [0, 1, 2, 16], [-1, 0, 1, 2]])
def test_tier_create_rejects_a_bad_initial_list_on_host(lib, initial):
    st, t = B.strata_tier_create(B.strata_tier_desc(16, 4, 4, 2, 0.5, 1.5), initial)
    assert st == B.STRATA_EINVAL and t is None


def test_tier_calls_accept_null(lib):
    assert B.strata_tier_destroy(None) == B.STRATA_OK
    assert B.strata_window_set_tier(None, None) == B.STRATA_EINVAL


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=0), B.STRATA_EINVAL), (dict(vocab=0), B.STRATA_EINVAL), (dict(max_rows=9), B.STRATA_EINVAL),
    (dict(bits=3), B.STRATA_EUNSUPPORTED), (dict(vocab=1000), B.STRATA_EUNSUPPORTED),
    (dict(hidden=96), B.STRATA_EUNSUPPORTED), (dict(bits=2, block=16, hidden=192), B.STRATA_EUNSUPPORTED),
])
def test_head_create_rejects_bad_desc_on_host(lib, kw, status):
    base = dict(hidden=256, vocab=4096, bits=4, block=32, max_rows=8)
    base.update(kw)
    q = B.strata_qmat(0x1000, 0x1000, 0x1000)
    st, h = B.strata_head_create(B.strata_head_desc(**base), q)
    assert st == status and h is None


def test_head_create_rejects_null_weight_pointers(lib):
    q = B.strata_qmat(0x1000, None, 0x1000)
    st, h = B.strata_head_create(B.strata_head_desc(256, 4096, 4, 32, 8), q)
    assert st == B.STRATA_EINVAL and h is None
    assert B.strata_head_destroy(None) == B.STRATA_OK
