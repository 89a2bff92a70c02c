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
