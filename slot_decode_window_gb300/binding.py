"""Thin ctypes binding of ``include/strata_window.h``.

Argument marshalling only: the functions keep the C names
(``strata_window_create``, ``strata_moe_window_forward``, ``strata_window_sync``,
``strata_window_query``, ``strata_window_destroy``, ``strata_status_str``) and
every step of a window runs in the library's CUDA kernels.  Loading fails
loudly when the shared library has not been built; there is no fallback.

``Window`` wraps a handle for torch tensors (device memory and streams come
from PyTorch; nothing is computed by it).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libstrata_window.so")

STRATA_OK, STRATA_EINVAL, STRATA_ENOMEM, STRATA_ECUDA, STRATA_EUNSUPPORTED, STRATA_EDEVICE = range(6)

EXPORTED = ("strata_window_create", "strata_moe_window_forward", "strata_window_sync", "strata_window_query",
            "strata_window_set_profiling", "strata_window_timings", "strata_window_destroy", "strata_status_str",
            "strata_moe_window_forward_noalloc", "strata_moe_window_forward_graph", "strata_stack_create", "strata_stack_forward", "strata_stack_sync",
            "strata_stack_query", "strata_stack_set_profiling", "strata_stack_timings", "strata_stack_destroy",
            "strata_window_plan", "strata_tier_create", "strata_window_set_tier", "strata_tier_read",
            "strata_tier_destroy", "strata_head_create", "strata_head_forward", "strata_head_sync",
            "strata_head_query", "strata_head_set_profiling", "strata_head_timings", "strata_head_destroy",
            "strata_window_slots", "strata_stack_set_kv", "strata_stack_forward_kv")
NOALLOC_SCRATCH_BYTES = 4 << 20


class StrataError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_str(status)} ({status})")
        self.status = status


class strata_qmat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("min", ctypes.c_void_p)]


class strata_moe_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("hidden", "n_experts", "top_k", "ffn", "shared_ffn", "bits", "block",
                                              "max_rows", "renorm_topk")]


class strata_moe_weights(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_b", ctypes.c_void_p), ("gate", strata_qmat),
                ("up", strata_qmat), ("down", strata_qmat), ("shared_gate", strata_qmat),
                ("shared_up", strata_qmat), ("shared_down", strata_qmat)]


class strata_routing_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("topk_idx", "topk_w", "counts", "offsets", "entries", "distinct",
                                               "n_distinct")]


class strata_window_info(ctypes.Structure):
    _fields_ = [("n_sm", ctypes.c_int32), ("stages", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("packed_bytes", ctypes.c_int64),
                ("expert_bytes", ctypes.c_int64), ("shared_bytes", ctypes.c_int64), ("router_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64)]


class strata_attn_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("heads", "kv_heads", "head_dim")]


class strata_attn_weights(ctypes.Structure):
    _fields_ = [("q", strata_qmat), ("k", strata_qmat), ("v", strata_qmat), ("o", strata_qmat)]


class strata_stack_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "topk_idx", "topk_w", "n_distinct")]


class strata_stack_info(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_sm", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("stage_bytes", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("dense_bytes", ctypes.c_int64),
                ("expert_bytes", ctypes.c_int64), ("shared_bytes", ctypes.c_int64), ("router_bytes", ctypes.c_int64)]


class strata_tier_desc(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("capacity", ctypes.c_int32), ("adapt_every", ctypes.c_int32),
                ("adapt_swaps", ctypes.c_int32), ("decay", ctypes.c_float), ("min_gain", ctypes.c_float)]


class strata_tier_stats(ctypes.Structure):
    _fields_ = [("windows", ctypes.c_int64), ("rounds", ctypes.c_int64), ("n_swaps", ctypes.c_int32)]


class strata_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("n_slots", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32)]


class strata_head_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("hidden", "vocab", "bits", "block", "max_rows")]


class strata_draw_in(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("position", "seed", "temperature", "fed")]


class strata_draw_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("tokens", "n_emit", "logits")]


_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with slot_decode_window_gb300.build.build() "
                           "(the window step has no non-CUDA implementation)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.strata_window_create.argtypes = [P(strata_moe_desc), P(strata_moe_weights), ctypes.c_void_p,
                                         P(ctypes.c_void_p)]
    lib.strata_window_create.restype = ctypes.c_int
    lib.strata_moe_window_forward.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                              P(strata_routing_out), ctypes.c_void_p]
    lib.strata_moe_window_forward.restype = ctypes.c_int
    lib.strata_moe_window_forward_graph.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                    ctypes.c_void_p, ctypes.c_void_p]
    lib.strata_moe_window_forward_graph.restype = ctypes.c_int
    lib.strata_moe_window_forward_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                      ctypes.c_void_p, ctypes.c_void_p]
    lib.strata_moe_window_forward_noalloc.restype = ctypes.c_int
    lib.strata_stack_create.argtypes = [ctypes.c_int32, P(strata_moe_desc), P(strata_attn_desc),
                                        P(strata_moe_weights), P(strata_attn_weights), ctypes.c_void_p,
                                        P(ctypes.c_void_p)]
    lib.strata_stack_create.restype = ctypes.c_int
    lib.strata_stack_forward.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                         P(strata_stack_out), ctypes.c_void_p]
    lib.strata_stack_forward.restype = ctypes.c_int
    lib.strata_stack_sync.argtypes = [ctypes.c_void_p]
    lib.strata_stack_sync.restype = ctypes.c_int
    lib.strata_stack_query.argtypes = [ctypes.c_void_p, P(strata_stack_info)]
    lib.strata_stack_query.restype = ctypes.c_int
    lib.strata_stack_set_profiling.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.strata_stack_set_profiling.restype = ctypes.c_int
    lib.strata_stack_timings.argtypes = [ctypes.c_void_p, P(ctypes.c_float)]
    lib.strata_stack_timings.restype = ctypes.c_int
    lib.strata_stack_destroy.argtypes = [ctypes.c_void_p]
    lib.strata_stack_destroy.restype = ctypes.c_int
    lib.strata_window_sync.argtypes = [ctypes.c_void_p]
    lib.strata_window_sync.restype = ctypes.c_int
    lib.strata_window_query.argtypes = [ctypes.c_void_p, P(strata_window_info)]
    lib.strata_window_query.restype = ctypes.c_int
    lib.strata_window_plan.argtypes = [P(strata_moe_desc), ctypes.c_int32, P(strata_window_info)]
    lib.strata_window_plan.restype = ctypes.c_int
    lib.strata_window_set_profiling.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.strata_window_set_profiling.restype = ctypes.c_int
    lib.strata_window_timings.argtypes = [ctypes.c_void_p, P(ctypes.c_float)]
    lib.strata_window_timings.restype = ctypes.c_int
    lib.strata_window_destroy.argtypes = [ctypes.c_void_p]
    lib.strata_window_destroy.restype = ctypes.c_int
    lib.strata_tier_create.argtypes = [P(strata_tier_desc), ctypes.c_void_p, P(ctypes.c_void_p)]
    lib.strata_tier_create.restype = ctypes.c_int
    lib.strata_window_set_tier.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.strata_window_set_tier.restype = ctypes.c_int
    lib.strata_tier_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, P(strata_tier_stats)]
    lib.strata_tier_read.restype = ctypes.c_int
    lib.strata_tier_destroy.argtypes = [ctypes.c_void_p]
    lib.strata_tier_destroy.restype = ctypes.c_int
    lib.strata_head_create.argtypes = [P(strata_head_desc), P(strata_qmat), ctypes.c_void_p, P(ctypes.c_void_p)]
    lib.strata_head_create.restype = ctypes.c_int
    lib.strata_head_forward.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, P(strata_draw_in),
                                        P(strata_draw_out), ctypes.c_void_p]
    lib.strata_head_forward.restype = ctypes.c_int
    lib.strata_head_sync.argtypes = [ctypes.c_void_p]
    lib.strata_head_sync.restype = ctypes.c_int
    lib.strata_head_query.argtypes = [ctypes.c_void_p, P(ctypes.c_int64), P(ctypes.c_int64)]
    lib.strata_head_query.restype = ctypes.c_int
    lib.strata_head_set_profiling.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.strata_head_set_profiling.restype = ctypes.c_int
    lib.strata_head_timings.argtypes = [ctypes.c_void_p, P(ctypes.c_float)]
    lib.strata_head_timings.restype = ctypes.c_int
    lib.strata_head_destroy.argtypes = [ctypes.c_void_p]
    lib.strata_head_destroy.restype = ctypes.c_int
    lib.strata_window_slots.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p, P(ctypes.c_int32), P(ctypes.c_int32)]
    lib.strata_window_slots.restype = ctypes.c_int
    lib.strata_stack_set_kv.argtypes = [ctypes.c_void_p, P(strata_kv_cache)]
    lib.strata_stack_set_kv.restype = ctypes.c_int
    lib.strata_stack_forward_kv.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, P(strata_stack_out), ctypes.c_void_p]
    lib.strata_stack_forward_kv.restype = ctypes.c_int
    lib.strata_status_str.argtypes = [ctypes.c_int]
    lib.strata_status_str.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().strata_status_str(status).decode()


# --- the C calls, same names ---------------------------------------------------


def strata_window_create(desc: strata_moe_desc, weights: strata_moe_weights, stream: int = 0):
    """Returns (status, handle or None)."""
    h = ctypes.c_void_p()
    st = load().strata_window_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.c_void_p(stream),
                                     ctypes.byref(h))
    return st, (h.value if st == STRATA_OK else None)


def strata_moe_window_forward(handle, x_ptr: int, T: int, y_ptr: int, routing: Optional[strata_routing_out] = None,
                              stream: int = 0) -> int:
    return load().strata_moe_window_forward(ctypes.c_void_p(handle), ctypes.c_void_p(x_ptr), T,
                                            ctypes.c_void_p(y_ptr),
                                            ctypes.byref(routing) if routing is not None else None,
                                            ctypes.c_void_p(stream))


def strata_moe_window_forward_graph(handle, x_ptr: int, T: int, y_ptr: int, stream: int = 0) -> int:
    return load().strata_moe_window_forward_graph(ctypes.c_void_p(handle), ctypes.c_void_p(x_ptr), T,
                                                  ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def strata_moe_window_forward_noalloc(handle, x_ptr: int, T: int, y_ptr: int, stream: int = 0) -> int:
    return load().strata_moe_window_forward_noalloc(ctypes.c_void_p(handle), ctypes.c_void_p(x_ptr), T,
                                                    ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream))


def strata_stack_create(n_layers: int, desc: strata_moe_desc, attn: strata_attn_desc, moe_w, attn_w,
                        stream: int = 0):
    """moe_w / attn_w: ctypes arrays of n_layers weight structs.  Returns (status, handle or None)."""
    h = ctypes.c_void_p()
    st = load().strata_stack_create(n_layers, ctypes.byref(desc), ctypes.byref(attn), moe_w, attn_w,
                                    ctypes.c_void_p(stream), ctypes.byref(h))
    return st, (h.value if st == STRATA_OK else None)


def strata_stack_forward(handle, x_ptr: int, T: int, y_ptr: int, out: Optional[strata_stack_out] = None,
                         stream: int = 0) -> int:
    return load().strata_stack_forward(ctypes.c_void_p(handle), ctypes.c_void_p(x_ptr), T, ctypes.c_void_p(y_ptr),
                                       ctypes.byref(out) if out is not None else None, ctypes.c_void_p(stream))


def strata_stack_sync(handle) -> int:
    return load().strata_stack_sync(ctypes.c_void_p(handle))


def strata_stack_query(handle):
    info = strata_stack_info()
    st = load().strata_stack_query(ctypes.c_void_p(handle), ctypes.byref(info))
    return st, info


def strata_stack_set_profiling(handle, enable: bool) -> int:
    return load().strata_stack_set_profiling(ctypes.c_void_p(handle), 1 if enable else 0)


def strata_stack_timings(handle):
    ms = ctypes.c_float()
    st = load().strata_stack_timings(ctypes.c_void_p(handle), ctypes.byref(ms))
    return st, ms.value


def strata_stack_destroy(handle) -> int:
    return load().strata_stack_destroy(ctypes.c_void_p(handle))


def strata_window_sync(handle) -> int:
    return load().strata_window_sync(ctypes.c_void_p(handle))


def strata_window_query(handle):
    info = strata_window_info()
    st = load().strata_window_query(ctypes.c_void_p(handle), ctypes.byref(info))
    return st, info


def strata_window_plan(desc: strata_moe_desc, smem_limit: int = 0):
    info = strata_window_info()
    st = load().strata_window_plan(ctypes.byref(desc), smem_limit, ctypes.byref(info))
    return st, info


def strata_window_set_profiling(handle, enable: bool) -> int:
    return load().strata_window_set_profiling(ctypes.c_void_p(handle), 1 if enable else 0)


def strata_window_timings(handle):
    """Returns (status, window kernel ms)."""
    ms = ctypes.c_float()
    st = load().strata_window_timings(ctypes.c_void_p(handle), ctypes.byref(ms))
    return st, ms.value


def strata_window_destroy(handle) -> int:
    return load().strata_window_destroy(ctypes.c_void_p(handle))


def strata_tier_create(desc: strata_tier_desc, initial=None):
    """initial: a sequence of expert ids or None.  Returns (status, tier or None)."""
    h = ctypes.c_void_p()
    arr = None
    if initial is not None:
        arr = (ctypes.c_int32 * len(initial))(*[int(e) for e in initial])
    st = load().strata_tier_create(ctypes.byref(desc), arr, ctypes.byref(h))
    return st, (h.value if st == STRATA_OK else None)


def strata_window_set_tier(handle, tier) -> int:
    return load().strata_window_set_tier(ctypes.c_void_p(handle), ctypes.c_void_p(tier) if tier else None)


def strata_tier_read(tier, n_experts: int):
    """Returns (status, dict of numpy arrays counters/resident/swap_in/swap_out and the stats)."""
    import numpy as np
    c = np.zeros(n_experts, np.float32)
    r = np.zeros(n_experts, np.int32)
    si = np.zeros(n_experts, np.int32)
    so = np.zeros(n_experts, np.int32)
    stats = strata_tier_stats()
    st = load().strata_tier_read(ctypes.c_void_p(tier), c.ctypes.data, r.ctypes.data, si.ctypes.data, so.ctypes.data,
                                 ctypes.byref(stats))
    return st, dict(counters=c, resident=r, swap_in=si[:stats.n_swaps], swap_out=so[:stats.n_swaps],
                    windows=stats.windows, rounds=stats.rounds, n_swaps=stats.n_swaps)


def strata_tier_destroy(tier) -> int:
    return load().strata_tier_destroy(ctypes.c_void_p(tier) if tier else None)


def strata_head_create(desc: strata_head_desc, weight: strata_qmat, stream: int = 0):
    """Returns (status, head or None)."""
    h = ctypes.c_void_p()
    st = load().strata_head_create(ctypes.byref(desc), ctypes.byref(weight), ctypes.c_void_p(stream), ctypes.byref(h))
    return st, (h.value if st == STRATA_OK else None)


def strata_head_forward(handle, x_ptr: int, T: int, draw_in: strata_draw_in, draw_out: strata_draw_out,
                        stream: int = 0) -> int:
    return load().strata_head_forward(ctypes.c_void_p(handle), ctypes.c_void_p(x_ptr), T, ctypes.byref(draw_in),
                                      ctypes.byref(draw_out), ctypes.c_void_p(stream))


def strata_head_sync(handle) -> int:
    return load().strata_head_sync(ctypes.c_void_p(handle))


def strata_head_query(handle):
    hb, wb = ctypes.c_int64(), ctypes.c_int64()
    st = load().strata_head_query(ctypes.c_void_p(handle), ctypes.byref(hb), ctypes.byref(wb))
    return st, hb.value, wb.value


def strata_head_set_profiling(handle, enable: bool) -> int:
    return load().strata_head_set_profiling(ctypes.c_void_p(handle), 1 if enable else 0)


def strata_head_timings(handle):
    ms = ctypes.c_float()
    st = load().strata_head_timings(ctypes.c_void_p(handle), ctypes.byref(ms))
    return st, ms.value


def strata_head_destroy(handle) -> int:
    return load().strata_head_destroy(ctypes.c_void_p(handle) if handle else None)


def strata_window_slots(rows_per_slot, start: int, max_rows: int = 8):
    """Returns (status, slots of the next window, next start)."""
    n = len(rows_per_slot)
    rows = (ctypes.c_int32 * max(n, 1))(*[int(r) for r in rows_per_slot])
    out = (ctypes.c_int32 * max(n, 1))()
    cnt, nxt = ctypes.c_int32(), ctypes.c_int32()
    st = load().strata_window_slots(n, rows if n else None, start, max_rows, out, ctypes.byref(cnt), ctypes.byref(nxt))
    return st, [out[i] for i in range(cnt.value)] if st == STRATA_OK else [], nxt.value


def strata_stack_set_kv(handle, kv) -> int:
    return load().strata_stack_set_kv(ctypes.c_void_p(handle), ctypes.byref(kv) if kv is not None else None)


def strata_stack_forward_kv(handle, x_ptr: int, T: int, y_ptr: int, slot_ptr: int, pos_ptr: int,
                            out: Optional["strata_stack_out"] = None, stream: int = 0) -> int:
    return load().strata_stack_forward_kv(ctypes.c_void_p(handle), ctypes.c_void_p(x_ptr), T, ctypes.c_void_p(y_ptr),
                                          ctypes.c_void_p(slot_ptr), ctypes.c_void_p(pos_ptr),
                                          ctypes.byref(out) if out is not None else None, ctypes.c_void_p(stream))


def check(status: int, what: str) -> None:
    if status != STRATA_OK:
        raise StrataError(status, what)


# --- torch convenience -----------------------------------------------------------


def _qmat(q) -> strata_qmat:
    return strata_qmat(q.codes.data_ptr(), q.scale.data_ptr(), q.min.data_ptr())


def desc_of(spec, max_rows: int = 8) -> strata_moe_desc:
    return strata_moe_desc(spec.hidden, spec.n_experts, spec.top_k, spec.ffn, spec.shared_ffn, spec.bits, spec.block,
                           max_rows, spec.renorm_topk)


def weights_of(layer) -> strata_moe_weights:
    w = strata_moe_weights()
    w.router_w = layer.router_w.data_ptr()
    w.router_b = layer.router_b.data_ptr() if layer.router_b is not None else None
    w.gate, w.up, w.down = _qmat(layer.gate), _qmat(layer.up), _qmat(layer.down)
    if layer.shared_gate is not None:
        w.shared_gate, w.shared_up, w.shared_down = (_qmat(layer.shared_gate), _qmat(layer.shared_up),
                                                     _qmat(layer.shared_down))
    return w


class Window:
    """A handle for one MoE layer whose weights are CUDA torch tensors."""

    def __init__(self, layer, max_rows: int = 8, stream=None):
        import torch
        self.spec = layer.spec
        self.max_rows = max_rows
        s = (stream or torch.cuda.current_stream()).cuda_stream
        st, h = strata_window_create(desc_of(layer.spec, max_rows), weights_of(layer), s)
        check(st, "strata_window_create")
        self.handle = h

    def info(self) -> strata_window_info:
        st, info = strata_window_query(self.handle)
        check(st, "strata_window_query")
        return info

    def forward(self, x, y=None, routing: bool = False, stream=None):
        """Enqueue one window on x [T][d] (CUDA fp32); returns y (and routing tensors)."""
        import torch
        assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
        T, d = x.shape
        if y is None:
            y = torch.empty_like(x)
        r = None
        rt = None
        if routing:
            E, k = self.spec.n_experts, self.spec.top_k
            dev = x.device
            rt = dict(topk_idx=torch.empty(T, k, dtype=torch.int32, device=dev),
                      topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
                      counts=torch.empty(E, dtype=torch.int32, device=dev),
                      offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                      entries=torch.empty(T * k, dtype=torch.int32, device=dev),
                      distinct=torch.full((E,), -1, dtype=torch.int32, device=dev),
                      n_distinct=torch.empty(1, dtype=torch.int32, device=dev))
            r = strata_routing_out(*(rt[n].data_ptr() for n in ("topk_idx", "topk_w", "counts", "offsets", "entries",
                                                               "distinct", "n_distinct")))
        s = (stream or torch.cuda.current_stream()).cuda_stream
        check(strata_moe_window_forward(self.handle, x.data_ptr(), T, y.data_ptr(), r, s),
              "strata_moe_window_forward")
        return (y, rt) if routing else y

    def forward_graph(self, x, y, stream=None):
        """Enqueue one window through the handle's graph cache (x, y fixed CUDA buffers)."""
        import torch
        assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous() and y.is_contiguous()
        s = (stream or torch.cuda.current_stream()).cuda_stream
        check(strata_moe_window_forward_graph(self.handle, x.data_ptr(), x.shape[0], y.data_ptr(), s),
              "strata_moe_window_forward_graph")
        return y

    def set_profiling(self, enable: bool) -> None:
        check(strata_window_set_profiling(self.handle, enable), "strata_window_set_profiling")

    def timings(self):
        st, ms = strata_window_timings(self.handle)
        check(st, "strata_window_timings")
        return ms

    def sync(self) -> None:
        check(strata_window_sync(self.handle), "strata_window_sync")

    def close(self) -> None:
        if getattr(self, "handle", None):
            strata_window_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def attn_desc_of(wl) -> strata_attn_desc:
    return strata_attn_desc(wl.heads, wl.kv_heads, wl.head_dim)


def attn_weights_of(dl) -> strata_attn_weights:
    return strata_attn_weights(_qmat(dl.q), _qmat(dl.k), _qmat(dl.v), _qmat(dl.o))


class Stack:
    """A handle for a stack of decoder layers whose weights are CUDA torch tensors.

    moe_layers / dense_layers: per-layer ``workloads.MoELayer`` / ``DenseLayer``;
    wl: the workload (attention shapes).  The handle keeps its own
    kernel-ordered copies, so the tensors may be freed after construction.
    """

    def __init__(self, wl, moe_layers, dense_layers, max_rows: int = 8, stream=None):
        import torch
        n = len(moe_layers)
        assert n == len(dense_layers) and n >= 1
        self.wl, self.n_layers, self.spec = wl, n, moe_layers[0].spec
        mw = (strata_moe_weights * n)(*[weights_of(m) for m in moe_layers])
        aw = (strata_attn_weights * n)(*[attn_weights_of(dl) for dl in dense_layers])
        s = (stream or torch.cuda.current_stream()).cuda_stream
        st, h = strata_stack_create(n, desc_of(self.spec, max_rows), attn_desc_of(wl), mw, aw, s)
        check(st, "strata_stack_create")
        self.handle = h

    def info(self) -> strata_stack_info:
        st, info = strata_stack_query(self.handle)
        check(st, "strata_stack_query")
        return info

    def set_kv(self, k, v, n_slots: int, max_ctx: int) -> None:
        """Attend over the fp16 caches k, v (CUDA tensors of
        [n_layers][n_slots][kv_heads][max_ctx][head_dim], float16) from now on
        (forward with slot and position); None drops them."""
        if k is None:
            check(strata_stack_set_kv(self.handle, None), "strata_stack_set_kv")
            self.kv = None
            return
        check(strata_stack_set_kv(self.handle, strata_kv_cache(k.data_ptr(), v.data_ptr(), n_slots, max_ctx)),
              "strata_stack_set_kv")
        self.kv = (k, v)

    def forward(self, x, y=None, outputs: bool = False, stream=None, slot=None, position=None):
        """Enqueue one window on x [T][d]; returns y (and per-layer q, k, routing).
        With slot and position (CUDA int32 [T]) the window attends over the caches set by set_kv."""
        import torch
        assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
        T, d = x.shape
        if y is None:
            y = torch.empty_like(x)
        o = None
        res = None
        if outputs:
            n, wl, k = self.n_layers, self.wl, self.spec.top_k
            dev = x.device
            res = dict(q=torch.empty(n, T, wl.heads * wl.head_dim, device=dev),
                       k=torch.empty(n, T, wl.kv_heads * wl.head_dim, device=dev),
                       topk_idx=torch.empty(n, T, k, dtype=torch.int32, device=dev),
                       topk_w=torch.empty(n, T, k, device=dev),
                       n_distinct=torch.empty(n, dtype=torch.int32, device=dev))
            o = strata_stack_out(*(res[m].data_ptr() for m in ("q", "k", "topk_idx", "topk_w", "n_distinct")))
        s = (stream or torch.cuda.current_stream()).cuda_stream
        if slot is not None:
            check(strata_stack_forward_kv(self.handle, x.data_ptr(), T, y.data_ptr(), slot.data_ptr(),
                                          position.data_ptr(), o, s), "strata_stack_forward_kv")
        else:
            check(strata_stack_forward(self.handle, x.data_ptr(), T, y.data_ptr(), o, s), "strata_stack_forward")
        return (y, res) if outputs else y

    def set_profiling(self, enable: bool) -> None:
        check(strata_stack_set_profiling(self.handle, enable), "strata_stack_set_profiling")

    def timings(self):
        st, ms = strata_stack_timings(self.handle)
        check(st, "strata_stack_timings")
        return ms

    def sync(self) -> None:
        check(strata_stack_sync(self.handle), "strata_stack_sync")

    def close(self) -> None:
        if getattr(self, "handle", None):
            strata_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Head:
    """The output head for a block-format weight ``QMat`` [1][V][d] on the GPU."""

    def __init__(self, weight, max_rows: int = 8, stream=None):
        import torch
        self.V, self.d = weight.rows, weight.cols
        s = (stream or torch.cuda.current_stream()).cuda_stream
        desc = strata_head_desc(weight.cols, weight.rows, weight.bits, weight.block, max_rows)
        st, h = strata_head_create(desc, _qmat(weight), s)
        check(st, "strata_head_create")
        self.handle = h

    def forward(self, x, position, seed, temperature, fed, logits: bool = False, stream=None):
        """Enqueue one window's head on x [T][d]; the per-row inputs are CUDA
        tensors (int32, int64 seeds, float32, int32).  Returns (tokens, n_emit,
        logits or None), int32 / float32 CUDA tensors."""
        import torch
        assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
        T = x.shape[0]
        dev = x.device
        tokens = torch.empty(T, dtype=torch.int32, device=dev)
        n_emit = torch.empty(T, dtype=torch.int32, device=dev)
        lg = torch.empty(T, self.V, device=dev) if logits else None
        di = strata_draw_in(position.data_ptr(), seed.data_ptr(), temperature.data_ptr(), fed.data_ptr())
        do = strata_draw_out(tokens.data_ptr(), n_emit.data_ptr(), lg.data_ptr() if logits else None)
        s = (stream or torch.cuda.current_stream()).cuda_stream
        check(strata_head_forward(self.handle, x.data_ptr(), T, di, do, s), "strata_head_forward")
        return tokens, n_emit, lg

    def sync(self) -> None:
        check(strata_head_sync(self.handle), "strata_head_sync")

    def set_profiling(self, enable: bool) -> None:
        check(strata_head_set_profiling(self.handle, enable), "strata_head_set_profiling")

    def timings(self):
        st, ms = strata_head_timings(self.handle)
        check(st, "strata_head_timings")
        return ms

    def head_bytes(self) -> int:
        st, hb, _ = strata_head_query(self.handle)
        check(st, "strata_head_query")
        return hb

    def close(self) -> None:
        if getattr(self, "handle", None):
            strata_head_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
