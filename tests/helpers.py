"""Glue between the seeded workloads (torch tensors) and the oracle (numpy)."""
from __future__ import annotations

import numpy as np

import oracle
from slot_decode_window_gb300 import workloads as wlm


def oqmat(q: "wlm.QMat") -> "oracle.OQMat":
    return oracle.OQMat(q.codes.cpu().numpy(), q.scale.cpu().numpy().view(np.uint16),
                        q.min.cpu().numpy().view(np.uint16), q.rows, q.cols, q.bits, q.block)


def omoe(layer: "wlm.MoELayer") -> "oracle.OMoELayer":
    s = layer.spec
    f = lambda q: None if q is None else oqmat(q)
    return oracle.OMoELayer(
        n_experts=s.n_experts, top_k=s.top_k,
        router_w=layer.router_w.cpu().numpy(),
        router_b=None if layer.router_b is None else layer.router_b.cpu().numpy(),
        gate=oqmat(layer.gate), up=oqmat(layer.up), down=oqmat(layer.down),
        shared_gate=f(layer.shared_gate), shared_up=f(layer.shared_up),
        shared_down=f(layer.shared_down), renorm=bool(s.renorm_topk))


def odense(dl: "wlm.DenseLayer", wl: "wlm.Workload") -> "oracle.ODenseLayer":
    return oracle.ODenseLayer(oqmat(dl.q), oqmat(dl.k), oqmat(dl.v), oqmat(dl.o),
                              wl.heads, wl.kv_heads, wl.head_dim)


MARGIN = 1e-3


def margin_accept(ol: "oracle.OMoELayer", margin: float = MARGIN):
    """A row predicate: the fp64 top-k logit margin is at least ``margin``."""
    def ok(row: np.ndarray) -> bool:
        return oracle.topk_margin(row, ol.router_w, ol.router_b, ol.top_k) >= margin
    return ok


def small_spec(**kw) -> "wlm.MoESpec":
    base = dict(hidden=64, n_experts=6, top_k=2, ffn=32, shared_ffn=32, bits=4, block=32)
    base.update(kw)
    return wlm.MoESpec(**base)
