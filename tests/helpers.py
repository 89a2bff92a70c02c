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


class _LazyStack:
    """Index ``[i]`` of a torch tensor stack, fetched to numpy on first use."""

    def __init__(self, t, view=None):
        self.t, self.view, self.cache = t, view, {}

    def __getitem__(self, i):
        if i not in self.cache:
            a = self.t[i].cpu().numpy()
            self.cache[i] = a.view(self.view) if self.view is not None else a
        return self.cache[i]


def oqmat_lazy(q: "wlm.QMat") -> "oracle.OQMat":
    """An oracle matrix stack that copies each matrix off the GPU only when used."""
    return oracle.OQMat(_LazyStack(q.codes), _LazyStack(q.scale, np.uint16), _LazyStack(q.min, np.uint16),
                        q.rows, q.cols, q.bits, q.block)


def omoe_lazy(layer: "wlm.MoELayer") -> "oracle.OMoELayer":
    s = layer.spec
    f = lambda q: None if q is None else oqmat_lazy(q)
    return oracle.OMoELayer(
        n_experts=s.n_experts, top_k=s.top_k,
        router_w=layer.router_w.cpu().numpy(),
        router_b=None if layer.router_b is None else layer.router_b.cpu().numpy(),
        gate=oqmat_lazy(layer.gate), up=oqmat_lazy(layer.up), down=oqmat_lazy(layer.down),
        shared_gate=f(layer.shared_gate), shared_up=f(layer.shared_up),
        shared_down=f(layer.shared_down), renorm=bool(s.renorm_topk))


def stack_trajectory(x: np.ndarray, dense, moe):
    """One row through the oracle's layers: (y, [q], [k], [selected], min router margin)."""
    h = x.astype(np.float64)
    qs, ks, sels, margin = [], [], [], float("inf")
    for dl, ml in zip(dense, moe):
        tr = {}
        h, q, k, (sel, _) = oracle.decoder_layer_row(h, dl, ml, trace=tr)
        qs.append(q)
        ks.append(k)
        sels.append(sel)
        margin = min(margin, tr["margin"])
    return h, qs, ks, sels, margin
