"""The oracle's window and stack, evaluated expert by expert -- TEST INFRASTRUCTURE.

The full-size workloads (a 2-bit d=4096 layer with up to 64 distinct experts,
the 48-layer stack) are too large for ``oracle.moe_window``'s per-window cache
of dequantized experts and too slow for ``oracle.stack_row`` row by row.  The
functions here call only the oracle's own functions (``router``, ``dequant``,
``expert_ffn``, ``rmsnorm``, ``dense_attention_len1``, ``topk_margin``,
``group_rows``) in the same per-row order of operations, so every output is
bitwise the oracle's (``tests/test_oracle_lean.py`` checks that on small
cases); they only change which matrix is dequantized when: each routed expert
once per layer, applied to every row that chose it, then dropped.  An optional
process pool (created with the ``spawn`` start method) spreads the experts
over the host's cores.

This module imports only numpy and the oracle, so spawned workers start fast.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

import oracle


def one(q: "oracle.OQMat", i: int) -> "oracle.OQMat":
    """Matrix ``i`` of a stack as a stack of one (works for lazily fetched stacks too)."""
    return oracle.OQMat(np.asarray(q.codes[i])[None], np.asarray(q.scale[i])[None], np.asarray(q.min[i])[None],
                        q.rows, q.cols, q.bits, q.block)


def _ffn_rows(args):
    """Worker: one expert's SwiGLU FFN on each of the given rows."""
    g, u, d, xs = args
    wg, wu, wd = oracle.dequant(g), oracle.dequant(u), oracle.dequant(d)
    return [oracle.expert_ffn(x, wg, wu, wd) for x in xs]


def spawn_pool(n: Optional[int] = None):
    """A process pool of the ``spawn`` start method (safe beside an initialised
    GPU context); a worker that dies makes the map raise instead of hanging."""
    import concurrent.futures as cf
    n = n or min(16, os.cpu_count() or 1)
    return cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn"))


def moe_rows(xs: Sequence[np.ndarray], layer: "oracle.OMoELayer", pool=None):
    """``oracle.moe_row`` of every row of ``xs``: (ys, selected, gates), bitwise equal.

    moe_row computes ``y = shared(x)``, then ``y = y + g_j * expert_{e_j}(x)``
    for j in order; the same operations run here, with each expert's
    outputs computed once per expert for all rows that chose it.
    """
    routes = [oracle.router(x, layer.router_w, layer.router_b, layer.top_k, layer.renorm) for x in xs]
    sels = [r[2] for r in routes]
    gates = [r[3] for r in routes]
    by_e: Dict[int, List[Tuple[int, int]]] = {}
    for t, sel in enumerate(sels):
        for j, e in enumerate(sel):
            by_e.setdefault(int(e), []).append((t, j))
    experts = sorted(by_e)
    jobs = [(one(layer.gate, e), one(layer.up, e), one(layer.down, e), [xs[t] for t, _ in by_e[e]])
            for e in experts]
    if layer.shared_gate is not None:
        jobs.append((layer.shared_gate, layer.shared_up, layer.shared_down, list(xs)))
    outs = list(pool.map(_ffn_rows, jobs)) if pool is not None else [_ffn_rows(a) for a in jobs]
    out: Dict[Tuple[int, int], np.ndarray] = {}
    for e, o in zip(experts, outs):
        for (t, j), v in zip(by_e[e], o):
            out[(t, j)] = v
    d = layer.down.rows
    ys = []
    for t in range(len(xs)):
        y = outs[-1][t] if layer.shared_gate is not None else np.zeros(d, dtype=np.float64)
        for j in range(layer.top_k):
            y = y + gates[t][j] * out[(t, j)]
        ys.append(y)
    return ys, sels, gates


def moe_window(x: np.ndarray, layer: "oracle.OMoELayer", pool=None):
    """``oracle.moe_window(x, layer)`` (all rows), bitwise equal."""
    ys, sels, gates = moe_rows([x[t] for t in range(x.shape[0])], layer, pool)
    topk_idx = np.stack(sels).astype(np.int64)
    counts, offsets, entries, distinct = oracle.group_rows(topk_idx, layer.n_experts)
    return dict(y=np.stack(ys), topk_idx=topk_idx, topk_w=np.stack(gates), counts=counts, offsets=offsets,
                entries=entries, distinct=distinct, n_distinct=len(distinct))


def stack_rows(x: np.ndarray, dense: List["oracle.ODenseLayer"], moe: List["oracle.OMoELayer"], pool=None):
    """Every row of ``x`` through the oracle's decoder layers, as
    ``tests.helpers.stack_trajectory`` reports one row: a list over rows of
    (y, [q per layer], [k per layer], [selected per layer], min router margin),
    bitwise equal to ``oracle.decoder_layer_row`` applied layer after layer."""
    T = x.shape[0]
    hs = [x[t].astype(np.float64) for t in range(T)]
    qs: List[list] = [[] for _ in range(T)]
    ks: List[list] = [[] for _ in range(T)]
    sels: List[list] = [[] for _ in range(T)]
    margin = [float("inf")] * T
    for dl, ml in zip(dense, moe):
        wq, wk, wv, wo = oracle.dequant(dl.q), oracle.dequant(dl.k), oracle.dequant(dl.v), oracle.dequant(dl.o)
        x1s, bs = [], []
        for t in range(T):
            a = oracle.rmsnorm(hs[t])
            qs[t].append(wq @ a)
            ks[t].append(wk @ a)
            v = wv @ a
            att = oracle.dense_attention_len1(v, dl.heads, dl.kv_heads, dl.head_dim)
            x1 = hs[t].astype(np.float64) + wo @ att
            b = oracle.rmsnorm(x1)
            x1s.append(x1)
            bs.append(b)
            margin[t] = min(margin[t], oracle.topk_margin(b, ml.router_w, ml.router_b, ml.top_k))
        ys, sel, _ = moe_rows(bs, ml, pool)
        for t in range(T):
            sels[t].append(sel[t])
            hs[t] = x1s[t] + ys[t]
    return [(hs[t], qs[t], ks[t], sels[t], margin[t]) for t in range(T)]
