"""fp64 oracle of the verify-window MoE step -- TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  The CUDA library never calls it.

What the Strata pages fix ("BATCHING.md", section "Several requests at once
(batch slots)", opening paragraph): a verify window carries one token of each
open conversation, and the dense weights, the shared expert, the head and every
routed expert two conversations share are read once per window for all of them.
Section "Exactness" of the same page: a batch row's arithmetic is the
single-token window's.  The pages give no router formula, quantization layout,
SwiGLU or shared-expert gating; the readings taken here are:

* router: ``logit = Wr x + b`` in fp64, top-k by logit (descending, ties to
  the lower expert index), gate weight = full-softmax probability of the
  selected expert (or renormalised over the k selected when ``renorm``);
* expert FFN: ``Wd (silu(Wg x) * (Wu x))`` with ``silu(z) = z / (1 + e^-z)``;
* shared expert: the same FFN with weight 1 and no gate;
* block format: ``w = scale * q + min`` per block of ``block`` elements,
  codes least-significant-bits first (see ``unpack_codes``);
* window output: ``y_t = shared(x_t) + sum_j g_tj * expert_{e_tj}(x_t)``;
* row groups: a counting sort of the entries ``t*k + j`` by expert, expert
  ascending, entries ascending within an expert.

Because reading a weight once per window is a scheduling choice, the oracle
evaluates each row on its own, as the definition states, and never groups
rows.  Every matrix is dequantized exactly in fp64 before use.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass
class OQMat:
    """A stack of block-quantized matrices ``[n][rows][cols]``."""
    codes: np.ndarray   # uint8 [n][rows][cols*bits/8]
    scale: np.ndarray   # uint16/int16 fp16 bit patterns [n][rows][cols/block]
    min: np.ndarray     # same shape as scale
    rows: int
    cols: int
    bits: int
    block: int


@dataclasses.dataclass
class OMoELayer:
    n_experts: int
    top_k: int
    router_w: np.ndarray              # fp32 [E][d]
    router_b: Optional[np.ndarray]    # fp32 [E] or None
    gate: OQMat                       # [E][F][d]
    up: OQMat                         # [E][F][d]
    down: OQMat                       # [E][d][F]
    shared_gate: Optional[OQMat] = None   # [1][Fs][d]
    shared_up: Optional[OQMat] = None
    shared_down: Optional[OQMat] = None   # [1][d][Fs]
    renorm: bool = False


@dataclasses.dataclass
class ODenseLayer:
    q: OQMat
    k: OQMat
    v: OQMat
    o: OQMat
    heads: int
    kv_heads: int
    head_dim: int


# ----------------------------------------------------------------------------
# block format


def fp16_bits(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (any 16-bit integer dtype) -> exact fp64 values."""
    return np.ascontiguousarray(bits).view(np.uint16).view(np.float16).astype(np.float64)


def unpack_codes(codes: np.ndarray, cols: int, bits: int) -> np.ndarray:
    """Codes of one matrix ``[rows][cols*bits/8]`` -> integers ``[rows][cols]``.

    Element ``i`` of a row sits in byte ``i*bits//8`` at bit ``bits*(i % (8//bits))``
    (4-bit: even element in the low nibble; 2-bit: element i%4 at bits 2*(i%4)).
    """
    per_byte = 8 // bits
    mask = (1 << bits) - 1
    c = codes.astype(np.int64)
    q = np.empty((codes.shape[0], cols), dtype=np.int64)
    for i in range(per_byte):
        q[:, i::per_byte] = (c >> (bits * i)) & mask
    return q


def dequant(m: OQMat, index: int = 0) -> np.ndarray:
    """Matrix ``index`` of the stack as exact fp64 ``[rows][cols]``: w = scale*q + min."""
    q = unpack_codes(m.codes[index], m.cols, m.bits).astype(np.float64)
    s = np.repeat(fp16_bits(m.scale[index]), m.block, axis=1)
    mn = np.repeat(fp16_bits(m.min[index]), m.block, axis=1)
    return s * q + mn


# ----------------------------------------------------------------------------
# router


def router(x: np.ndarray, router_w: np.ndarray, router_b: Optional[np.ndarray], k: int,
           renorm: bool = False):
    """One row's routing: (logits, probs, selected experts, gate weights).

    Logits ``Wr x + b`` in fp64; softmax over all experts, max-subtracted;
    top-k by logit, descending, ties to the lower index (a stable sort);
    gate = softmax probability of each selected expert, optionally
    renormalised over the k selected.
    """
    logits = router_w.astype(np.float64) @ x.astype(np.float64)
    if router_b is not None:
        logits = logits + router_b.astype(np.float64)
    order = np.argsort(-logits, kind="stable")[:k]
    e = np.exp(logits - logits.max())
    probs = e / e.sum()
    gates = probs[order]
    if renorm:
        gates = gates / gates.sum()
    return logits, probs, order.astype(np.int64), gates


def topk_margin(x: np.ndarray, router_w: np.ndarray, router_b: Optional[np.ndarray], k: int) -> float:
    """fp64 gap between the k-th and (k+1)-th largest logit of one row (inf if k == E)."""
    logits, _, _, _ = router(x, router_w, router_b, k)
    if k >= logits.size:
        return float("inf")
    srt = np.sort(logits)[::-1]
    return float(srt[k - 1] - srt[k])


# ----------------------------------------------------------------------------
# expert FFN


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def expert_ffn(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """SwiGLU expert on one row: Wd (silu(Wg x) * (Wu x))."""
    x = x.astype(np.float64)
    h = silu(wg @ x) * (wu @ x)
    return wd @ h


def shared_ffn(x: np.ndarray, layer: OMoELayer) -> np.ndarray:
    """Shared expert on one row, weight 1, no gate (zeros if the layer has none)."""
    if layer.shared_gate is None:
        return np.zeros(layer.down.rows, dtype=np.float64)
    return expert_ffn(x, dequant(layer.shared_gate), dequant(layer.shared_up), dequant(layer.shared_down))


# ----------------------------------------------------------------------------
# a window


def moe_row(x: np.ndarray, layer: OMoELayer, experts: Optional[Dict[int, Tuple]] = None):
    """One row of the window: (y, selected experts, gate weights).

    ``experts`` optionally caches dequantized (Wg, Wu, Wd) per expert; it only
    avoids repeating the same exact fp64 dequantization.
    """
    _, _, sel, g = router(x, layer.router_w, layer.router_b, layer.top_k, layer.renorm)
    y = shared_ffn(x, layer)
    for j in range(layer.top_k):
        e = int(sel[j])
        if experts is not None and e in experts:
            wg, wu, wd = experts[e]
        else:
            wg, wu, wd = dequant(layer.gate, e), dequant(layer.up, e), dequant(layer.down, e)
            if experts is not None:
                experts[e] = (wg, wu, wd)
        y = y + g[j] * expert_ffn(x, wg, wu, wd)
    return y, sel, g


def group_rows(topk_idx: np.ndarray, n_experts: int):
    """Row groups of a window by counting sort of entries t*k + j by expert.

    Returns (counts [E], offsets [E+1], entries [T*k], distinct experts
    ascending).  Entries of one expert appear in ascending (t, j) order.
    """
    T, k = topk_idx.shape
    counts = np.zeros(n_experts, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[topk_idx[t, j]] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    entries = np.empty(T * k, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = topk_idx[t, j]
            entries[fill[e]] = t * k + j
            fill[e] += 1
    distinct = np.nonzero(counts)[0]
    return counts, offsets, entries, distinct


def moe_window(x: np.ndarray, layer: OMoELayer, rows: Optional[Sequence[int]] = None,
               cache: bool = True):
    """The window step on rows ``x [T][d]``.

    Returns a dict with ``y [T][d]`` (rows not in ``rows`` left as NaN),
    ``topk_idx [T][k]``, ``topk_w [T][k]``, and the row groups
    ``counts, offsets, entries, distinct, n_distinct`` (routing is always
    computed for every row).
    """
    T = x.shape[0]
    k = layer.top_k
    d = layer.down.rows
    want = set(range(T)) if rows is None else set(int(r) for r in rows)
    y = np.full((T, d), np.nan)
    topk_idx = np.empty((T, k), dtype=np.int64)
    topk_w = np.empty((T, k), dtype=np.float64)
    experts: Optional[Dict[int, Tuple]] = {} if cache else None
    for t in range(T):
        if t in want:
            y[t], topk_idx[t], topk_w[t] = moe_row(x[t], layer, experts)
        else:
            _, _, topk_idx[t], topk_w[t] = router(x[t], layer.router_w, layer.router_b, k, layer.renorm)
    counts, offsets, entries, distinct = group_rows(topk_idx, layer.n_experts)
    return dict(y=y, topk_idx=topk_idx, topk_w=topk_w, counts=counts, offsets=offsets,
                entries=entries, distinct=distinct, n_distinct=len(distinct))


# ----------------------------------------------------------------------------
# decoder stack (dense projections + MoE per layer)


RMS_EPS = 1e-6


def rmsnorm(x: np.ndarray) -> np.ndarray:
    """x / sqrt(mean(x^2) + 1e-6), unit gain (a reading: the pages give no eps or gain)."""
    x = x.astype(np.float64)
    return x / np.sqrt(np.mean(x * x) + RMS_EPS)


def dense_attention_len1(v: np.ndarray, heads: int, kv_heads: int, head_dim: int) -> np.ndarray:
    """Attention of one row over a context of length one.

    With a single key the softmax weight is 1, so query head h outputs the
    value of its kv head ``h // (heads // kv_heads)`` (grouped-query sharing).
    """
    group = heads // kv_heads
    vh = v.reshape(kv_heads, head_dim)
    return np.concatenate([vh[h // group] for h in range(heads)])


def decoder_layer_row(x: np.ndarray, dense: ODenseLayer, moe: OMoELayer, trace: Optional[dict] = None):
    """One decoder layer on one row: pre-norm attention + residual, pre-norm MoE + residual.

    Returns (x_out, q, k, routing (selected, gates)).  ``trace``, if given,
    receives ``x1`` (the residual stream after attention) and ``margin`` (the
    router's top-k logit margin on ``rmsnorm(x1)``).
    """
    a = rmsnorm(x)
    q = dequant(dense.q) @ a
    kk = dequant(dense.k) @ a
    v = dequant(dense.v) @ a
    att = dense_attention_len1(v, dense.heads, dense.kv_heads, dense.head_dim)
    x1 = x.astype(np.float64) + dequant(dense.o) @ att
    b = rmsnorm(x1)
    y, sel, g = moe_row(b, moe)
    if trace is not None:
        trace["x1"] = x1
        trace["margin"] = topk_margin(b, moe.router_w, moe.router_b, moe.top_k)
    return x1 + y, q, kk, (sel, g)


def stack_row(x: np.ndarray, dense: List[ODenseLayer], moe: List[OMoELayer]):
    """A row through every layer; returns (x_out, per-layer routing list)."""
    h = x.astype(np.float64)
    routing = []
    for dl, ml in zip(dense, moe):
        h, _, _, r = decoder_layer_row(h, dl, ml)
        routing.append(r)
    return h, routing
