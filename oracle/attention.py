"""Oracle of a verify window's attention over each slot's KV cache -- TEST
INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import
this module; the CUDA library never calls it.

What the Strata pages fix ("BATCHING.md", section "Several requests at once
(batch slots)"): every open conversation is a slot that keeps its own state,
its KV cache among it (the slot paragraph; "What a slot costs" names the
per-slot KV and --kv-resident, the 32K attention window it streams); a verify
window carries one row per slot, plus the slot's MTP proposal as a second row
with --batch-mtp, so a proposal row at position p + 1 attends to its token
row's entry at p written in the same window.  The pages give no formulas; the
readings taken here:

* one cache per layer, K and V ``[slots][kv_heads][ctx][head_dim]``, fp16;
* a row t of slot s_t at position p_t first stores its k and v (the dense
  projections of RMSNorm(x_t)), rounded to fp16, at position p_t of its slot;
  every row of the window does so before any row attends;
* row t then attends, for query head h, over positions 0..p_t of slot s_t
  with kv head ``h // (heads / kv_heads)``: weights softmax_j(q_h . K_j /
  sqrt(head_dim)), output sum_j w_j V_j;
* no rotary or other position encoding (the pages name none);
* the rest of the layer is the length-one reading's: x1 = x + Wo att, then
  x1 + MoE(RMSNorm(x1)).

Plain fp64 numpy; each function cites the step it follows.
"""
from __future__ import annotations

import math
from typing import List, Sequence

import numpy as np

from .moe_window import ODenseLayer, OMoELayer, dequant, moe_row, rmsnorm, topk_margin


def fp16_round(a: np.ndarray) -> np.ndarray:
    """Round to the nearest fp16 value (ties to even), returned as fp64."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).astype(np.float64)


def append_kv(kc: np.ndarray, vc: np.ndarray, k: np.ndarray, v: np.ndarray, slot: int, pos: int) -> None:
    """Store one row's k and v (kv_heads x head_dim each) at position pos of its slot, in fp16."""
    kvh, _, hd = kc.shape[1], kc.shape[2], kc.shape[3]
    kc[slot, :, pos, :] = fp16_round(k.reshape(kvh, hd))
    vc[slot, :, pos, :] = fp16_round(v.reshape(kvh, hd))


def attention_row(q: np.ndarray, kc: np.ndarray, vc: np.ndarray, slot: int, pos: int, heads: int) -> np.ndarray:
    """One row's attention output [heads * head_dim] over positions 0..pos of its slot."""
    kvh, hd = kc.shape[1], kc.shape[3]
    group = heads // kvh
    out = np.empty(heads * hd)
    for h in range(heads):
        g = h // group
        K = kc[slot, g, :pos + 1, :]
        V = vc[slot, g, :pos + 1, :]
        s = K @ q[h * hd:(h + 1) * hd] / math.sqrt(hd)
        w = np.exp(s - s.max())
        w /= w.sum()
        out[h * hd:(h + 1) * hd] = w @ V
    return out


def decoder_layer_window(X: np.ndarray, dense: ODenseLayer, moe: OMoELayer, kc: np.ndarray, vc: np.ndarray,
                         slots: Sequence[int], positions: Sequence[int]):
    """Every row of a window through one decoder layer with cache attention.

    kc / vc are this layer's caches, updated in place with the window's rows.
    Returns (rows out [T][d], q [T][.], k [T][.], selected experts per row,
    min router margin per row).
    """
    T = X.shape[0]
    wq, wk, wv, wo = dequant(dense.q), dequant(dense.k), dequant(dense.v), dequant(dense.o)
    xs = [np.asarray(X[t], dtype=np.float64) for t in range(T)]
    A = [rmsnorm(x) for x in xs]
    qs = [wq @ a for a in A]
    ks = [wk @ a for a in A]
    vs = [wv @ a for a in A]
    for t in range(T):
        append_kv(kc, vc, ks[t], vs[t], int(slots[t]), int(positions[t]))
    outs, sels, margins = [], [], []
    for t in range(T):
        att = attention_row(qs[t], kc, vc, int(slots[t]), int(positions[t]), dense.heads)
        x1 = xs[t] + wo @ att
        b = rmsnorm(x1)
        y, sel, _ = moe_row(b, moe)
        outs.append(x1 + y)
        sels.append(sel)
        margins.append(topk_margin(b, moe.router_w, moe.router_b, moe.top_k))
    return np.stack(outs), qs, ks, sels, margins


def stack_window(X: np.ndarray, dense: List[ODenseLayer], moe: List[OMoELayer], kcs: List[np.ndarray],
                 vcs: List[np.ndarray], slots: Sequence[int], positions: Sequence[int]):
    """A window through every layer (caches updated in place).  Returns (y [T][d],
    per-layer q, per-layer k, per-layer selected experts, min margin per row)."""
    h = np.asarray(X, dtype=np.float64)
    Q, K, S = [], [], []
    margin = np.full(X.shape[0], np.inf)
    for dl, ml, kc, vc in zip(dense, moe, kcs, vcs):
        h, q, k, sel, m = decoder_layer_window(h, dl, ml, kc, vc, slots, positions)
        Q.append(q)
        K.append(k)
        S.append(sel)
        margin = np.minimum(margin, m)
    return h, Q, K, S, margin
