"""Seeded synthetic workloads for the batched verify-window MoE step.

This module only *draws* inputs: router weights, block-quantized expert
weights and hidden rows.  It holds none of the window's arithmetic (no
router GEMV, no dequantization, no expert FFN).  The one place where a
window's arithmetic would be needed -- keeping each row's top-k logit margin
above a floor -- is delegated to a caller-supplied ``accept_row`` predicate.

Quantized format (a reading: the Strata pages name block formats such as
UD-Q4_K_XL, Q2_0 and IQ3_S but define none of them): a matrix ``[rows][cols]``
is cut along ``cols`` into blocks of ``block`` consecutive elements; each block
stores ``block*bits/8`` bytes of codes plus one fp16 ``scale`` and one fp16
``min``; the weight value is ``scale*q + min``.  Codes are packed row-major,
element ``i`` of a row in byte ``i*bits//8``, least-significant bits first
(for 4-bit: even element in the low nibble).  Scales and mins are fp16 bit
patterns ``[rows][cols/block]``.

Workloads (the sizes of the window the Strata docs describe: at most 8 rows
per verify window, "BATCHING.md", section "Several requests at once (batch
slots)"; two rows per slot with --batch-mtp, same page, --batch-mtp paragraph):

* ``tiny``    d=256,  E=8 top-2,   F=128,  shared 128,  4-bit/32, T=2
* ``mid``     d=2048, E=128 top-8, F=768,  shared 768,  4-bit/32, T in 1,2,4,8
* ``zipf``    d=4096, E=160 top-8, F=1536, shared 1536, 4-bit/32, T=8 as
               4 slots x (token, MTP proposal = token + N(0, 0.1) noise),
               log-Zipf(1.1) router bias so rows share experts
* ``lowbit``  d=4096, E=256 top-8, F=2048, shared 2048, 2-bit/16, T in 1,2,4,8
* ``stack48`` 48 layers of dense 4-bit q/k/v/o (2048 -> 4096/512/512,
               4096 -> 2048) + the ``mid`` MoE block, T=8

Weights are N(0, 0.02) before quantization; hidden rows are N(0, 1) drawn in
fp64 and rounded to fp32; the router is fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, Optional, Sequence, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoESpec:
    """Shape of one MoE layer of a verify window."""
    hidden: int
    n_experts: int
    top_k: int
    ffn: int
    shared_ffn: int
    bits: int
    block: int
    renorm_topk: int = 0
    zipf_bias: float = 0.0  # 0 = no router bias; s > 0 = -s*ln(rank) bias

    @property
    def kstep(self) -> int:
        return 64 if self.bits == 4 else 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    moe: MoESpec
    rows: Tuple[int, ...]          # the T values the workload is run at
    mtp_pairs: bool = False        # rows are (token, proposal) per slot
    n_layers: int = 1              # > 1: dense projections + MoE per layer
    heads: int = 32
    kv_heads: int = 4
    head_dim: int = 128


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, MoESpec(256, 8, 2, 128, 128, 4, 32), (2,)),
    "mid": Workload("mid", 2, MoESpec(2048, 128, 8, 768, 768, 4, 32), (1, 2, 4, 8)),
    "zipf": Workload("zipf", 3, MoESpec(4096, 160, 8, 1536, 1536, 4, 32, zipf_bias=1.1), (8,),
                     mtp_pairs=True),
    "stack48": Workload("stack48", 4, MoESpec(2048, 128, 8, 768, 768, 4, 32), (8,), n_layers=48),
    "lowbit": Workload("lowbit", 5, MoESpec(4096, 256, 8, 2048, 2048, 2, 16), (1, 2, 4, 8)),
}

WEIGHT_STD = 0.02
PROPOSAL_NOISE_STD = 0.1

# tensor ids for seed derivation
_T_ROUTER, _T_BIAS, _T_GATE, _T_UP, _T_DOWN, _T_SGATE, _T_SUP, _T_SDOWN = range(8)
_T_Q, _T_K, _T_V, _T_O = range(8, 12)


def derive_seed(*words: int) -> int:
    """A 63-bit seed from a tuple of non-negative integers (SeedSequence)."""
    state = np.random.SeedSequence([int(w) for w in words]).generate_state(2, np.uint32)
    return (int(state[0]) << 31) ^ int(state[1])


def _normal(shape: Sequence[int], std: float, seed: int, device: str) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std


def quantize_blocks(w: torch.Tensor, bits: int, block: int):
    """Encode an fp32 matrix ``[rows][cols]`` as (codes, scale, min).

    Per block: ``scale = fp16((hi-lo)/(2^bits-1))``, ``min = fp16(lo)``,
    ``q = clip(round_half_even((w - min)/scale), 0, 2^bits-1)`` using the
    fp16-rounded scale and min; a zero scale gives q = 0.
    Returns codes uint8 ``[rows][cols*bits/8]`` and fp16 bit patterns as
    int16 ``[rows][cols/block]``.
    """
    rows, cols = w.shape
    assert cols % block == 0
    levels = (1 << bits) - 1
    wb = w.reshape(rows, cols // block, block)
    lo = wb.amin(dim=2)
    hi = wb.amax(dim=2)
    scale16 = ((hi - lo) / levels).to(torch.float16)
    min16 = lo.to(torch.float16)
    s = scale16.to(torch.float32).unsqueeze(2)
    m = min16.to(torch.float32).unsqueeze(2)
    safe = torch.where(s == 0, torch.ones_like(s), s)
    q = torch.round((wb - m) / safe).clamp_(0, levels)
    q = torch.where(s == 0, torch.zeros_like(q), q).to(torch.uint8).reshape(rows, cols)
    per_byte = 8 // bits
    qv = q.reshape(rows, cols // per_byte, per_byte).to(torch.int32)
    packed = torch.zeros(rows, cols // per_byte, dtype=torch.int32, device=w.device)
    for i in range(per_byte):
        packed |= qv[:, :, i] << (bits * i)
    return (packed.to(torch.uint8).contiguous(),
            scale16.view(torch.int16).contiguous(),
            min16.view(torch.int16).contiguous())


@dataclasses.dataclass
class QMat:
    """A stack of quantized matrices ``[n][rows][cols]`` in the block format."""
    codes: torch.Tensor   # uint8 [n][rows][cols*bits/8]
    scale: torch.Tensor   # int16 (fp16 bits) [n][rows][cols/block]
    min: torch.Tensor     # int16 (fp16 bits) [n][rows][cols/block]
    rows: int
    cols: int
    bits: int
    block: int

    def to(self, device) -> "QMat":
        return QMat(self.codes.to(device), self.scale.to(device), self.min.to(device),
                    self.rows, self.cols, self.bits, self.block)

    @property
    def nbytes(self) -> int:
        return self.codes.numel() + 2 * self.scale.numel() + 2 * self.min.numel()


def make_qmat(n: int, rows: int, cols: int, bits: int, block: int, seeds: Sequence[int],
              device: str) -> QMat:
    codes = torch.empty(n, rows, cols * bits // 8, dtype=torch.uint8, device=device)
    scale = torch.empty(n, rows, cols // block, dtype=torch.int16, device=device)
    mn = torch.empty(n, rows, cols // block, dtype=torch.int16, device=device)
    for i in range(n):
        w = _normal((rows, cols), WEIGHT_STD, seeds[i], device)
        c, s, m = quantize_blocks(w, bits, block)
        codes[i].copy_(c)
        scale[i].copy_(s)
        mn[i].copy_(m)
    return QMat(codes, scale, mn, rows, cols, bits, block)


@dataclasses.dataclass
class MoELayer:
    spec: MoESpec
    router_w: torch.Tensor            # fp32 [E][d]
    router_b: Optional[torch.Tensor]  # fp32 [E] or None
    gate: QMat                        # [E][F][d]
    up: QMat                          # [E][F][d]
    down: QMat                        # [E][d][F]
    shared_gate: Optional[QMat]       # [1][Fs][d]
    shared_up: Optional[QMat]
    shared_down: Optional[QMat]       # [1][d][Fs]

    def to(self, device) -> "MoELayer":
        f = lambda q: None if q is None else q.to(device)
        return MoELayer(self.spec, self.router_w.to(device),
                        None if self.router_b is None else self.router_b.to(device),
                        f(self.gate), f(self.up), f(self.down),
                        f(self.shared_gate), f(self.shared_up), f(self.shared_down))

    @property
    def expert_bytes(self) -> int:
        """Bytes of one routed expert's gate+up+down blocks."""
        return (self.gate.nbytes + self.up.nbytes + self.down.nbytes) // self.spec.n_experts

    @property
    def shared_bytes(self) -> int:
        if self.shared_gate is None:
            return 0
        return self.shared_gate.nbytes + self.shared_up.nbytes + self.shared_down.nbytes


def zipf_bias(n_experts: int, s: float, seed: int) -> np.ndarray:
    """Router bias -s*ln(rank_e), ranks 1..E from a seeded permutation."""
    rng = np.random.default_rng(seed)
    ranks = rng.permutation(n_experts) + 1
    return (-s * np.log(ranks.astype(np.float64))).astype(np.float32)


def make_moe_layer(spec: MoESpec, seed: int = 0, cfg_id: int = 0, layer: int = 0,
                   device: str = "cpu") -> MoELayer:
    E, d, F, Fs = spec.n_experts, spec.hidden, spec.ffn, spec.shared_ffn
    sd = lambda tid, i=0: derive_seed(seed, cfg_id, layer, tid, i)
    router_w = _normal((E, d), WEIGHT_STD, sd(_T_ROUTER), device)
    router_b = None
    if spec.zipf_bias > 0:
        router_b = torch.from_numpy(zipf_bias(E, spec.zipf_bias, sd(_T_BIAS))).to(device)
    b, B = spec.bits, spec.block
    gate = make_qmat(E, F, d, b, B, [sd(_T_GATE, e) for e in range(E)], device)
    up = make_qmat(E, F, d, b, B, [sd(_T_UP, e) for e in range(E)], device)
    down = make_qmat(E, d, F, b, B, [sd(_T_DOWN, e) for e in range(E)], device)
    sg = su = sdn = None
    if Fs > 0:
        sg = make_qmat(1, Fs, d, b, B, [sd(_T_SGATE)], device)
        su = make_qmat(1, Fs, d, b, B, [sd(_T_SUP)], device)
        sdn = make_qmat(1, d, Fs, b, B, [sd(_T_SDOWN)], device)
    return MoELayer(spec, router_w, router_b, gate, up, down, sg, su, sdn)


@dataclasses.dataclass
class DenseLayer:
    """Dense 4-bit q/k/v/o projections of one decoder layer."""
    q: QMat   # [1][H*Dh][d]
    k: QMat   # [1][Hkv*Dh][d]
    v: QMat   # [1][Hkv*Dh][d]
    o: QMat   # [1][d][H*Dh]

    def to(self, device) -> "DenseLayer":
        return DenseLayer(self.q.to(device), self.k.to(device), self.v.to(device), self.o.to(device))


def make_dense_layer(wl: Workload, seed: int, layer: int, device: str) -> DenseLayer:
    d = wl.moe.hidden
    b, B = wl.moe.bits, wl.moe.block
    qd, kvd = wl.heads * wl.head_dim, wl.kv_heads * wl.head_dim
    sd = lambda tid: derive_seed(seed, wl.cfg_id, layer, tid, 0)
    return DenseLayer(make_qmat(1, qd, d, b, B, [sd(_T_Q)], device),
                      make_qmat(1, kvd, d, b, B, [sd(_T_K)], device),
                      make_qmat(1, kvd, d, b, B, [sd(_T_V)], device),
                      make_qmat(1, d, qd, b, B, [sd(_T_O)], device))


# The output head of the 48-layer stack's model shape: d = 2048 and a
# vocabulary of 151,936 tokens (a reading: the pages name no vocabulary; this is
# the vocabulary of the model family whose layer shapes the stack workload
# has), 4-bit/32 blocks like the dense weights.
HEAD_VOCAB = 151936
_T_HEAD = 12


def make_head(vocab: int, hidden: int, bits: int, block: int, seed: int, cfg_id: int, device: str) -> QMat:
    """A head weight [1][vocab][hidden] in the block format, N(0, 0.02) before quantization."""
    return make_qmat(1, vocab, hidden, bits, block, [derive_seed(seed, cfg_id, 0, _T_HEAD, 0)], device)


AcceptFn = Callable[[np.ndarray], bool]


def hidden_row(seed: int, cfg_id: int, window: int, row: int, attempt: int, d: int) -> np.ndarray:
    """One hidden row ~ N(0, 1), drawn in fp64 and rounded to fp32."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, cfg_id, 1000 + window, row, attempt]))
    return rng.standard_normal(d).astype(np.float32)


def proposal_noise(seed: int, cfg_id: int, window: int, slot: int, attempt: int, d: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, cfg_id, 50000 + window, slot, attempt]))
    return (rng.standard_normal(d) * PROPOSAL_NOISE_STD).astype(np.float32)


def make_window(wl: Workload, T: int, seed: int = 0, window: int = 0,
                accept_row: Optional[AcceptFn] = None, max_attempts: int = 1000) -> np.ndarray:
    """Hidden rows ``[T][d]`` fp32 of one verify window.

    Rows failing ``accept_row`` are redrawn from the next substream.  For a
    workload of MTP pairs, row 2s is slot s's token and row 2s+1 its proposal
    (token + N(0, 0.1) noise, added in fp32); a failing proposal redraws
    only its noise.
    """
    d = wl.moe.hidden
    x = np.empty((T, d), dtype=np.float32)
    ok = accept_row if accept_row is not None else (lambda r: True)
    if wl.mtp_pairs:
        assert T % 2 == 0
        for s in range(T // 2):
            for a in range(max_attempts):
                tok = hidden_row(seed, wl.cfg_id, window, 2 * s, a, d)
                if ok(tok):
                    break
            else:
                raise RuntimeError("no acceptable token row")
            for a in range(max_attempts):
                prop = tok + proposal_noise(seed, wl.cfg_id, window, s, a, d)
                if ok(prop):
                    break
            else:
                raise RuntimeError("no acceptable proposal row")
            x[2 * s], x[2 * s + 1] = tok, prop
        return x
    for t in range(T):
        for a in range(max_attempts):
            r = hidden_row(seed, wl.cfg_id, window, t, a, d)
            if ok(r):
                x[t] = r
                break
        else:
            raise RuntimeError("no acceptable row")
    return x
