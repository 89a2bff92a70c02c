"""GPU parity of the output head, the token draw and the proposal check
against the oracle in oracle/head.py, through the C ABI.

Logits must be within 2e-3 x RMS of the fp64 oracle's.  A token is an integer
decided by floating point, so it is compared where the decision is robust:
a greedy row's token must equal the oracle's argmax when the oracle's gap
between the two largest logits exceeds twice the largest logit error seen, and
otherwise be a token whose oracle logit is within that bound of the maximum; a
sampled row's token must equal the oracle's inverse-CDF token when the row's
uniform lies farther than a bound (from the logit error and fp32 summation)
from both edges of that token's CDF interval, and otherwise be a token whose
interval comes within the bound of the uniform.  The slots' emitted counts are
integers computed from the tokens: they must equal the oracle's check applied
to the GPU's tokens, and the oracle's own counts when every token was robust.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import head as oh
from slot_decode_window_gb300 import workloads as wlm
from tests.helpers import oqmat

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def B():
    from slot_decode_window_gb300 import binding, build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    return binding


def _rows(T, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, d)).astype(np.float32)


def _check_tokens(lg_gpu, lg_ref, tokens, temps, seeds, positions):
    """Per-row robust comparison; returns the rows whose oracle decision was robust."""
    err = np.abs(lg_gpu - lg_ref).max(axis=1)
    robust = []
    for t in range(lg_ref.shape[0]):
        ref, tok, tau = lg_ref[t], int(tokens[t]), float(temps[t])
        assert 0 <= tok < ref.size
        delta = 2.0 * err[t] + 1e-12
        if tau <= 0:
            best = int(np.argmax(ref))
            top2 = np.sort(ref)[-2:]
            if top2[1] - top2[0] > delta:
                assert tok == best, f"row {t}: greedy token {tok} != {best}"
                robust.append(t)
            else:
                assert ref[tok] >= ref.max() - delta
        else:
            z = ref / tau
            p = np.exp(z - z.max())
            cdf = np.cumsum(p / p.sum())
            u = oh.row_uniform(int(seeds[t]), int(positions[t]))
            want = oh.draw_token(ref, tau, int(seeds[t]), int(positions[t]))
            eps = 4.0 * delta / tau + 1e-4
            lo = cdf[want - 1] if want > 0 else 0.0
            if u - lo > eps and cdf[want] - u > eps:
                assert tok == want, f"row {t}: drawn token {tok} != {want}"
                robust.append(t)
            else:
                lo_t = cdf[tok - 1] if tok > 0 else 0.0
                assert lo_t - eps <= u <= cdf[tok] + eps, f"row {t}: token {tok} far from the draw"
    return robust


def _case(B, V, d, bits, block, T, temps, fed_fn, seed=0, check_logits=True):
    W = wlm.make_head(V, d, bits, block, seed=seed, cfg_id=70 + bits, device="cuda")
    head = B.Head(W, max_rows=8)
    try:
        x = _rows(T, d, seed + 1)
        Wo = oqmat(W)
        ref = np.stack([oh.head_logits(x[t], Wo) for t in range(T)])
        positions = np.arange(100, 100 + T, dtype=np.int32) * 7
        seeds = np.array([1234567 + 31 * t for t in range(T)], dtype=np.int64)
        want = [oh.draw_token(ref[t], float(temps[t]), int(seeds[t]), int(positions[t])) for t in range(T)]
        fed = np.array(fed_fn(want), dtype=np.int32)
        args = [torch.from_numpy(a).cuda() for a in (positions, seeds, np.asarray(temps, np.float32), fed)]
        tok, nem, lg = head.forward(torch.from_numpy(x).cuda(), *args, logits=True)
        head.sync()
        tok, nem, lg = tok.cpu().numpy(), nem.cpu().numpy(), lg.cpu().numpy().astype(np.float64)
        if check_logits:
            rms = np.sqrt(np.mean(ref * ref))
            assert np.abs(lg - ref).max() <= TOL * rms
        robust = _check_tokens(lg, ref, tok, temps, seeds, positions)
        assert list(nem) == oh.verify_slots(list(tok), list(fed))
        if len(robust) == T:
            assert list(nem) == oh.verify_slots(want, list(fed))
        # the same window again: bit for bit
        tok2, nem2, lg2 = head.forward(torch.from_numpy(x).cuda(), *args, logits=True)
        head.sync()
        assert np.array_equal(tok2.cpu().numpy(), tok) and np.array_equal(nem2.cpu().numpy(), nem)
        assert np.array_equal(lg2.cpu().numpy().astype(np.float64), lg)
        return tok, nem, want, fed
    finally:
        head.close()


def _pairs_fed(accept):
    """Slots of (token row, proposal row): the proposal is the oracle's token of
    the slot's first row where accept[s] (so it should be accepted), else another token."""
    def f(want):
        fed = []
        for s in range(len(want) // 2):
            fed += [-1, want[2 * s] if accept[s] else (want[2 * s] + 1)]
        return fed
    return f


@pytest.mark.parametrize("bits,block,d", [(4, 32, 256), (2, 16, 512)])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_small_head_greedy_and_sampled(B, bits, block, d, T):
    temps = [0.0 if t % 2 == 0 else 0.8 for t in range(T)]
    tok, nem, want, fed = _case(B, 4096, d, bits, block, T, temps, lambda w: [-1] * len(w))
    assert list(nem) == [1] * T


def test_small_head_mtp_slots_accept_and_reject(B):
    T = 8
    temps = [0.0, 0.0, 0.7, 0.7, 0.0, 1.3, 0.9, 0.0]
    accept = [True, False, True, True]
    tok, nem, want, fed = _case(B, 4096, 256, 4, 32, T, temps, _pairs_fed(accept), seed=3)
    # an accepted proposal whose slot's first token was robust emits two tokens
    for s in range(4):
        if tok[2 * s] == want[2 * s]:
            assert nem[2 * s] == (2 if accept[s] else 1)
        assert nem[2 * s + 1] == 0


def test_full_vocabulary_head_t8_mtp_slots(B):
    """The stack model shape's head: d 2048, V 151,936, 4-bit/32, a T = 8 window
    of 4 slots x (token, proposal), greedy and sampled rows."""
    temps = [0.0, 0.0, 0.6, 0.6, 1.0, 1.0, 0.0, 0.0]
    _case(B, wlm.HEAD_VOCAB, 2048, 4, 32, 8, temps, _pairs_fed([True, True, False, True]), seed=5)


def test_head_argument_errors(B):
    W = wlm.make_head(256, 256, 4, 32, seed=0, cfg_id=74, device="cuda")
    head = B.Head(W, max_rows=4)
    try:
        x = torch.zeros(8, 256, device="cuda")
        z = torch.zeros(8, dtype=torch.int32, device="cuda")
        zs = torch.zeros(8, dtype=torch.int64, device="cuda")
        zf = torch.zeros(8, device="cuda")
        di = B.strata_draw_in(z.data_ptr(), zs.data_ptr(), zf.data_ptr(), z.data_ptr())
        do = B.strata_draw_out(z.data_ptr(), z.data_ptr(), None)
        assert B.strata_head_forward(head.handle, x.data_ptr(), 5, di, do) == B.STRATA_EINVAL
        assert B.strata_head_forward(head.handle, x.data_ptr(), 0, di, do) == B.STRATA_EINVAL
        bad = B.strata_draw_out(None, z.data_ptr(), None)
        assert B.strata_head_forward(head.handle, x.data_ptr(), 2, di, bad) == B.STRATA_EINVAL
        assert B.strata_head_sync(head.handle) == B.STRATA_OK
    finally:
        head.close()
