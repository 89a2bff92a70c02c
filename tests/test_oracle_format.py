"""Pins of the oracle's block-format decoding (no GPU)."""
import os

import numpy as np
import pytest
import torch

import oracle
from slot_decode_window_gb300 import workloads as wlm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_blocks.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split("|")
            bits, block, s_hex, m_hex, codes_hex = head.split()
            cases.append((int(bits), int(block), int(s_hex, 16), int(m_hex, 16),
                          bytes.fromhex(codes_hex), [float(v) for v in vals.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases())
def test_dequant_hand_derived_blocks(case):
    bits, block, s, m, codes, expected = case
    q = oracle.OQMat(np.frombuffer(codes, np.uint8).reshape(1, 1, -1),
                     np.array([[[s]]], np.uint16), np.array([[[m]]], np.uint16), 1, block, bits, block)
    np.testing.assert_array_equal(oracle.dequant(q)[0], np.array(expected))


def _bit_loop_unpack(codes_row: bytes, cols: int, bits: int):
    """Element i read bit by bit from the packed bytes (pure Python)."""
    out = []
    for i in range(cols):
        v = 0
        for b in range(bits):
            bit = i * bits + b
            v |= ((codes_row[bit // 8] >> (bit % 8)) & 1) << b
        out.append(v)
    return out


@pytest.mark.parametrize("bits", [4, 2])
def test_unpack_matches_bitwise_reading(bits):
    rng = np.random.default_rng(3)
    cols = 96
    codes = rng.integers(0, 256, size=(3, cols * bits // 8), dtype=np.uint8)
    q = oracle.unpack_codes(codes, cols, bits)
    for r in range(3):
        assert list(q[r]) == _bit_loop_unpack(bytes(codes[r]), cols, bits)


def test_fp16_bits_exact():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 65504.0, 6.103515625e-05, 5.960464477539063e-08], np.float16)
    np.testing.assert_array_equal(oracle.fp16_bits(vals.view(np.uint16)), vals.astype(np.float64))


@pytest.mark.parametrize("bits,block", [(4, 32), (2, 16)])
def test_quantizer_round_trip_within_half_step(bits, block):
    """dequant(quantize(w)) is within scale/2 (+ fp16 rounding of min) of w, and hits both ends."""
    w = wlm._normal((24, 8 * block), 0.02, 11, "cpu")
    codes, scale, mn = wlm.quantize_blocks(w, bits, block)
    q = oracle.OQMat(codes.numpy()[None], scale.numpy().view(np.uint16)[None],
                     mn.numpy().view(np.uint16)[None], 24, 8 * block, bits, block)
    back = oracle.dequant(q)
    s = np.repeat(oracle.fp16_bits(q.scale[0]), block, axis=1)
    m16 = np.repeat(oracle.fp16_bits(q.min[0]), block, axis=1)
    w64 = w.numpy().astype(np.float64)
    lo = np.repeat(w64.reshape(24, -1, block).min(axis=2), block, axis=1)
    # error bound: half a step, plus the min's own fp16 rounding, plus the scale's
    bound = s / 2 + np.abs(m16 - lo) + np.abs(s) * ((1 << bits) - 1) * 2 ** -11 + 1e-12
    assert np.all(np.abs(back - w64) <= bound)
    qi = oracle.unpack_codes(q.codes[0], q.cols, bits).reshape(24, -1, block)
    assert np.all(qi.min(axis=2) == 0) and np.all(qi.max(axis=2) >= (1 << bits) - 2)


def test_quantizer_constant_block_gives_zero_scale():
    w = torch.full((2, 32), 0.3)
    codes, scale, mn = wlm.quantize_blocks(w, 4, 32)
    assert int(scale.view(torch.uint8).sum()) == 0 and int(codes.sum()) == 0
    q = oracle.OQMat(codes.numpy()[None], scale.numpy().view(np.uint16)[None],
                     mn.numpy().view(np.uint16)[None], 2, 32, 4, 32)
    np.testing.assert_array_equal(oracle.dequant(q), np.float64(np.float16(0.3)))
