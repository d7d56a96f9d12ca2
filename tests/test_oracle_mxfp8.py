"""Pins of the oracle's MXFP8 quantizer (1x32 E4M3 blocks, one E8M0 scale per
block, rowwise and columnwise copies) against a hand-worked block, format
invariants and exact round trips."""
import numpy as np
import torch

import oracle
from moe_mx8_quantize_gb300 import inputs


def bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(vals, dtype=torch.float32)), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def test_worked_block():
    """One 32-element block with amax = 448 * 2^3, so the shared exponent is 3
    (scale code 130) and every element is divided by 8 exactly:
        3584 -> 448        code 0x7E
        8.5  -> 1.0625     tie between 1.0 (0x38) and 1.125 (0x39): even 0x38
        9.5  -> 1.1875     tie between 1.125 and 1.25 (0x3A): even 0x3A
       -9.5  -> -1.1875    0xBA
        3*2^-7 -> 1.5*2^-9 tie between subnormals 2^-9 (1) and 2^-8 (2): 0x02
        2^-7 -> 2^-10      tie between 0 and 2^-9: 0x00
       -2^-7 -> -2^-10     negative tie to zero keeps the sign: 0x80
        0    -> 0x00, and the rest 1.0*8 -> 1.0 (0x38)."""
    vals = [3584.0, 8.5, 9.5, -9.5, 3 * 2.0 ** -7, 2.0 ** -7, -(2.0 ** -7), 0.0] + [8.0] * 24
    x = bf16_bits(vals).reshape(1, 32)
    q, s = oracle.mxfp8_quantize_rowwise(x)
    assert s.tolist() == [[130]]
    assert q[0, :8].tolist() == [0x7E, 0x38, 0x3A, 0xBA, 0x02, 0x00, 0x80, 0x00]
    assert q[0, 8:].tolist() == [0x38] * 24


def test_zero_block_and_signed_zero():
    x = np.zeros((1, 32), np.uint16)
    x[0, 5] = 0x8000  # -0.0
    q, s = oracle.mxfp8_quantize_rowwise(x)
    assert s.tolist() == [[0]]               # e = -127 (clamped), code 0
    assert q[0, 5] == 0x80 and (np.delete(q[0], 5) == 0).all()


def test_bf16_max_block_and_dequant_overflow():
    """bf16 max = 1.9921875 * 2^127: the smallest e with amax <= 448*2^e is 120
    (code 247); amax/2^120 = 255 rounds to 256 (code 0x78); decoding gives
    256 * 2^120 = 2^128, which overflows binary32 to +inf."""
    x = np.zeros((1, 32), np.uint16)
    x[0, 0] = 0x7F7F
    x[0, 1] = 0xFF7F
    q, s = oracle.mxfp8_quantize_rowwise(x)
    assert s.tolist() == [[247]]
    assert q[0, 0] == 0x78 and q[0, 1] == 0xF8
    d = oracle.dequant_mxfp8(q, s)
    assert d[0, 0] == np.inf and d[0, 1] == -np.inf


def test_subnormal_block_hits_exponent_clamp():
    """amax = 2^-133 (a bf16 subnormal) would need e = -141, clamped to -127:
    elements are multiplied by 2^127, so 2^-133 -> 2^-6 (code 0x08)."""
    x = np.zeros((1, 32), np.uint16)
    x[0, 0] = 0x0001       # 2^-133
    x[0, 1] = 0x8001
    q, s = oracle.mxfp8_quantize_rowwise(x)
    assert s.tolist() == [[0]]
    assert q[0, 0] == 0x08 and q[0, 1] == 0x88


def _scale_invariants(x_bits, q, s):
    xf = oracle.bf16_to_f32(x_bits).astype(np.float64)
    R, C = xf.shape
    amax = np.abs(xf.reshape(R, C // 32, 32)).max(-1)
    e = s.astype(np.int64) - 127
    assert (s != 255).all()
    ratio = amax / np.exp2(e)
    # amax maps to at most the E4M3 maximum, and at most one binade is wasted
    assert (ratio <= 448).all()
    clamped = e == -127
    assert ((ratio > 224) | clamped).all()


def test_invariants_on_sweep_mix():
    x = inputs.bits(inputs.sweep(256, 512, seed=5))
    q, s = oracle.mxfp8_quantize_rowwise(x)
    _scale_invariants(x, q, s)
    # no NaN codes for finite input
    assert not ((q & 0x7F) == 0x7F).any()
    # dequantization error is at most half an E4M3 step at that scale, except
    # where 2^e * 448 overflows binary32
    d = oracle.dequant_mxfp8(q, s).astype(np.float64)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    scale = np.repeat(np.exp2(s.astype(np.float64) - 127), 32, axis=1)
    y = np.abs(xf) / scale
    step = np.where(y < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(y, 1e-300))) - 3))
    fin = np.isfinite(d)
    assert (np.abs(d - xf)[fin] <= 0.5 * (step * scale)[fin] * (1 + 1e-12)).all()
    assert (~fin <= (np.abs(xf) > 2.0 ** 127)).all()


def test_round_trip_of_representable_blocks():
    """Blocks made of E4M3 values times 2^e, with one element equal to 448*2^e
    (so the shared exponent is exactly e), dequantize to themselves."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 127, size=(64, 128))
    codes[:, ::32] = 0x7E
    sign = np.where(rng.random((64, 128)) < 0.5, -1.0, 1.0)
    e = rng.integers(-40, 40, size=(64, 4))
    mag = np.array([oracle.e4m3_decode(int(c)) for c in range(127)])[codes]
    xf = (mag * sign * np.repeat(np.exp2(e), 32, axis=1)).astype(np.float32)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(xf))
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.mxfp8_quantize_rowwise(xb)
    assert np.array_equal(s.astype(np.int64) - 127, e)
    assert np.array_equal(oracle.dequant_mxfp8(q, s), xf)


def test_colwise_is_rowwise_of_transpose():
    """The columnwise copy uses 32x1 blocks of the original input, stored
    transposed: it must equal the rowwise quantization of x^T."""
    x = inputs.bits(inputs.sweep(96, 160, seed=6))
    qT, sT = oracle.mxfp8_quantize_colwise(x)
    qr, sr = oracle.mxfp8_quantize_rowwise(np.ascontiguousarray(x.T))
    assert np.array_equal(qT, qr) and np.array_equal(sT, sr)


def test_rowwise_and_colwise_differ_numerically():
    """1x32 and 32x1 blocks group different elements under one scale, so the
    two dequantized copies differ (MXFP8 paragraph of the Miles recipes page)."""
    x = inputs.bits(inputs.pr1()["X"])
    q, s = oracle.mxfp8_quantize_rowwise(x)
    qT, sT = oracle.mxfp8_quantize_colwise(x)
    dr = oracle.dequant_mxfp8(q, s)
    dc = oracle.dequant_mxfp8(qT, sT).T
    assert not np.array_equal(dr, dc)
