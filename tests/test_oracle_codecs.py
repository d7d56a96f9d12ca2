"""Pins of the oracle's element and scale codecs against facts fixed outside
the oracle: the E2M1 grid the pages print, PyTorch's float8_e4m3fn codec and
ml_dtypes' float4_e2m1fn codec (library special cases), exact rational
arithmetic, and hand-worked round-to-nearest-even ties."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def test_e2m1_decode_is_the_printed_grid():
    for code, val in _read_golden("e2m1_grid.txt"):
        got = oracle.e2m1_decode(int(code))
        exp = float(val)
        assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (code, got, exp)


def test_e2m1_ties_and_saturation():
    for v, code in _read_golden("e2m1_rne_ties.txt"):
        assert oracle.e2m1_encode(float(v)) == int(code), v


def test_e2m1_encode_is_nearest_on_grid():
    # Brute force: for many values the encoded grid point is a nearest grid point.
    grid = [oracle.e2m1_decode(c) for c in range(8)]
    rng = np.random.default_rng(0)
    for v in rng.uniform(-7, 7, 4000).astype(np.float32):
        c = oracle.e2m1_encode(float(v))
        got = oracle.e2m1_decode(c)
        best = min(abs(abs(float(v)) - g) for g in grid)
        if abs(v) <= 6:
            assert abs(abs(float(v)) - abs(got)) == best
        else:
            assert abs(got) == 6.0
        assert (got < 0) == (v < 0) or got == 0


def test_e2m1_encode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-6, 6, 3000), np.arange(-6, 6.01, 0.25)]).astype(np.float32)
    ref = vals.astype(ml.float4_e2m1fn).astype(np.float32)
    for v, r in zip(vals, ref):
        assert oracle.e2m1_decode(oracle.e2m1_encode(float(v))) == r, v


def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == float(ref[c]) and math.copysign(1, got) == math.copysign(1, ref[c]), c


def test_e4m3_format_constants():
    # largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(2)
    mag = np.exp2(rng.uniform(-12, math.log2(448), 20000))
    sign = np.where(rng.random(20000) < 0.5, -1.0, 1.0)
    vals = (mag * sign).astype(np.float32)
    # every midpoint between neighbouring codes (ties to even)
    pos = np.array([oracle.e4m3_decode(c) for c in range(127)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids, pos.astype(np.float32)])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(vals[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_encode_saturates_and_keeps_signed_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-9) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00
    # half of the smallest subnormal is a tie: rounds to the even code 0
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02


def test_e8m0_decodes_to_powers_of_two():
    # "Los factores de escala de bloque se almacenan en UE8M0, lo que los
    # restringe a potencias de dos" (NVFP4 pretraining page, "Que es realmente NVFP4")
    for c in range(255):
        v = oracle.e8m0_decode(c)
        m, e = math.frexp(v)
        assert m == 0.5 and e - 1 == c - 127
    assert math.isnan(oracle.e8m0_decode(255))


def test_mxfp8_block_exponent_brute_force_all_bf16():
    """For every positive finite bf16 amax, the oracle's shared exponent is the
    smallest e in [-127, 127] with amax <= 448 * 2^e (exact rationals)."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    for v in vals[::1]:
        fv = Fraction(float(v))
        e = max(-127, math.floor(math.log2(float(v) / 448.0)) - 2)
        while fv > 448 * Fraction(2) ** e:
            e += 1
        e = min(max(e, -127), 127)
        assert oracle.mxfp8_block_exp(float(v)) == e, float(v)
    assert oracle.mxfp8_block_exp(0.0) == -127


def test_bf16_round_trip_helpers():
    x = np.array([1.0, -2.5, 3.3, 1e-40, 65504.0, 1.00390625, 1.005859375], np.float32)
    b = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)
    assert np.array_equal(oracle.bf16_to_f32(b), torch.from_numpy(x).to(torch.bfloat16).float().numpy())
