"""Pins of the oracle's SwiGLU, h = RN_bf16(silu(g) * u) with
silu(g) = g / (1 + e^-g) ("Miles Blackwell RL Cambia la Uniformidad BF16 por
MXFP8 y NVFP4 Nativos", section "Un Cuantizador Compartido Es el Mecanismo
Real": gate and up of a SwiGLU expert come out of one fused GEMM).

The reference here is independent of the oracle's binary64 evaluation: the
exact value is computed with Python's `decimal` at 80 significant digits
(its exp is correctly rounded at that precision) and rounded to bf16 by
comparing it with the exact decimal values of the neighbouring bf16 codes.
Also pinned: g = 0, the large-|g| limits, hand-made ties of the final bf16
cast, and the identity silu(g) - silu(-g) = g."""
import struct
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle

getcontext().prec = 80


def _bf16_value(bits):
    """Exact Decimal value of a bf16 bit pattern (finite)."""
    return Decimal(struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0])


def _bf16_of_float(x):
    return struct.unpack("<I", struct.pack("<f", x))[0] >> 16


def _rn_bf16(v):
    """Nearest bf16 to the Decimal v (exact comparison with the neighbours;
    ties to even -- never met for the irrational values compared here)."""
    if v == 0:
        return 0x8000 if v.is_signed() else 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a >= Decimal(2) ** 128 - Decimal(2) ** 119:    # max + half a unit and above: infinity
        return sign | 0x7F80
    base = min(_bf16_of_float(float(a)), 0x7F7F)        # near a; magnitudes are monotonic in the code
    best = None
    for c in range(max(0, base - 2), min(0x7F7F, base + 2) + 1):
        d = abs(_bf16_value(c) - a)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return sign | best[1]


def _silu_mul_exact(g_bits, u_bits):
    g, u = _bf16_value(g_bits), _bf16_value(u_bits)
    return g / (1 + (-g).exp()) * u


def _oracle_h(g_bits, u_bits):
    g_bits = np.asarray(g_bits, np.uint16).reshape(-1)
    u_bits = np.asarray(u_bits, np.uint16).reshape(-1)
    gu = np.concatenate([g_bits[:, None], u_bits[:, None]], axis=1)   # rows of [g | u], F = 1
    return oracle.swiglu(gu).reshape(-1)


def _bits(values):
    return oracle.f32_to_bf16(np.asarray(values, np.float32))


def test_matches_exact_rounding_on_random_and_swept_inputs():
    """Every bf16 g in [-120, 120] with step 1/8 on a coarse grid plus random
    bf16 pairs across magnitudes: the oracle equals the correctly rounded
    exact value bit for bit."""
    rng = np.random.default_rng(20)
    g_sweep = np.arange(-120.0, 120.0, 0.125, dtype=np.float32)
    u_sweep = rng.normal(0, 2, g_sweep.size).astype(np.float32)
    g_rand = (rng.normal(0, 1, 6000) * 10.0 ** rng.integers(-3, 2, 6000)).astype(np.float32)
    u_rand = (rng.normal(0, 1, 6000) * 10.0 ** rng.integers(-30, 30, 6000)).astype(np.float32)
    gb = np.concatenate([_bits(g_sweep), _bits(g_rand)])
    ub = np.concatenate([_bits(u_sweep), _bits(u_rand)])
    got = _oracle_h(gb, ub)
    want = np.array([_rn_bf16(_silu_mul_exact(g, u)) for g, u in zip(gb, ub)], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(gb[i]), hex(ub[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_gate_and_up_are_not_interchangeable():
    """silu is applied to the gate half (the first F columns), not the up half."""
    g, u = _bits([3.0, -2.0]), _bits([-2.0, 3.0])
    h = _oracle_h(g, u)
    assert [_rn_bf16(_silu_mul_exact(a, b)) for a, b in zip(g, u)] == list(h)
    assert _rn_bf16(_silu_mul_exact(u[0], g[0])) != h[0]


def test_zero_gate_gives_zero():
    g = _bits([0.0] * 4)
    u = _bits([1.0, -3.5, 1e30, -1e-30])
    h = _oracle_h(g, u)
    assert all((int(x) & 0x7FFF) == 0 for x in h)


def test_large_gate_limits():
    """silu(g) -> g for large g (h = RN(g u) when g u is not a tie) and
    silu(g) -> 0 for very negative g."""
    g = _bits([40.0, 64.0, 1000.0, 3.0e38])
    u = _bits([1.5, -0.75, 2.0, 1.0])
    h = _oracle_h(g, u)
    assert list(h) == list(_bits([60.0, -48.0, 2000.0, 3.0e38]))
    gn = _bits([-200.0, -1000.0, -3.0e38])
    un = _bits([1.0, -2.0, 5.0])
    hn = _oracle_h(gn, un)
    assert all((int(x) & 0x7FFF) == 0 for x in hn)
    assert [int(x) >> 15 for x in hn] == [1, 0, 1]      # silu(g) < 0: the sign of -u


@pytest.mark.parametrize("g,u,want", [
    # g u = 96.75, halfway between 96.5 (odd code) and 97.0 (even code); the
    # exact value lies just below 96.75, so 96.5 (ties-to-even would give 97)
    (96.0, 1.0078125, 96.5),
    (96.0, -1.0078125, -96.5),
    # g u = 98.25 lies halfway between 98.0 (even code) and 98.5 (odd): 98.0
    # either way
    (96.0, 1.0234375, 98.0),
    # moderate g: e^-g still moves the value visibly below the tie
    (24.0, 1.0078125, 24.1875 - 0.0625),
])
def test_ties_of_the_final_cast_go_toward_zero(g, u, want):
    gb, ub = _bits([g]), _bits([u])
    exact = _silu_mul_exact(gb[0], ub[0])
    prod = _bf16_value(gb[0]) * _bf16_value(ub[0])
    assert abs(exact) < abs(prod)                       # silu(g) < g for g > 0
    assert _rn_bf16(exact) == _bits([want])[0]
    assert _oracle_h(gb, ub)[0] == _bits([want])[0]


def test_silu_difference_identity():
    """silu(g) - silu(-g) = g: with u = 1 the two outputs are each within half
    a bf16 unit of silu(+-g), so their difference is within one unit of g."""
    rng = np.random.default_rng(5)
    g = _bits(rng.normal(0, 4, 3000).astype(np.float32))
    gneg = g ^ np.uint16(0x8000)
    one = _bits(np.ones(g.size, np.float32))
    hp = oracle.bf16_to_f32(_oracle_h(g, one)).astype(np.float64)
    hm = oracle.bf16_to_f32(_oracle_h(gneg, one)).astype(np.float64)
    gv = oracle.bf16_to_f32(g).astype(np.float64)

    def unit(x):
        return 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126))) - 7)
    err = np.abs(hp - hm - gv)
    assert (err <= 0.5 * unit(hp) + 0.5 * unit(hm)).all()
    # and the sign convention: silu(g) > 0 for g > 0, silu(g) < 0 for g < 0
    assert (np.sign(hp[gv > 0]) > 0).all() and (np.sign(hp[gv < -0.01]) < 0).all()
