"""Pins of the oracle's FP64 block-scaled GEMM references and of its
tensor-core scale layout: exact rational brute force on tiny shapes (decoded
through PyTorch's float8 codec and the printed E2M1 grid, not through the
oracle), one-nonzero closed forms, and an independent reshape-based
construction of the 128x4 scale tiles."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _grid():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_grid.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = Fraction(float(v))
    return vals


E2M1 = _grid()
E4M3 = {c: (None if np.isnan(v) else Fraction(float(v))) for c, v in enumerate(
    torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().tolist())}


def _dec_row(fmt, qrow, srow, K, s32):
    out = []
    for k in range(K):
        if fmt == 0:
            v = E4M3[int(qrow[k])] * Fraction(2) ** (int(srow[k // 32]) - 127)
        else:
            b = int(qrow[k // 2])
            nib = (b >> 4) if k % 2 else (b & 15)
            v = E2M1[nib] * E4M3[int(srow[k // 16])]
        out.append(v * s32)
    return out


def _rand_operands(rng, fmt, rows, K):
    if fmt == 0:
        q = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3C                  # no NaN codes
        s = rng.integers(110, 140, size=(rows, K // 32), dtype=np.uint8)
    else:
        q = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
        s = rng.integers(0, 0x7F, size=(rows, K // 16), dtype=np.uint8)
    return q, s


@pytest.mark.parametrize("fmt,K", [(0, 64), (0, 96), (1, 32), (1, 64)])
def test_gemm_brute_force_exact(fmt, K):
    rng = np.random.default_rng(10 + fmt)
    M, N = 3, 2
    A, SA = _rand_operands(rng, fmt, M, K)
    B, SB = _rand_operands(rng, fmt, N, K)
    a32 = rng.uniform(0.1, 3, M).astype(np.float32) if fmt == 1 else None
    b32 = np.array([0.37], np.float32) if fmt == 1 else None
    ref, absref = oracle.gemm_ref(fmt, A, SA, B, SB, K, a32, b32)
    for m in range(M):
        ar = _dec_row(fmt, A[m], SA[m], K, Fraction(float(a32[m])) if a32 is not None else 1)
        for n in range(N):
            br = _dec_row(fmt, B[n], SB[n], K, Fraction(float(b32[0])) if b32 is not None else 1)
            exact = sum(x * y for x, y in zip(ar, br))
            aexact = sum(abs(x) * abs(y) for x, y in zip(ar, br))
            assert abs(Fraction(ref[m, n]) - exact) <= Fraction(1, 10 ** 12) * aexact + Fraction(1, 10 ** 300)
            assert abs(Fraction(absref[m, n]) - aexact) <= Fraction(1, 10 ** 12) * aexact


def test_gemm_one_nonzero_closed_form():
    """A has a single nonzero at (1, 37), B at (2, 37):
    Y[1,2] = a * b * 2^(sa-127) * 2^(sb-127), every other output is 0."""
    M, N, K = 4, 3, 64
    A = np.zeros((M, K), np.uint8); B = np.zeros((N, K), np.uint8)
    SA = np.full((M, 2), 127, np.uint8); SB = np.full((N, 2), 127, np.uint8)
    A[1, 37] = 0x4C   # E4M3 6.0
    B[2, 37] = 0xB9   # E4M3 -1.125
    SA[1, 1] = 130
    SB[2, 1] = 120
    ref, _ = oracle.gemm_ref(0, A, SA, B, SB, K)
    a = float(E4M3[0x4C]); b = float(E4M3[0xB9])
    want = np.zeros((M, N)); want[1, 2] = a * b * 2.0 ** 3 * 2.0 ** -7
    assert np.array_equal(ref, want)


def test_grouped_gemm_brute_force_with_empty_groups():
    rng = np.random.default_rng(12)
    K, N = 32, 2
    offs = np.array([0, 2, 2, 5, 5])   # groups of 2, 0, 3, 0 rows
    G = len(offs) - 1
    A, SA = _rand_operands(rng, 1, 5, K)
    B, SB = _rand_operands(rng, 1, G * N, K)
    a32 = rng.uniform(0.5, 2, 5).astype(np.float32)
    b32 = rng.uniform(0.5, 2, G).astype(np.float32)
    pairs = np.array([(m, n) for m in range(5) for n in range(N)])
    ref, _ = oracle.grouped_gemm_ref(1, offs, A, SA, B.reshape(G, N, K // 2), SB, K, a32, b32, pairs)
    for p, (m, n) in enumerate(pairs):
        g = [h for h in range(G) if offs[h] <= m < offs[h + 1]][0]
        ar = _dec_row(1, A[m], SA[m], K, Fraction(float(a32[m])))
        br = _dec_row(1, B[g * N + n], SB[g * N + n], K, Fraction(float(b32[g])))
        exact = sum(x * y for x, y in zip(ar, br))
        assert abs(Fraction(ref[p]) - exact) <= Fraction(1, 10 ** 12) * sum(abs(x * y) for x, y in zip(ar, br)) + Fraction(1, 10 ** 300)


def _swizzle_by_reshape(canon):
    """Independent construction of the tensor-core scale tiles: pad to
    (rows up to 128, scols up to 4), view as (row-tile, 4 row-quads, 32 rows,
    col-tile, 4 cols) and order as (row-tile, col-tile, 32 rows, 4 quads, 4 cols)."""
    rows, scols = canon.shape
    Rp = -(-rows // 128) * 128
    Sp = -(-scols // 4) * 4
    pad = np.zeros((Rp, Sp), np.uint8)
    pad[:rows, :scols] = canon
    t = pad.reshape(Rp // 128, 4, 32, Sp // 4, 4).transpose(0, 3, 2, 1, 4)
    return t.reshape(-1)


@pytest.mark.parametrize("rows,scols", [(1, 1), (128, 4), (130, 5), (300, 64), (257, 7)])
def test_swizzle_matches_reshape_construction(rows, scols):
    rng = np.random.default_rng(rows * 131 + scols)
    canon = rng.integers(1, 256, size=(rows, scols), dtype=np.uint8)
    got = oracle.swizzle_scales(canon)
    assert np.array_equal(got, _swizzle_by_reshape(canon))
    # a bijection onto the non-pad bytes; padding is zero
    assert np.count_nonzero(got) == rows * scols


def test_grouped_swizzle_pads_every_group_to_whole_tiles():
    rng = np.random.default_rng(5)
    offs = np.array([0, 130, 130, 131, 400])
    canon = rng.integers(1, 256, size=(400, 6), dtype=np.uint8)
    got = oracle.swizzle_scales(canon, offs)
    parts = [_swizzle_by_reshape(canon[offs[g]:offs[g + 1]]) for g in range(4) if offs[g + 1] > offs[g]]
    assert np.array_equal(got, np.concatenate(parts))
    assert got.size == oracle.swizzled_bytes(400, 6, offs) == (2 + 1 + 3) * 128 * 8


# ------------------------------------------------------------------ BF16 GEMM
def _bf16_fraction(bits):
    """Exact value of bf16 bit patterns, decoded through PyTorch's bfloat16."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()
    return [Fraction(v) for v in t.ravel().tolist()]


def _rand_bf16(rng, shape):
    """Finite bf16 patterns with exponents in [-40, 40] and random signs."""
    sign = rng.integers(0, 2, size=shape).astype(np.uint16) << 15
    exp = rng.integers(127 - 40, 127 + 40, size=shape).astype(np.uint16) << 7
    man = rng.integers(0, 128, size=shape).astype(np.uint16)
    return (sign | exp | man).astype(np.uint16)


def test_bf16_gemm_brute_force_exact():
    rng = np.random.default_rng(21)
    M, N, K = 3, 2, 24
    a, b = _rand_bf16(rng, (M, K)), _rand_bf16(rng, (N, K))
    ref, absref = oracle.bf16_gemm_ref(a, b)
    for m in range(M):
        ar = _bf16_fraction(a[m])
        for n in range(N):
            br = _bf16_fraction(b[n])
            exact = sum(x * y for x, y in zip(ar, br))
            aexact = sum(abs(x * y) for x, y in zip(ar, br))
            assert abs(Fraction(ref[m, n]) - exact) <= Fraction(1, 10 ** 12) * aexact
            assert abs(Fraction(absref[m, n]) - aexact) <= Fraction(1, 10 ** 12) * aexact


@pytest.mark.parametrize("fmt", [0, 2])
def test_bf16_gemm_on_dequantized_operands_equals_block_scaled(fmt):
    """The dequantized-backward identity: E4M3 / E2M1 codes times a power of
    two are exact in bf16, so the BF16 GEMM over the dequantized operands sums
    the very products the block-scaled reference sums, in the same order."""
    from moe_mx8_quantize_gb300 import inputs
    K = 160
    xa = inputs.bits(inputs.normal_bf16((5, K), 1.0, torch.Generator().manual_seed(1), "cpu"))
    xb = inputs.bits(inputs.normal_bf16((7, K), 0.02, torch.Generator().manual_seed(2), "cpu"))
    if fmt == 0:
        (qa, sa), (qb, sb) = oracle.mxfp8_quantize_rowwise(xa), oracle.mxfp8_quantize_rowwise(xb)
        da, db = oracle.dequant_mxfp8(qa, sa), oracle.dequant_mxfp8(qb, sb)
    else:
        (qa, sa), (qb, sb) = oracle.mxfp4_quantize_rowwise(xa), oracle.mxfp4_quantize_rowwise(xb)
        da, db = oracle.dequant_mxfp4(qa, sa), oracle.dequant_mxfp4(qb, sb)
    ba, bb = oracle.f32_to_bf16(da), oracle.f32_to_bf16(db)
    assert np.array_equal(oracle.bf16_to_f32(ba), da) and np.array_equal(oracle.bf16_to_f32(bb), db)
    ref, absref = oracle.bf16_gemm_ref(ba, bb)
    want, awant = oracle.gemm_ref(fmt, qa, sa, qb, sb, K)
    assert np.array_equal(ref, want) and np.array_equal(absref, awant)


def test_bf16_gemm_sampled_pairs_match_full():
    rng = np.random.default_rng(22)
    a, b = _rand_bf16(rng, (9, 40)), _rand_bf16(rng, (6, 40))
    full, afull = oracle.bf16_gemm_ref(a, b)
    pairs = np.array([(8, 5), (0, 0), (3, 2), (3, 1)])
    ref, absref = oracle.bf16_gemm_ref(a, b, pairs)
    assert np.array_equal(ref, full[pairs[:, 0], pairs[:, 1]])
    assert np.array_equal(absref, afull[pairs[:, 0], pairs[:, 1]])


# ------------------------------------------------------------------ MoE combine
def test_moe_combine_one_hot_is_a_gather():
    rng = np.random.default_rng(31)
    y = rng.integers(0, 2 ** 16, size=(40, 24), dtype=np.uint16)
    y[(y & 0x7F80) == 0x7F80] = 0x3F80            # no inf / nan patterns
    rows = rng.integers(0, 40, size=(10, 3))
    w = np.zeros((10, 3), np.float32)
    pick = rng.integers(0, 3, 10)
    w[np.arange(10), pick] = 1.0
    out = oracle.moe_combine(y, rows, w)
    assert np.array_equal(out, oracle.bf16_to_f32(y[rows[np.arange(10), pick]]))


def test_moe_combine_exact_on_small_integers_and_skips_bad_rows():
    """Small integers and weights that are multiples of 1/8: every binary32
    step is exact, so the result is the exact weighted sum; rows outside the
    matrix contribute nothing."""
    rng = np.random.default_rng(32)
    yv = rng.integers(-50, 50, size=(30, 16)).astype(np.float32)
    y = torch.tensor(yv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rows = rng.integers(0, 30, size=(12, 8))
    rows[3, 5] = -1
    rows[7, 0] = 30
    w = (rng.integers(0, 9, size=(12, 8)) / 8.0).astype(np.float32)
    out = oracle.moe_combine(y, rows, w)
    valid = (rows >= 0) & (rows < 30)
    want = np.einsum("tj,tjh->th", np.where(valid, w, 0).astype(np.float64),
                     yv[np.clip(rows, 0, 29)].astype(np.float64))
    assert np.array_equal(out.astype(np.float64), want)
