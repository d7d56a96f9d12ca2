"""Pins of the oracle's MXFP4 path (32-element blocks of E2M1 under one UE8M0
scale; "NVIDIA presenta una metodologia de preentrenamiento de 4 bits
utilizando NVFP4", section "Que es realmente NVFP4") against a hand-worked
block, the exponent rule checked by search, format invariants and an exact
GEMM on values the format represents exactly."""
import numpy as np
import torch

import oracle
from moe_mx8_quantize_gb300 import inputs

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(vals, dtype=torch.float32)), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def nibbles(qrow):
    out = []
    for b in qrow.tolist():
        out += [b & 15, b >> 4]
    return out


def test_worked_block():
    """amax = 24 = 6 * 2^2, so e = 2 (scale code 129) and every element is
    divided by 4 exactly; E2M1 codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6:
        24  -> 6       code 7
         5  -> 1.25    tie between 1 (code 2) and 1.5 (code 3): even code 2
       -10  -> -2.5    tie between 2 (4) and 3 (5): even 4, sign bit -> 0xC
         1  -> 0.25    tie between 0 and 0.5: code 0
        -1  -> -0.25   negative tie to zero keeps the sign: 0x8
        14  -> 3.5     tie between 3 (5) and 4 (6): even code 6
        20  -> 5       tie between 4 (6) and 6 (7): even code 6
        22  -> 5.5     nearer to 6: code 7
    and 24 zeros -> code 0.  Element 2j sits in the low nibble of byte j."""
    vals = [24.0, 5.0, -10.0, 1.0, -1.0, 14.0, 20.0, 22.0] + [0.0] * 24
    x = bf16_bits(vals).reshape(1, 32)
    q, s = oracle.mxfp4_quantize_rowwise(x)
    assert s.tolist() == [[129]]
    assert nibbles(q[0])[:8] == [7, 2, 0xC, 0, 0x8, 6, 6, 7]
    assert nibbles(q[0])[8:] == [0] * 24
    assert q[0, 0] == (2 << 4) | 7


def test_exponent_rule_by_search():
    """e is the smallest integer with amax <= 6 * 2^e (clamped to [-127, 127]);
    checked against the two inequalities that define it."""
    rng = np.random.default_rng(3)
    amaxes = [0.0, 6.0, 6.0000005, 5.99, 3.0, 3.0000002, 2.0 ** -140, 1e30, 3.3e38]
    amaxes += list(np.float32(rng.lognormal(0, 20, 200)))
    for a in amaxes:
        a = float(np.float32(a))
        e = oracle.mxfp4_block_exp(a)
        assert -127 <= e <= 127
        if a == 0.0:
            assert e == -127
            continue
        if e < 127:
            assert a <= 6.0 * 2.0 ** e
        if e > -127:
            assert a > 6.0 * 2.0 ** (e - 1)


def test_no_saturation_and_half_spacing_round_trip():
    """With amax <= 6 * 2^e no element saturates, so each decoded value is within
    half an E2M1 spacing (times 2^e) of the input: 0.25 below 2, 0.5 below 4,
    1 up to 6."""
    x = inputs.bits(inputs.sweep(96, 256, seed=11))
    q, s = oracle.mxfp4_quantize_rowwise(x)
    # decoded in float64 from the E2M1 table (a code times 2^e can exceed the
    # binary32 range, e.g. 4 * 2^126 for the bf16 maximum)
    codes = np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], -1)
    mag = np.array(E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    xv = oracle.bf16_to_f32(x).astype(np.float64)
    e = s.astype(np.int64) - 127
    scale = np.repeat(np.ldexp(1.0, e), 32, axis=1)
    d = mag * scale
    m = np.abs(xv) / scale
    assert (m <= 6.0).all()
    half = np.where(m < 2, 0.25, np.where(m < 4, 0.5, 1.0)) * scale
    assert (np.abs(d - xv) <= half).all()


def test_colwise_is_rowwise_of_transpose():
    x = inputs.bits(inputs.sweep(64, 96, seed=12))
    qc, sc = oracle.mxfp4_quantize_colwise(x)
    qr, sr = oracle.mxfp4_quantize_rowwise(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qr) and np.array_equal(sc, sr)


def test_gemm_exact_on_representable_values():
    """Every 32-block holds one element 6 * 2^k and otherwise E2M1 grid values
    times 2^k, so quantization is exact (e = k) and the FP64 reference must
    equal numpy's product of the original values, which is exact here."""
    rng = np.random.default_rng(5)
    M, N, K = 8, 12, 128

    def make(rows):
        v = rng.choice(E2M1, size=(rows, K)) * rng.choice([-1.0, 1.0], size=(rows, K))
        v[:, ::32] = 6.0
        k = rng.integers(-6, 6, size=(rows, K // 32))
        return v * np.repeat(np.ldexp(1.0, k), 32, axis=1)

    a, b = make(M), make(N)
    qa, sa = oracle.mxfp4_quantize_rowwise(bf16_bits(a.ravel().tolist()).reshape(M, K))
    qb, sb = oracle.mxfp4_quantize_rowwise(bf16_bits(b.ravel().tolist()).reshape(N, K))
    assert np.array_equal(oracle.dequant_mxfp4(qa, sa).astype(np.float64), a)
    ref, absref = oracle.gemm_ref(2, qa, sa, qb, sb, K)
    assert np.array_equal(ref, a @ b.T)
    assert np.array_equal(absref, np.abs(a) @ np.abs(b).T)
