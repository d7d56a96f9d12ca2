"""Pins of the oracle's stochastic rounding for gradients ("NVIDIA presenta una
metodologia de preentrenamiento de 4 bits utilizando NVFP4", section "La
metodologia de formacion de cuatro partes": round up or down with
probabilities given by the distances to the two nearest representable
values).  The counter-based generator (Philox4x32-10) is checked against
the known-answer vectors published with it; the rounding against its
thresholds and its expectation."""
import numpy as np
import pytest

import oracle

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# Known-answer vectors of Philox4x32-10 distributed with the generator
# (Random123 "kat_vectors": counter words, key words -> output words).
PHILOX4X32_KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX4X32_KAT)
def test_philox_known_answers(ctr, key, want):
    assert [int(w) for w in oracle.philox4x32_10(ctr, key)] == list(want)


def test_sr_bits_word_layout():
    """Element e takes word e % 4 of the block with counter (e / 4 split in
    two 32-bit words, 0, 0) and key (seed split in two 32-bit words)."""
    for seed, e in ((0, 0), (5, 7), (0x243F6A8885A308D3, 2 ** 35 + 6), (2 ** 64 - 1, 2 ** 64 - 1)):
        blk = oracle.philox4x32_10([(e >> 2) & 0xFFFFFFFF, e >> 34, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.sr_bits(seed, e) == int(blk[e % 4])
    # the first KAT vector is element 0..3 of seed 0
    assert [oracle.sr_bits(0, e) for e in range(4)] == list(PHILOX4X32_KAT[0][2])


def test_sr_bits_are_uniform():
    u = np.array([oracle.sr_bits(99, e) >> 8 for e in range(40000)], np.float64) / 2 ** 24
    assert abs(u.mean() - 0.5) < 0.01 and abs((u < 0.25).mean() - 0.25) < 0.01
    assert len({oracle.sr_bits(99, e) for e in range(64)}) == 64


def test_sr_thresholds():
    up = lambda p: (int(p * 2 ** 24) - 1) << 8          # largest 24-bit draw that still rounds up
    down = lambda p: int(p * 2 ** 24) << 8
    assert oracle.e2m1_sr(0.75, up(0.5)) == 2 and oracle.e2m1_sr(0.75, down(0.5)) == 1
    assert oracle.e2m1_sr(5.0, up(0.5)) == 7 and oracle.e2m1_sr(5.0, down(0.5)) == 6
    assert oracle.e2m1_sr(2.25, up(0.25)) == 5 and oracle.e2m1_sr(2.25, down(0.25)) == 4
    assert oracle.e2m1_sr(-0.25, up(0.5)) == 0x9 and oracle.e2m1_sr(-0.25, down(0.5)) == 0x8
    for v in E2M1:                                       # grid values never move
        for bits in (0, 0x12345678, 0xFFFFFFFF):
            assert oracle.e2m1_sr(v, bits) == E2M1.index(v)
    assert oracle.e2m1_sr(7.5, 0) == 7 and oracle.e2m1_sr(-100.0, 0) == 0xF
    assert oracle.e2m1_sr(-0.0, 0) == 0x8


@pytest.mark.parametrize("v", [0.1, 0.3, 1.2, 2.7, 3.9, 4.4, 5.999])
def test_sr_expectation_is_the_value(v):
    """Over the draws, the rounded value averages to v (unbiased to 2^-12 on a
    2^12-point grid of draws)."""
    vals = [E2M1[oracle.e2m1_sr(v, (u << 20))] for u in range(4096)]
    assert abs(np.mean(vals) - np.float32(v)) < 2.0 ** -10


def test_sr_quantizer_keeps_scales_and_brackets_codes():
    """Same FP32 and block scales as round-to-nearest NVFP4; every code is one
    of the two grid neighbours of the scaled value; and on a tensor where a
    value sits at 0.6 of a grid interval, the rounded values average to it
    (round to nearest would give the upper neighbour every time)."""
    rng = np.random.default_rng(0)
    import torch
    x = torch.tensor(rng.standard_normal((64, 256)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q, s, s32 = oracle.nvfp4_quantize_sr(xb, 7)
    q0, s0, t0 = oracle.nvfp4_quantize(xb)
    assert np.array_equal(s, s0) and np.array_equal(s32.view(np.uint32), t0.view(np.uint32))
    mag = lambda qq: np.array(E2M1)[np.stack([qq & 7, (qq >> 4) & 7], -1).reshape(qq.shape[0], -1)]
    assert (np.abs(mag(q) - mag(q0)) <= 2.0).all()      # at most one grid step apart
    # 1.0 and 0.3 alternating: block amax 1 -> S scaled 0.3 lands on 1.8 = 1.5 + 0.6 * 0.5
    row = np.tile(np.array([1.0, 0.3], np.float32), 128)
    xr = torch.tensor(np.tile(row, (64, 1))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qs, ss, _ = oracle.nvfp4_quantize_sr(xr, 11)
    qr, _, _ = oracle.nvfp4_quantize(xr)
    odd_sr = mag(qs)[:, 1::2]
    assert set(np.unique(odd_sr)) <= {1.5, 2.0}
    assert (mag(qr)[:, 1::2] == 2.0).all()
    scaled = float(np.float32(np.float32(0.30078125) * np.float32(6.0 / 1.0)))   # bf16(0.3) * r
    assert abs(odd_sr.mean() - 1.8) < 0.03 and abs(odd_sr.mean() - scaled) < 0.03
