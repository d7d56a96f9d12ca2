"""Pins of the oracle's NVFP4 weights with 2-D 16x16 block scaling ("NVIDIA
presenta una metodologia de preentrenamiento de 4 bits utilizando NVFP4",
section "La metodologia de formacion de cuatro partes": one quantized
representation for the forward and the transposed backward weight): a
hand-worked two-block tensor, the columnwise copy equal to the transpose of
the rowwise one, the reduction to tensor-scope 1x16 NVFP4 when every 16-row
block repeats one row, and the 256-element block maximum."""
import numpy as np
import torch

import oracle
from moe_mx8_quantize_gb300 import inputs

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(vals, np.float32))), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def nib(q, r, k):
    b = int(q[r, k // 2])
    return (b >> 4) if k & 1 else (b & 15)


def test_worked_two_block_tensor():
    """Block 0 (columns 0..15) holds amax 6, block 1 (columns 16..31) amax 3.
    Tensor amax 6: S_enc = 2688 / 6 = 448, S_dec = 6 / 2688.
    Block 0: RN(6/6) * 448 = 448 -> sb = E4M3 448 (0x7E), r = 448/448 = 1,
      so codes are RNE_E2M1(x): 6 -> 7, 1.25 -> 2 (tie to even), -2.5 -> 0xC.
    Block 1: RN(3/6) * 448 = 224 -> sb = E4M3 224 (0x76), r = 448/224 = 2,
      so 3 -> 6 (code 7), 0.75 -> 1.5 (code 3), -0.625 -> -1.25 -> tie -> 0xA."""
    x = np.zeros((16, 32), np.float32)
    x[0, 0], x[5, 3], x[9, 7] = 6.0, 1.25, -2.5
    x[2, 16], x[15, 20], x[7, 31] = 3.0, 0.75, -0.625
    q, s, qc, sc, s32 = oracle.nvfp4_quantize_2d(bf16_bits(x))
    assert s32[0] == np.float32(6.0) / np.float32(2688.0)
    assert (s[:, 0] == 0x7E).all() and (s[:, 1] == 0x76).all()
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x76) == 224.0
    assert nib(q, 0, 0) == 7 and nib(q, 5, 3) == 2 and nib(q, 9, 7) == 0xC
    assert nib(q, 2, 16) == 7 and nib(q, 15, 20) == 3 and nib(q, 7, 31) == 0xA
    assert sum(nib(q, r, k) != 0 for r in range(16) for k in range(32)) == 6


def _unpack(q):
    return np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], -1)


def test_columnwise_copy_is_the_transpose():
    x = inputs.bits(inputs.normal_bf16((96, 160), 0.02, torch.Generator().manual_seed(3), "cpu", 0.01, 30))
    q, s, qc, sc, _ = oracle.nvfp4_quantize_2d(x)
    assert np.array_equal(_unpack(qc), _unpack(q).T)
    assert np.array_equal(np.repeat(sc, 16, axis=1), np.repeat(s, 16, axis=1).T)
    # every row of a 16-row block carries that block's scale
    assert (s.reshape(6, 16, 10) == s.reshape(6, 16, 10)[:, :1, :]).all()


def test_repeated_rows_reduce_to_tensor_scope_1x16():
    """When the 16 rows of every block row are equal, each 16x16 block amax is
    the 1x16 amax of each of its rows, so the rowwise copy equals tensor-scope
    1x16 NVFP4 of the same matrix (codes, scales and the FP32 scale)."""
    base = inputs.bits(inputs.normal_bf16((4, 128), 1.0, torch.Generator().manual_seed(5), "cpu", 0.02, 40))
    x = np.repeat(base, 16, axis=0)
    q, s, _, _, s32 = oracle.nvfp4_quantize_2d(x)
    q1, s1, t1 = oracle.nvfp4_quantize(x, oracle.SCOPE_TENSOR)
    assert np.array_equal(q, q1) and np.array_equal(s, s1)
    assert s32.view(np.uint32)[0] == t1.view(np.uint32)[0]


def test_block_max_spans_all_256_elements():
    """One large value in row 9 of a block raises that block's scale for all
    16 rows; the 1x16 quantization would only change row 9's."""
    x = np.full((32, 32), 0.5, np.float32)
    x[9, 4] = 6.0
    q, s, _, _, _ = oracle.nvfp4_quantize_2d(bf16_bits(x))
    _, s1, _ = oracle.nvfp4_quantize(bf16_bits(x), oracle.SCOPE_TENSOR)
    assert len(set(s[:16, 0].tolist())) == 1 and s[0, 0] == s1[9, 0]
    assert s1[0, 0] != s1[9, 0]
    assert (s[16:, 0] == s1[16:, 0]).all() and (s[:, 1] == s1[:, 1]).all()
