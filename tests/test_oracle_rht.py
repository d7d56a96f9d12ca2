"""Pins of the oracle's 16x16 random Hadamard transform and of the RHT
columnwise NVFP4 quantizer ("NVIDIA presenta una metodologia de
preentrenamiento de 4 bits utilizando NVFP4", section "La metodologia de
formacion de cuatro partes": Wgrad inputs multiplied in 16-element tiles by a
16x16 Hadamard matrix with a shared random sign vector; orthogonal, so it
cancels in the Wgrad product).  The Hadamard matrix of the pins is SciPy's
Sylvester construction, not the oracle's butterfly."""
import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle

H16 = hadamard(16).astype(np.float64)


def _signs(mask):
    return np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])


@pytest.mark.parametrize("mask", [0, 0xFFFF, 0xA5C3, 0x0001, 0x8000])
def test_transform_is_the_matrix_definition(mask):
    """Small integers keep every binary32 butterfly exact, so the oracle's
    result equals H16 diag(s) x / 4 exactly."""
    rng = np.random.default_rng(mask)
    for _ in range(20):
        x = rng.integers(-64, 64, 16).astype(np.float64)
        want = H16 @ (_signs(mask) * x) / 4
        assert np.array_equal(oracle.rht16(x, mask).astype(np.float64), want)


def test_transform_is_orthogonal_and_inverts():
    rng = np.random.default_rng(1)
    mask = 0x3C96
    x = rng.integers(-100, 100, 16).astype(np.float64)
    y = oracle.rht16(x, mask).astype(np.float64)
    assert np.array_equal(_signs(mask) * (H16 @ y) / 4, x)          # the inverse is diag(s) H16 / 4
    assert np.sum(y * y) == np.sum(x * x)                            # norms kept


def test_wgrad_product_is_unchanged():
    """sum_t RHT(dy)_t RHT(x)_t = sum_t dy_t x_t over 16-token tiles, exactly
    for small integers: the transform cancels in the dot product."""
    rng = np.random.default_rng(2)
    T, O, Hd = 64, 5, 7
    dy = rng.integers(-20, 20, (T, O)).astype(np.float64)
    x = rng.integers(-20, 20, (T, Hd)).astype(np.float64)
    mask = 0x1234

    def cols(m):
        out = np.empty(m.shape[::-1])
        for c in range(m.shape[1]):
            for k in range(T // 16):
                out[c, 16 * k:16 * k + 16] = oracle.rht16(m[16 * k:16 * k + 16, c], mask)
        return out
    assert np.array_equal(cols(dy) @ cols(x).T, dy.T @ x)


def _bf16(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(vals, np.float32)))
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("mask", [0, 0x5A5A])
def test_quantizer_is_transform_then_tensor_scope_nvfp4(mask):
    """With small-integer inputs the transformed values are exact in bf16, so
    the RHT quantizer must equal tensor-scope 1x16 NVFP4 of the transposed,
    transformed matrix (built here with SciPy's Hadamard matrix)."""
    rng = np.random.default_rng(3 + mask)
    R, C = 64, 48
    x = rng.integers(-4, 5, (R, C)).astype(np.float32)       # |y| <= 16 in steps of 1/4: exact in bf16
    y = np.empty((C, R))
    for c in range(C):
        for k in range(R // 16):
            y[c, 16 * k:16 * k + 16] = H16 @ (_signs(mask) * x[16 * k:16 * k + 16, c]) / 4
    qT, sT, s32 = oracle.nvfp4_quantize_rht_colwise(_bf16(x), mask)
    q1, s1, t1 = oracle.nvfp4_quantize(_bf16(y), oracle.SCOPE_TENSOR)
    assert np.array_equal(qT, q1) and np.array_equal(sT, s1)
    assert s32.view(np.uint32)[0] == t1.view(np.uint32)[0]
