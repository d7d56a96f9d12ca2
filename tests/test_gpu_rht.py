"""GPU parity of the RHT columnwise NVFP4 quantizer for Wgrad inputs ("NVIDIA
presenta una metodologia de preentrenamiento de 4 bits utilizando NVFP4",
section "La metodologia de formacion de cuatro partes") against the CPU
oracle: codes, every byte of the scale-tile buffer and the FP32 scale, bit
for bit; then the Wgrad GEMM over two RHT-quantized operands against the
FP64 reference over the same operands, and against the untransformed product
within the quantization error (the transform cancels)."""
import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import dev, ensure_built, gemm_tolerance_ok, host

pytestmark = pytest.mark.gpu

MASK = 0xB2D5      # the shared sign vector of these tests


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(xb, mask=MASK, x=None):
    q, s, s32 = mx.nvfp4_quantize_rht_colwise(dev(xb) if x is None else x, mask)
    oq, os_, o32 = oracle.nvfp4_quantize_rht_colwise(xb, mask)
    assert host(s32).view(np.uint32)[0] == o32.view(np.uint32)[0], "fp32 scale"
    assert np.array_equal(host(q), oq), "codes"
    sw = oracle.swizzle_scales(os_)
    assert np.array_equal(host(s)[: sw.size], sw), "scales"
    return q, s, s32, oq, os_, o32


@pytest.mark.parametrize("shape,mask", [((32, 8), 0), ((96, 168), MASK), ((256, 512), 0xFFFF),
                                        ((160, 1000), MASK), ((2048, 256), 0x0F0F)])
def test_rht_colwise_shapes(shape, mask):
    xb = inputs.bits(inputs.normal_bf16(shape, 1.0, torch.Generator().manual_seed(shape[1]), "cpu", 0.005, 100))
    _check(xb, mask)


@pytest.mark.parametrize("seed", [0, 0xFEEDFACE12345678])
def test_rht_colwise_stochastic(seed):
    """Gradient inputs: codes by stochastic rounding with the Philox bits of
    each element's position, bit-exact against the oracle."""
    xb = inputs.bits(inputs.normal_bf16((256, 200), 1e-3, torch.Generator().manual_seed(8), "cpu", 0.01, 20))
    q, s, s32 = mx.nvfp4_quantize_rht_colwise(dev(xb), MASK, stochastic=True, seed=seed)
    oq, os_, o32 = oracle.nvfp4_quantize_rht_colwise(xb, MASK, stochastic=True, seed=seed)
    assert host(s32).view(np.uint32)[0] == o32.view(np.uint32)[0]
    assert np.array_equal(host(q), oq)
    sw = oracle.swizzle_scales(os_)
    assert np.array_equal(host(s)[: sw.size], sw)


@pytest.mark.parametrize("shape", [(5, 16), (130, 96), (3, 1008), (70, 1536), (33, 4096), (2048, 8192),
                                   (40, 12288), (9, 20480)])
def test_per_token_stochastic(shape):
    """Per-token NVFP4 of a gradient with stochastic codes, bit-exact against
    the oracle (codes, scale tiles with padding, S_dec); the widths take every
    team size of the kernel (32 .. 256 threads a row), 1, 2 and 4 blocks a
    thread, and the two-read path of rows over 16384 values."""
    xb = inputs.bits(inputs.normal_bf16(shape, 1e-3, torch.Generator().manual_seed(shape[0]), "cpu", 0.01, 30))
    q, s, s32 = mx.nvfp4_quantize_per_token_sr(dev(xb), 1234567 + shape[0])
    oq, os_, o32 = oracle.nvfp4_quantize_sr(xb, 1234567 + shape[0])
    assert np.array_equal(host(s32).view(np.uint32), o32.view(np.uint32))
    assert np.array_equal(host(q), oq)
    sw = oracle.swizzle_scales(os_)
    assert np.array_equal(host(s)[: sw.size], sw)


def test_rht_colwise_sweep_values():
    _check(inputs.bits(inputs.sweep(128, 256, seed=13).float().clamp(-3e4, 3e4).to(torch.bfloat16)))


def test_rht_colwise_linear_full_size():
    """X [2048, 2048] and dY [2048, 8192] of the linear layer (tokens first)."""
    d = inputs.linear(device="cuda")
    for name in ("X", "dY"):
        _check(inputs.bits(d[name]), x=d[name])


def test_wgrad_over_rht_operands():
    """dW = dY^T X over the RHT-quantized columnwise copies of dY and X (same
    signs): within the GEMM tolerance of the FP64 reference over the same
    operands; and close to the product of the untransformed bf16 inputs,
    since the transform cancels in the dot products."""
    T, O, H = 256, 192, 160
    g = torch.Generator().manual_seed(4)
    dYb = inputs.bits(inputs.normal_bf16((T, O), 1.0, g, "cpu"))
    Xb = inputs.bits(inputs.normal_bf16((T, H), 1.0, g, "cpu"))
    qa, sa, a32, oqa, osa, oa32 = _check(dYb)
    qb, sb, b32, oqb, osb, ob32 = _check(Xb)
    y = host(mx.bs_gemm(mx.FMT_NVFP4, qa, sa, qb, sb, T, a32, b32))
    ref, absref = oracle.gemm_ref(1, oqa, osa, oqb, osb, T, oa32, ob32)
    ok, bad = gemm_tolerance_ok(y, ref, absref, False, T)
    assert ok, f"{bad.size} outputs out of tolerance"
    exact = oracle.bf16_to_f32(dYb).astype(np.float64).T @ oracle.bf16_to_f32(Xb).astype(np.float64)
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.3, rel          # NVFP4 error; a transform that did not cancel gives ~1.4
