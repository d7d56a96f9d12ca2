"""GPU parity of NVFP4 weights with 2-D 16x16 block scaling ("NVIDIA presenta
una metodologia de preentrenamiento de 4 bits utilizando NVFP4", section "La
metodologia de formacion de cuatro partes") against the CPU oracle: both
copies' codes, every byte of both scale-tile buffers (padding included) and
the FP32 tensor scale, bit for bit; then the forward and the transposed
backward GEMMs on those weights within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import dev, ensure_built, gemm_tolerance_ok, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check_2d(xb, flags=mx.ROWWISE | mx.COLWISE, x=None):
    if x is None:
        x = dev(xb)
    q_row, s_row, q_col, s_col, s32 = mx.nvfp4_quantize_2d(x, flags)
    torch.cuda.synchronize()
    oq, os_, oqc, osc, o32 = oracle.nvfp4_quantize_2d(xb)
    assert host(s32).view(np.uint32)[0] == o32.view(np.uint32)[0], "fp32 scale"
    if flags & mx.ROWWISE:
        assert np.array_equal(host(q_row), oq), "rowwise codes"
        sw = oracle.swizzle_scales(os_)
        assert np.array_equal(host(s_row)[: sw.size], sw), "rowwise scales"
    if flags & mx.COLWISE:
        assert np.array_equal(host(q_col), oqc), "columnwise codes"
        sw = oracle.swizzle_scales(osc)
        assert np.array_equal(host(s_col)[: sw.size], sw), "columnwise scales"
    return q_row, s_row, q_col, s_col, s32


@pytest.mark.parametrize("shape,flags", [
    ((32, 32), mx.ROWWISE | mx.COLWISE),
    ((96, 160), mx.ROWWISE | mx.COLWISE),      # ragged 128-tiles both ways
    ((160, 96), mx.ROWWISE),
    ((224, 544), mx.COLWISE),
    ((256, 2048), mx.ROWWISE | mx.COLWISE),
])
def test_nvfp4_2d_shapes(shape, flags):
    xb = inputs.bits(inputs.normal_bf16(shape, 0.02, torch.Generator().manual_seed(shape[0] + shape[1]), "cpu",
                                        0.01, 40))
    _check_2d(xb, flags)


def test_nvfp4_2d_sweep_values():
    """Zeros, bf16 extremes, subnormals and tie blocks of the sweep mixture."""
    _check_2d(inputs.bits(inputs.sweep(128, 256, seed=9)))


def test_nvfp4_2d_linear_weight_full_size():
    d = inputs.linear(device="cuda")
    _check_2d(inputs.bits(d["W"]), x=d["W"])


def _check(y, ref, absref, K):
    ok, bad = gemm_tolerance_ok(y, ref, absref, False, K)
    assert ok, f"{bad.size} outputs out of tolerance"


def test_forward_and_backward_gemms_use_one_weight():
    """Fprop Y = X W^T with the rowwise copy and Dgrad dX = dY W with the
    columnwise copy (per-token NVFP4 activations / gradients): both against
    the FP64 reference over the same 2-D quantized weight."""
    T, O, H = 128, 256, 512
    g = torch.Generator().manual_seed(2)
    Wb = inputs.bits(inputs.normal_bf16((O, H), 0.02, g, "cpu"))
    Xb = inputs.bits(inputs.normal_bf16((T, H), 1.0, g, "cpu"))
    dYb = inputs.bits(inputs.normal_bf16((T, O), 1e-3, g, "cpu"))
    q_row, s_row, q_col, s_col, s32 = _check_2d(Wb)
    oq, os_, oqc, osc, o32 = oracle.nvfp4_quantize_2d(Wb)
    xq, xs, x32 = oracle.nvfp4_quantize(Xb)
    y = host(mx.bs_gemm(mx.FMT_NVFP4, dev(xq), dev(oracle.swizzle_scales(xs)), q_row, s_row, H, dev(x32), s32))
    ref, absref = oracle.gemm_ref(1, xq, xs, oq, os_, H, x32, o32)
    _check(y, ref, absref, H)
    gq, gs, g32 = oracle.nvfp4_quantize(dYb)
    dx = host(mx.bs_gemm(mx.FMT_NVFP4, dev(gq), dev(oracle.swizzle_scales(gs)), q_col, s_col, O, dev(g32), s32))
    ref, absref = oracle.gemm_ref(1, gq, gs, oqc, osc, O, g32, o32)
    _check(dx, ref, absref, O)
