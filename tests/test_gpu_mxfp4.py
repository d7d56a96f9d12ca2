"""GPU parity of the MXFP4 path (32-element blocks of E2M1 under one E8M0
scale; "NVIDIA presenta una metodologia de preentrenamiento de 4 bits
utilizando NVFP4", section "Que es realmente NVFP4") against the CPU oracle:
the quantizer bit-exact (codes and every byte of the tensor-core scale tiles),
the dequantizer bit-exact, and the block-scaled GEMM (kind::mxf4nvf4 with two
UE8M0 scales per MMA) within 1e-5 * sum_k |a^||b^| of the FP64 reference.
GEMM operands are quantized by the oracle, so no expected value comes from the
GPU path."""
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


# ------------------------------------------------------------------ quantizer
def _q_check(xb, flags=mx.ROWWISE | mx.COLWISE, x=None):
    if x is None:
        x = dev(xb)
    q_row, s_row, q_col, s_col = mx.mxfp4_quantize(x, flags)
    torch.cuda.synchronize()
    if flags & mx.ROWWISE:
        q, s = oracle.mxfp4_quantize_rowwise(xb)
        assert np.array_equal(host(q_row), q), "rowwise codes"
        sw = oracle.swizzle_scales(s)
        assert np.array_equal(host(s_row)[: sw.size], sw), "rowwise scales"
    if flags & mx.COLWISE:
        qT, sT = oracle.mxfp4_quantize_colwise(xb)
        assert np.array_equal(host(q_col), qT), "colwise codes"
        sw = oracle.swizzle_scales(sT)
        assert np.array_equal(host(s_col)[: sw.size], sw), "colwise scales"


def test_mxfp4_pr1():
    d = inputs.pr1()
    _q_check(inputs.bits(d["X"]))
    _q_check(inputs.bits(d["W"]))


@pytest.mark.parametrize("shape,flags", [
    ((96, 160), mx.ROWWISE | mx.COLWISE),     # ragged rows and columns of the 128x128 tile
    ((32, 32), mx.ROWWISE | mx.COLWISE),
    ((1, 32), mx.ROWWISE),
    ((200, 96), mx.ROWWISE),
    ((33, 4096), mx.ROWWISE),
    ((256, 544), mx.COLWISE),
    ((640, 384), mx.ROWWISE | mx.COLWISE),
])
def test_mxfp4_ragged_and_sweep_mix(shape, flags):
    _q_check(inputs.bits(inputs.sweep(*shape, seed=21 + shape[0])), flags)


def test_mxfp4_edge_values():
    """bf16 extremes, subnormals, signed zero, the E2M1 rounding ties and the
    exponent rule's boundary (amax exactly 6 * 2^k and just above it)."""
    xb = np.zeros((64, 64), np.uint16)
    xb[0, 0] = 0x7F7F           # +bf16 max
    xb[1, 5] = 0xFF7F           # -bf16 max
    xb[2, :] = 0x0001           # smallest subnormal
    xb[3, 7] = 0x8000           # -0
    xb[4, 3] = 0x8001           # negative subnormal
    xb[5, :32] = 0x3F80         # all equal blocks (1.0)
    xb[6, 32:] = 0xC0C0         # -6
    xb[7, :32] = 0x40C1         # just above 6: exponent steps up
    ties = [0x3E80, 0x3F40, 0x3FA0, 0x3FE0, 0x4020, 0x4060, 0x40A0]   # 0.25 .. 5: E2M1 midpoints
    for j, t in enumerate(ties):
        xb[8, j] = t
        xb[8, 8 + j] = t | 0x8000
    xb[8, 31] = 0x40C0          # block amax 6 -> scale 2^0, ties decided at scale 1
    _q_check(xb)


def test_mxfp4_linear_full_size():
    d = inputs.linear(device="cuda")
    for name in ("X", "W", "dY"):
        _q_check(inputs.bits(d[name]), x=d[name])


def test_mxfp4_strided_input():
    xb = inputs.bits(inputs.sweep(128, 256, seed=4))
    big = torch.zeros((128, 320), dtype=torch.bfloat16, device="cuda")
    big[:, :256] = dev(xb)
    _q_check(xb, x=big[:, :256])


def test_mxfp4_empty():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    mx.mxfp4_quantize(x, mx.ROWWISE)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ dequantize
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_dequant_mxfp4(out_dtype):
    xb = inputs.bits(inputs.sweep(160, 320, seed=41))
    q, s = oracle.mxfp4_quantize_rowwise(xb)
    ref = oracle.dequant_mxfp4(q, s)
    out = mx.dequantize(mx.FMT_MXFP4, dev(q), dev(oracle.swizzle_scales(s)), out_dtype=out_dtype)
    got = host(out)
    if out_dtype == torch.float32:
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(got, oracle.f32_to_bf16(ref))


# ------------------------------------------------------------------ GEMM
def _check(y, ref, absref, bf16=False, K=None):
    ok, bad = gemm_tolerance_ok(y, ref, absref, bf16, K)
    if not ok:
        yf = np.asarray(y, np.float64).ravel()
        i = bad[:5]
        raise AssertionError(f"{bad.size} outputs out of tolerance; e.g. idx {i}: "
                             f"got {yf[i]}, ref {ref.ravel()[i]}, abs {absref.ravel()[i]}")


def _run(A, SA, B, SB, K, out_dtype=torch.float32, a32=None, b32=None):
    return mx.bs_gemm(mx.FMT_MXFP4, dev(A), dev(oracle.swizzle_scales(SA)), dev(B),
                      dev(oracle.swizzle_scales(SB)), K,
                      None if a32 is None else dev(a32), None if b32 is None else dev(b32),
                      out_dtype=out_dtype)


def _operand(rows, K, seed):
    xb = inputs.bits(inputs.sweep(rows, K, seed=seed).float().clamp(-1e4, 1e4).to(torch.bfloat16))
    return oracle.mxfp4_quantize_rowwise(xb)


@pytest.mark.parametrize("k", [5, 40, 70, 100, 233, 300, 511])
def test_mxfp4_one_nonzero(k):
    """Pins operand order, nibble order, the K position and which of the two
    scales an MMA takes (scale id 0 or 2, first or second of the pair): one
    nonzero element at k in row 37 of A and row 90 of B."""
    M, N, K = 128, 128, 512
    A = np.zeros((M, K // 2), np.uint8); B = np.zeros((N, K // 2), np.uint8)
    SA = np.full((M, K // 32), 127, np.uint8); SB = np.full((N, K // 32), 127, np.uint8)
    sh = 4 * (k & 1)
    A[37, k // 2] = 0x7 << sh      # +6
    B[90, k // 2] = 0xB << sh      # -1.5
    SA[37, k // 32] = 130; SB[90, k // 32] = 125
    y = host(_run(A, SA, B, SB, K))
    ref, absref = oracle.gemm_ref(2, A, SA, B, SB, K)
    assert np.count_nonzero(ref) == 1 and ref[37, 90] == -18.0
    _check(y, ref, absref, K=K)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (200, 72, 96), (1, 8, 32), (257, 384, 1056),
                                   (128, 128, 64), (130, 520, 2080)])
def test_mxfp4_gemm_shapes(M, N, K):
    A, SA = _operand(M, K, M + 1)
    B, SB = _operand(N, K, N + 2)
    y = host(_run(A, SA, B, SB, K))
    ref, absref = oracle.gemm_ref(2, A, SA, B, SB, K)
    _check(y, ref, absref, K=K)
    yb = host(_run(A, SA, B, SB, K, torch.bfloat16))
    _check(oracle.bf16_to_f32(yb), ref, absref, bf16=True, K=K)


def test_mxfp4_gemm_fp32_row_scales():
    """FP32 decode scales applied in the epilogue (per row of A, per tensor of B)."""
    M, N, K = 256, 256, 256
    A, SA = _operand(M, K, 3)
    B, SB = _operand(N, K, 4)
    a32 = np.random.default_rng(5).uniform(0.5, 2.0, M).astype(np.float32)
    b32 = np.array([0.75], np.float32)
    y = host(_run(A, SA, B, SB, K, a32=a32, b32=b32))
    ref, absref = oracle.gemm_ref(2, A, SA, B, SB, K, a32, b32)
    _check(y, ref, absref, K=K)


def _sample_pairs(M, N, n, seed):
    rng = np.random.default_rng(seed)
    pairs = np.stack([rng.integers(0, M, n), rng.integers(0, N, n)], 1)
    corners = np.array([[0, 0], [M - 1, N - 1], [0, N - 1], [M - 1, 0]])
    return np.concatenate([corners, pairs])


def test_mxfp4_linear_fprop_dgrad_wgrad_full_size():
    """The 2048x2048 -> 8192 linear layer in MXFP4: Fprop from the rowwise
    copies, Dgrad from dY rowwise and W columnwise, Wgrad from the columnwise
    copies of dY and X, with operands quantized on the GPU (bit-exact against
    the oracle's, checked here); sampled outputs against the FP64 oracle."""
    d = inputs.linear(device="cuda")
    Xb, Wb, dYb = (inputs.bits(d[k]) for k in ("X", "W", "dY"))
    gx, gw, gdy = (mx.mxfp4_quantize(d[k]) for k in ("X", "W", "dY"))
    Xr, SXr = oracle.mxfp4_quantize_rowwise(Xb)
    Wr, SWr = oracle.mxfp4_quantize_rowwise(Wb)
    dYr, SdYr = oracle.mxfp4_quantize_rowwise(dYb)
    Wc, SWc = oracle.mxfp4_quantize_colwise(Wb)
    Xc, SXc = oracle.mxfp4_quantize_colwise(Xb)
    dYc, SdYc = oracle.mxfp4_quantize_colwise(dYb)
    for (qr, _, qc, _), (r, c) in ((gx, (Xr, Xc)), (gw, (Wr, Wc)), (gdy, (dYr, dYc))):
        assert np.array_equal(host(qr), r) and np.array_equal(host(qc), c)
    cases = {
        "fprop": ((gx[0], gx[1], gw[0], gw[1]), (Xr, SXr, Wr, SWr), 2048),
        "dgrad": ((gdy[0], gdy[1], gw[2], gw[3]), (dYr, SdYr, Wc, SWc), 8192),
        "wgrad": ((gdy[2], gdy[3], gx[2], gx[3]), (dYc, SdYc, Xc, SXc), 2048),
    }
    for name, (gpu_ops, ora_ops, K) in cases.items():
        y = mx.bs_gemm(mx.FMT_MXFP4, *gpu_ops, K, out_dtype=torch.bfloat16)
        A, SA, B, SB = ora_ops
        pairs = _sample_pairs(A.shape[0], B.shape[0], 2000, 17)
        ref, absref = oracle.gemm_ref(2, A, SA, B, SB, K, pairs=pairs)
        yh = host(y)
        _check(oracle.bf16_to_f32(yh[pairs[:, 0], pairs[:, 1]]), ref, absref, bf16=True, K=K)


@pytest.mark.parametrize("T,H,E,N,topk,zipf", [(64, 256, 5, 256, 2, False), (300, 512, 16, 384, 4, True),
                                               (40, 96, 7, 136, 1, False)])
def test_mxfp4_grouped(T, H, E, N, topk, zipf):
    """MoE grouped GEMM: routed tokens (grouped scale layout, groups padded to
    128-row tiles) times per-expert MXFP4 weights."""
    d = inputs.moe(T, "cpu", T, H, E, N // 2, topk, routing="zipf" if zipf else "uniform",
                   with_weights=True)
    disp = inputs.dispatch(d["topk_ids"], E)
    offs = disp.offsets.numpy()
    A, SA = oracle.mxfp4_quantize_rowwise(inputs.bits(d["X"][disp.token_of_row]))
    B, SB = oracle.mxfp4_quantize_rowwise(inputs.bits(d["W_gu"]).reshape(E * N, H))
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    y = host(mx.bs_grouped_gemm(mx.FMT_MXFP4, go, dev(A), dev(oracle.swizzle_scales(SA, offs)),
                                dev(B.reshape(E, N, H // 2)), dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N)),
                                H, out_dtype=torch.float32))
    rows = A.shape[0]
    pairs = np.array([(m, n) for m in range(rows) for n in range(N)])
    ref, absref = oracle.grouped_gemm_ref(2, offs, A, SA, B.reshape(E, N, H // 2), SB, H, pairs=pairs)
    _check(y.ravel(), ref, absref, K=H)
