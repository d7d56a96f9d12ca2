"""GPU parity of the block-scaled tcgen05 GEMMs against the oracle's FP64
reference over the same quantized operands: every output within
1e-5 * sum_k |a^||b^| (f32 output; bf16 output adds one bf16 rounding).
Operands are quantized by the oracle, so no expected value comes from the
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


def _mx8_operand(xb):
    q, s = oracle.mxfp8_quantize_rowwise(xb)
    return q, s


def _check(y, ref, absref, bf16=False, K=None):
    assert K is not None
    ok, bad = gemm_tolerance_ok(y, ref, absref, bf16, K)
    if not ok:
        yf = np.asarray(y, np.float64).ravel()
        i = bad[:5]
        raise AssertionError(f"{bad.size} outputs out of tolerance; e.g. idx {i}: "
                             f"got {yf[i]}, ref {ref.ravel()[i]}, abs {absref.ravel()[i]}")


def _run_mx8(A, SA, B, SB, K, out_dtype=torch.float32):
    return mx.bs_gemm(mx.FMT_MXFP8, dev(A), dev(oracle.swizzle_scales(SA)), dev(B),
                      dev(oracle.swizzle_scales(SB)), K, out_dtype=out_dtype)


def test_mxfp8_one_nonzero():
    """Pins operand order, K position and scale placement: a single nonzero in
    row 37 of A and row 90 of B at k = 200 gives one nonzero output."""
    M, N, K = 128, 128, 256
    A = np.zeros((M, K), np.uint8); B = np.zeros((N, K), np.uint8)
    SA = np.full((M, K // 32), 127, np.uint8); SB = np.full((N, K // 32), 127, np.uint8)
    A[37, 200] = 0x4C; B[90, 200] = 0xB9
    SA[37, 200 // 32] = 131; SB[90, 200 // 32] = 125
    y = host(_run_mx8(A, SA, B, SB, K))
    ref, absref = oracle.gemm_ref(0, A, SA, B, SB, K)
    assert np.count_nonzero(ref) == 1
    _check(y, ref, absref, K=K)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (200, 72, 96), (1, 8, 32), (257, 384, 1056),
                                   (128, 128, 32)])
def test_mxfp8_gemm_shapes(M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    xa = inputs.bits(inputs.sweep(M, K, seed=M + 1).float().clamp(-1e4, 1e4).to(torch.bfloat16))
    xb = inputs.bits(inputs.sweep(N, K, seed=N + 2).float().clamp(-1e4, 1e4).to(torch.bfloat16))
    A, SA = _mx8_operand(xa)
    B, SB = _mx8_operand(xb)
    y = host(_run_mx8(A, SA, B, SB, K))
    ref, absref = oracle.gemm_ref(0, A, SA, B, SB, K)
    _check(y, ref, absref, K=K)
    yb = host(_run_mx8(A, SA, B, SB, K, torch.bfloat16))
    _check(oracle.bf16_to_f32(yb), ref, absref, bf16=True, K=K)
    del rng


def test_mxfp8_pr1_fprop():
    d = inputs.pr1()
    A, SA = _mx8_operand(inputs.bits(d["X"]))
    B, SB = _mx8_operand(inputs.bits(d["W"]))
    y = host(_run_mx8(A, SA, B, SB, 512))
    ref, absref = oracle.gemm_ref(0, A, SA, B, SB, 512)
    _check(y, ref, absref, K=512)


def _sample_pairs(M, N, n, seed):
    rng = np.random.default_rng(seed)
    pairs = np.stack([rng.integers(0, M, n), rng.integers(0, N, n)], 1)
    # include the corners of the output
    corners = np.array([[0, 0], [M - 1, N - 1], [0, N - 1], [M - 1, 0]])
    return np.concatenate([corners, pairs])


def test_mxfp8_linear_fprop_dgrad_wgrad_full_size():
    """The 2048x2048 -> 8192 linear layer: Fprop from the rowwise copies,
    Dgrad from dY rowwise and W columnwise, Wgrad from the columnwise copies
    of dY and X; sampled outputs against the FP64 oracle."""
    d = inputs.linear(device="cuda")
    Xb, Wb, dYb = (inputs.bits(d[k]) for k in ("X", "W", "dY"))
    Xr, SXr = oracle.mxfp8_quantize_rowwise(Xb)
    Wr, SWr = oracle.mxfp8_quantize_rowwise(Wb)
    dYr, SdYr = oracle.mxfp8_quantize_rowwise(dYb)
    Wc, SWc = oracle.mxfp8_quantize_colwise(Wb)
    Xc, SXc = oracle.mxfp8_quantize_colwise(Xb)
    dYc, SdYc = oracle.mxfp8_quantize_colwise(dYb)
    cases = {
        "fprop": (Xr, SXr, Wr, SWr, 2048),     # Y[2048, 8192]
        "dgrad": (dYr, SdYr, Wc, SWc, 8192),   # dX[2048, 2048]
        "wgrad": (dYc, SdYc, Xc, SXc, 2048),   # dW[8192, 2048]
    }
    for seed, (name, (A, SA, B, SB, K)) in enumerate(cases.items()):
        y = host(_run_mx8(A, SA, B, SB, K))
        pairs = _sample_pairs(A.shape[0], B.shape[0], 3000, 100 + seed)
        ref, absref = oracle.gemm_ref(0, A, SA, B, SB, K, pairs=pairs)
        _check(y[pairs[:, 0], pairs[:, 1]], ref, absref, K=K)


# ------------------------------------------------------------------ NVFP4
def _nv_operand(xb, scope=oracle.SCOPE_TOKEN, offs=None):
    return oracle.nvfp4_quantize(xb, scope, offs)


def test_nvfp4_one_nonzero():
    M, N, K = 128, 128, 256
    A = np.zeros((M, K // 2), np.uint8); B = np.zeros((N, K // 2), np.uint8)
    SA = np.full((M, K // 16), 0x38, np.uint8); SB = np.full((N, K // 16), 0x38, np.uint8)
    A[5, 77] = 0x70      # element 155 = +6 (high nibble of byte 77)
    B[100, 77] = 0x30    # element 155 = +1.5
    SA[5, 155 // 16] = 0x40; SB[100, 155 // 16] = 0x30
    a32 = np.ones(M, np.float32); a32[5] = 0.25
    b32 = np.array([3.0], np.float32)
    y = host(mx.bs_gemm(mx.FMT_NVFP4, dev(A), dev(oracle.swizzle_scales(SA)), dev(B),
                        dev(oracle.swizzle_scales(SB)), K, dev(a32), dev(b32)))
    ref, absref = oracle.gemm_ref(1, A, SA, B, SB, K, a32, b32)
    assert np.count_nonzero(ref) == 1
    _check(y, ref, absref, K=K)


def test_nvfp4_pr1_per_token_x_per_tensor_w():
    d = inputs.pr1()
    A, SA, a32 = _nv_operand(inputs.bits(d["X"]))
    B, SB, b32 = _nv_operand(inputs.bits(d["W"]), oracle.SCOPE_TENSOR)
    y = host(mx.bs_gemm(mx.FMT_NVFP4, dev(A), dev(oracle.swizzle_scales(SA)), dev(B),
                        dev(oracle.swizzle_scales(SB)), 512, dev(a32), dev(b32)))
    ref, absref = oracle.gemm_ref(1, A, SA, B, SB, 512, a32, b32)
    _check(y, ref, absref, K=512)


@pytest.mark.parametrize("M,N,K", [(200, 136, 96), (128, 256, 1024), (3, 8, 32), (130, 128, 544)])
def test_nvfp4_gemm_shapes_per_row_scales(M, N, K):
    xa = inputs.bits(inputs.normal_bf16((M, K), 1.0, torch.Generator().manual_seed(M), "cpu", 0.01, 50))
    xb = inputs.bits(inputs.normal_bf16((N, K), 1.0, torch.Generator().manual_seed(N + 1), "cpu"))
    A, SA, a32 = _nv_operand(xa)
    B, SB, b32 = _nv_operand(xb)              # per-row FP32 scale on B too
    y = host(mx.bs_gemm(mx.FMT_NVFP4, dev(A), dev(oracle.swizzle_scales(SA)), dev(B),
                        dev(oracle.swizzle_scales(SB)), K, dev(a32), dev(b32)))
    ref, absref = oracle.gemm_ref(1, A, SA, B, SB, K, a32, b32)
    _check(y, ref, absref, K=K)


# ------------------------------------------------------------------ grouped
def _grouped_case(T, H, E, N, topk, seed, zipf=False):
    d = inputs.moe(seed, "cpu", T, H, E, N // 2, topk, routing="zipf" if zipf else "uniform",
                   with_weights=True)
    disp = inputs.dispatch(d["topk_ids"], E)
    offs = disp.offsets.numpy()
    Ab = inputs.bits(d["X"][disp.token_of_row])
    Wb = inputs.bits(d["W_gu"]).reshape(E * N, H)
    A, SA, a32 = _nv_operand(Ab)
    B, SB, b32 = _nv_operand(Wb, oracle.SCOPE_GROUP, np.arange(E + 1) * N)
    return offs, A, SA, a32, B.reshape(E, N, H // 2), SB, b32


@pytest.mark.parametrize("T,H,E,N,topk,zipf", [(64, 256, 5, 256, 2, False), (300, 512, 16, 384, 4, True),
                                               (40, 128, 7, 136, 1, False)])
def test_nvfp4_grouped_small(T, H, E, N, topk, zipf):
    offs, A, SA, a32, B, SB, b32 = _grouped_case(T, H, E, N, topk, seed=T, zipf=zipf)
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    y = host(mx.bs_grouped_gemm(mx.FMT_NVFP4, go, dev(A), dev(oracle.swizzle_scales(SA, offs)), dev(B),
                                dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N)), H, dev(a32), dev(b32),
                                out_dtype=torch.float32))
    rows = A.shape[0]
    pairs = np.array([(m, n) for m in range(rows) for n in range(N)])
    ref, absref = oracle.grouped_gemm_ref(1, offs, A, SA, B, SB, H, a32, b32, pairs)
    _check(y.ravel(), ref, absref, K=H)


@pytest.mark.parametrize("T,H,E,N,topk,zipf", [(64, 256, 5, 256, 2, False), (300, 512, 16, 384, 4, True),
                                               (40, 96, 7, 136, 1, False)])
def test_mxfp8_grouped(T, H, E, N, topk, zipf):
    """MXFP8 MoE grouped GEMM (one 512-byte scale tile per 128-element stage,
    staged into tensor memory by the producer warps and the MMA warp):
    routed token rows in the grouped scale layout times per-expert weights,
    ragged and Zipf-skewed groups, a K that ends inside a stage."""
    d = inputs.moe(T, "cpu", T, H, E, N // 2, topk, routing="zipf" if zipf else "uniform", with_weights=True)
    disp = inputs.dispatch(d["topk_ids"], E)
    offs = disp.offsets.numpy()
    A, SA = oracle.mxfp8_quantize_rowwise(inputs.bits(d["X"][disp.token_of_row]))
    B, SB = oracle.mxfp8_quantize_rowwise(inputs.bits(d["W_gu"]).reshape(E * N, H))
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    y = host(mx.bs_grouped_gemm(mx.FMT_MXFP8, go, dev(A), dev(oracle.swizzle_scales(SA, offs)),
                                dev(B.reshape(E, N, H)), dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N)), H,
                                out_dtype=torch.float32))
    rows = A.shape[0]
    pairs = np.array([(m, n) for m in range(rows) for n in range(N)])
    ref, absref = oracle.grouped_gemm_ref(0, offs, A, SA, B.reshape(E, N, H), SB, H, pairs=pairs)
    _check(y.ravel(), ref, absref, K=H)


def test_nvfp4_grouped_empty_and_single_row_groups():
    H, N, E = 256, 128, 6
    rng = np.random.default_rng(3)
    offs = np.array([0, 0, 1, 1, 129, 130, 260])
    Ab = inputs.bits(inputs.sweep(260, H, seed=5))
    Wb = inputs.bits(inputs.normal_bf16((E * N, H), 0.02, torch.Generator().manual_seed(9), "cpu"))
    A, SA, a32 = _nv_operand(Ab)
    B, SB, b32 = _nv_operand(Wb, oracle.SCOPE_GROUP, np.arange(E + 1) * N)
    B = B.reshape(E, N, H // 2)
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    y = host(mx.bs_grouped_gemm(mx.FMT_NVFP4, go, dev(A), dev(oracle.swizzle_scales(SA, offs)), dev(B),
                                dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N)), H, dev(a32), dev(b32),
                                out_dtype=torch.float32))
    pairs = np.array([(m, n) for m in range(260) for n in range(N)])
    ref, absref = oracle.grouped_gemm_ref(1, offs, A, SA, B, SB, H, a32, b32, pairs)
    _check(y.ravel(), ref, absref, K=H)
    del rng


def test_nvfp4_grouped_qwen_gate_up_sampled():
    """Qwen3-30B-A3B-shaped gate|up GEMM: 4096 tokens x top-8 over 128
    experts, hidden 2048 -> 2*768, bf16 output; sampled rows checked."""
    offs, A, SA, a32, B, SB, b32 = _grouped_case(4096, 2048, 128, 1536, 8, seed=2)
    E, N, H = 128, 1536, 2048
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    y = host(mx.bs_grouped_gemm(mx.FMT_NVFP4, go, dev(A), dev(oracle.swizzle_scales(SA, offs)), dev(B),
                                dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N)), H, dev(a32), dev(b32),
                                out_dtype=torch.bfloat16))
    pairs = _sample_pairs(A.shape[0], N, 3000, 7)
    ref, absref = oracle.grouped_gemm_ref(1, offs, A, SA, B, SB, H, a32, b32, pairs)
    _check(oracle.bf16_to_f32(y[pairs[:, 0], pairs[:, 1]]), ref, absref, bf16=True, K=H)
