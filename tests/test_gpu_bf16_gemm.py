"""GPU parity of the dense BF16 tcgen05 GEMM (kind::f16) of the
dequantized-backward mode ("Miles Blackwell RL Cambia la Uniformidad BF16 por
MXFP8 y NVFP4 Nativos", section "La Compatibilidad...": Dgrad and Wgrad in
BF16 on operands rebuilt from the low-precision copies) against the oracle's
FP64 reference: every output within 1e-5 * sum_k |a||b| (f32 output; bf16
output adds one bf16 rounding)."""
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


def _check(y, ref, absref, bf16=False, K=None):
    ok, bad = gemm_tolerance_ok(y, ref, absref, bf16, K)
    if not ok:
        yf = np.asarray(y, np.float64).ravel()
        i = bad[:5]
        raise AssertionError(f"{bad.size} outputs out of tolerance; e.g. idx {i}: "
                             f"got {yf[i]}, ref {ref.ravel()[i]}, abs {absref.ravel()[i]}")


def _normal(rows, K, std, seed):
    return inputs.bits(inputs.normal_bf16((rows, K), std, torch.Generator().manual_seed(seed), "cpu"))


@pytest.mark.parametrize("k", [5, 63, 64, 200])
def test_bf16_one_nonzero(k):
    """Pins operand order and the K position: a single nonzero in row 37 of A
    and row 90 of B at k gives one nonzero output, 3 * -0.5."""
    M, N, K = 128, 128, 256
    A = np.zeros((M, K), np.uint16); B = np.zeros((N, K), np.uint16)
    A[37, k] = 0x4040          # 3.0
    B[90, k] = 0xBF00          # -0.5
    y = host(mx.bf16_gemm(dev(A), dev(B)))
    ref, absref = oracle.bf16_gemm_ref(A, B)
    assert np.count_nonzero(ref) == 1 and ref[37, 90] == -1.5
    _check(y, ref, absref, K=K)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (200, 72, 96), (1, 8, 8), (257, 384, 1064),
                                   (130, 520, 40), (64, 256, 2048)])
def test_bf16_gemm_shapes(M, N, K):
    a, b = _normal(M, K, 1.0, M + 3), _normal(N, K, 0.5, N + 4)
    ref, absref = oracle.bf16_gemm_ref(a, b)
    y = host(mx.bf16_gemm(dev(a), dev(b)))
    _check(y, ref, absref, K=K)
    yb = host(mx.bf16_gemm(dev(a), dev(b), out_dtype=torch.bfloat16))
    _check(oracle.bf16_to_f32(yb), ref, absref, bf16=True, K=K)


def test_bf16_gemm_strided_operands_and_accumulate():
    M, N, K = 160, 200, 256
    a, b = _normal(M, K, 1.0, 8), _normal(N, K, 1.0, 9)
    big_a = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    big_b = torch.zeros((N, K + 8), dtype=torch.bfloat16, device="cuda")
    big_a[:, :K] = dev(a)
    big_b[:, :K] = dev(b)
    c0 = np.random.default_rng(3).standard_normal((M, N)).astype(np.float32)
    out = dev(c0)
    mx.bf16_gemm_into(big_a[:, :K], big_b[:, :K], out, accumulate=True)
    ref, absref = oracle.bf16_gemm_ref(a, b)
    _check(host(out).astype(np.float64) - c0, ref, absref + np.abs(c0), K=K)


def _sample_pairs(M, N, n, seed):
    rng = np.random.default_rng(seed)
    pairs = np.stack([rng.integers(0, M, n), rng.integers(0, N, n)], 1)
    corners = np.array([[0, 0], [M - 1, N - 1], [0, N - 1], [M - 1, 0]])
    return np.concatenate([corners, pairs])


def test_dequantized_backward_full_size():
    """The 2048x2048 -> 8192 linear layer: X, W and dY quantized to MXFP8 on
    the GPU (bytes checked against the oracle), the backward operands rebuilt
    by dequantize() in bf16, then Dgrad = deq(dY_row) deq(W_col)^T and
    Wgrad = deq(dY_col) deq(X_col)^T in BF16.  The reference is the oracle's
    block-scaled GEMM on the oracle's quantized operands: the dequantized
    values are exact in bf16, so both sum the same products."""
    d = inputs.linear(device="cuda")
    Xb, Wb, dYb = (inputs.bits(d[k]) for k in ("X", "W", "dY"))
    gx, gw, gdy = (mx.mx8_quantize(d[k]) for k in ("X", "W", "dY"))
    dYr, SdYr = oracle.mxfp8_quantize_rowwise(dYb)
    Wc, SWc = oracle.mxfp8_quantize_colwise(Wb)
    dYc, SdYc = oracle.mxfp8_quantize_colwise(dYb)
    Xc, SXc = oracle.mxfp8_quantize_colwise(Xb)
    assert np.array_equal(host(gdy[0]), dYr) and np.array_equal(host(gw[2]), Wc)
    assert np.array_equal(host(gdy[2]), dYc) and np.array_equal(host(gx[2]), Xc)
    deq = lambda q, s: mx.dequantize(mx.FMT_MXFP8, q, s, out_dtype=torch.bfloat16)
    cases = {
        "dgrad": (deq(gdy[0], gdy[1]), deq(gw[2], gw[3]), (dYr, SdYr, Wc, SWc), 8192),   # dX [2048, 2048]
        "wgrad": (deq(gdy[2], gdy[3]), deq(gx[2], gx[3]), (dYc, SdYc, Xc, SXc), 2048),   # dW [8192, 2048]
    }
    for name, (A, B, ops, K) in cases.items():
        y = host(mx.bf16_gemm(A, B, out_dtype=torch.float32))
        qa, sa, qb, sb = ops
        pairs = _sample_pairs(qa.shape[0], qb.shape[0], 2000, 23)
        ref, absref = oracle.gemm_ref(0, qa, sa, qb, sb, K, pairs=pairs)
        _check(y[pairs[:, 0], pairs[:, 1]], ref, absref, K=K)
