"""GPU parity of the fused MoE expert GEMM: tokens quantized once before
dispatch and gathered by the GEMM's producer, and the SwiGLU of the joint
gate|up output done in the epilogue ("Miles Blackwell RL Cambia la
Uniformidad BF16 por MXFP8 y NVFP4 Nativos", sections "La Compatibilidad..."
and "Un Cuantizador Compartido...").  References are the oracle's FP64
grouped GEMM over the dispatched operands (per-token quantization commutes
with the dispatch gather: an oracle pin; the before-dispatch quantizer is
checked byte for byte) and, for h, silu(g) * u
in FP64 over those references, with the GEMM tolerance carried through."""
import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import ensure_built, gemm_tolerance_ok, host, dev, swiglu_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _case(T, H, E, N, topk, seed, zipf=False):
    """Token-major NVFP4 activations and per-expert weights [E, N, H] with
    one FP32 scale per expert; N = 2F rows (gate then up)."""
    d = inputs.moe(seed, "cpu", T, H, E, N // 2, topk, routing="zipf" if zipf else "uniform",
                   with_weights=True)
    disp = inputs.dispatch(d["topk_ids"], E)
    offs = disp.offsets.numpy()
    tor = disp.token_of_row.numpy()
    Xb = inputs.bits(d["X"])
    Aq, SAq, a32 = oracle.nvfp4_quantize(Xb)                              # per token, before dispatch
    Wb = inputs.bits(d["W_gu"]).reshape(E * N, H)
    B, SB, b32 = oracle.nvfp4_quantize(Wb, oracle.SCOPE_GROUP, np.arange(E + 1) * N)
    return offs, tor, Xb, Aq, SAq, a32, B.reshape(E, N, H // 2), SB, b32


def _dispatched(tor, Aq, SAq, a32):
    return Aq[tor], SAq[tor], a32[tor]


def _dest_rows(tor, topk):
    """Inverse of the row -> token map: the topk dispatched rows of each token."""
    return np.argsort(tor, kind="stable").reshape(-1, topk)


@pytest.mark.parametrize("layout", [mx.DISPATCH_ROWS, mx.DISPATCH_TOKENS])
@pytest.mark.parametrize("T,H,E,topk,zipf", [(64, 256, 5, 2, False), (300, 2048, 16, 8, True),
                                             (40, 96, 7, 1, False), (33, 4096, 3, 3, False)])
def test_quantize_dispatch_bit_exact(T, H, E, topk, zipf, layout):
    """Codes and S_dec (per dispatched row, or token-major) and the
    dispatched rows' block scales in the grouped layout (padding zero), byte
    for byte against the oracle's quantization of the dispatched rows."""
    offs, tor, Xb, Aq, SAq, a32, *_ = _case(T, H, E, 128, topk, seed=T + 7, zipf=zipf)
    dest = torch.tensor(_dest_rows(tor, topk), dtype=torch.int64, device="cuda")
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    q, sb, s32 = mx.nvfp4_quantize_dispatch(dev(Xb), dest, topk, go, layout)
    dq, dsc, d32 = oracle.nvfp4_quantize(Xb[tor])          # the dispatched rows, quantized directly
    if layout == mx.DISPATCH_ROWS:
        assert np.array_equal(host(q), dq)
        assert np.array_equal(host(s32).view(np.uint32), d32.view(np.uint32))
    else:
        assert np.array_equal(host(q), Aq)
        assert np.array_equal(host(s32).view(np.uint32), a32.view(np.uint32))
    sw = oracle.swizzle_scales(dsc, offs)
    assert np.array_equal(host(sb)[: sw.size], sw)


def _check(y, ref, absref, bf16=False, K=None):
    ok, bad = gemm_tolerance_ok(y, ref, absref, bf16, K)
    if not ok:
        yf = np.asarray(y, np.float64).ravel()
        i = bad[:5]
        raise AssertionError(f"{bad.size} outputs out of tolerance; e.g. idx {i}: "
                             f"got {yf[i]}, ref {ref.ravel()[i]}, abs {absref.ravel()[i]}")


@pytest.mark.parametrize("T,H,E,N,topk,zipf", [(64, 256, 5, 256, 2, False), (300, 512, 16, 384, 4, True),
                                               (40, 96, 7, 136, 1, False)])
def test_gathered_grouped_gemm(T, H, E, N, topk, zipf):
    offs, tor, _, Aq, SAq, a32, B, SB, b32 = _case(T, H, E, N, topk, seed=T + 1, zipf=zipf)
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    rows_t = torch.tensor(tor, dtype=torch.int64, device="cuda")
    y = host(mx.bs_grouped_gemm_fused(mx.FMT_NVFP4, go, dev(Aq), dev(oracle.swizzle_scales(SAq[tor], offs)), dev(B),
                                      dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N)), H, dev(a32), dev(b32),
                                      a_rows=rows_t, out_dtype=torch.float32))
    A, SA, ad = _dispatched(tor, Aq, SAq, a32)
    rows = A.shape[0]
    pairs = np.array([(m, n) for m in range(rows) for n in range(N)])
    ref, absref = oracle.grouped_gemm_ref(1, offs, A, SA, B, SB, H, ad, b32, pairs)
    _check(y.ravel(), ref, absref, K=H)


@pytest.mark.parametrize("gather", [True, False])
@pytest.mark.parametrize("T,H,E,F,topk", [(64, 256, 5, 128, 2), (200, 512, 9, 256, 4)])
def test_swiglu_epilogue(gather, T, H, E, F, topk):
    N = 2 * F
    offs, tor, _, Aq, SAq, a32, B, SB, b32 = _case(T, H, E, N, topk, seed=T + F)
    A, SA, ad = _dispatched(tor, Aq, SAq, a32)
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    sbw = dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N))
    if gather:
        h = mx.bs_grouped_gemm_fused(mx.FMT_NVFP4, go, dev(Aq), dev(oracle.swizzle_scales(SA, offs)), dev(B), sbw, H,
                                     dev(a32), dev(b32), a_rows=torch.tensor(tor, dtype=torch.int64, device="cuda"),
                                     epilogue=mx.EPI_SWIGLU)
    else:
        h = mx.bs_grouped_gemm_fused(mx.FMT_NVFP4, go, dev(A), dev(oracle.swizzle_scales(SA, offs)), dev(B), sbw, H,
                                     dev(ad), dev(b32), epilogue=mx.EPI_SWIGLU)
    hh = oracle.bf16_to_f32(host(h)).astype(np.float64)
    rows = A.shape[0]
    pg = np.array([(m, n) for m in range(rows) for n in range(F)])
    pu = pg + np.array([0, F])
    g, ag = oracle.grouped_gemm_ref(1, offs, A, SA, B, SB, H, ad, b32, pg)
    u, au = oracle.grouped_gemm_ref(1, offs, A, SA, B, SB, H, ad, b32, pu)
    href, tol = swiglu_tolerance(g, ag, u, au, H)
    err = np.abs(hh.ravel() - href)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} h values out of tolerance, e.g. {hh.ravel()[bad[:4]]} vs {href[bad[:4]]}"
    # the fused epilogue rounds g and u to bf16 exactly where the unfused
    # gate|up output would be rounded, so it matches that path's SwiGLU
    gu = mx.bs_grouped_gemm(mx.FMT_NVFP4, go, dev(A), dev(oracle.swizzle_scales(SA, offs)), dev(B), sbw, H,
                            dev(ad), dev(b32), out_dtype=torch.bfloat16)
    h2 = mx.swiglu(gu)
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))


@pytest.mark.parametrize("T,H,E,topk,out_dtype", [(64, 256, 5, 2, torch.float32), (300, 512, 16, 8, torch.bfloat16),
                                                  (4096, 2048, 128, 8, torch.bfloat16)])
def test_moe_combine_bit_exact(T, H, E, topk, out_dtype):
    """The router-weighted sum of each token's expert outputs, bit for bit
    against the oracle's binary32 evaluation in the same order."""
    d = inputs.moe(T + 3, "cpu", T, H, E, 64, topk, with_weights=False)
    disp = inputs.dispatch(d["topk_ids"], E)
    rows = disp.row_of_slot
    w = inputs.route_weights(T, topk, T, "cpu")
    R = T * topk
    y = inputs.bits(inputs.normal_bf16((R, H), 1.0, torch.Generator().manual_seed(H), "cpu", 0.01, 30))
    out = mx.moe_combine(dev(y), rows.cuda(), w.cuda(), out_dtype=out_dtype)
    ref = oracle.moe_combine(y, rows.numpy(), w.numpy())
    if out_dtype == torch.float32:
        assert np.array_equal(host(out).view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(host(out), oracle.f32_to_bf16(ref))


@pytest.mark.parametrize("T,H,E,F,topk", [(64, 256, 5, 128, 2), (200, 512, 9, 256, 4), (150, 256, 4, 768, 3),
                                          (90, 512, 6, 1024, 2)])
def test_swiglu_quantized_h_bit_exact(T, H, E, F, topk):
    """gate|up GEMM + SwiGLU + per-token NVFP4 of h in one kernel (clusters of
    F / 128 CTAs exchanging row maxima): h equals the SwiGLU epilogue's, and
    the codes, block scales (grouped layout, padding zero) and S_dec of h
    equal the oracle's per-token quantization of that h byte for byte -- and
    the separate GPU quantizer's.  Without the h output the bytes are the
    same."""
    N = 2 * F
    offs, tor, _, Aq, SAq, a32, B, SB, b32 = _case(T, H, E, N, topk, seed=T + F + 3, zipf=True)
    A, SA, ad = _dispatched(tor, Aq, SAq, a32)
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    sa, sbw = dev(oracle.swizzle_scales(SA, offs)), dev(oracle.swizzle_scales(SB, np.arange(E + 1) * N))
    h_ref = mx.bs_grouped_gemm_fused(mx.FMT_NVFP4, go, dev(A), sa, dev(B), sbw, H, dev(ad), dev(b32),
                                     epilogue=mx.EPI_SWIGLU)
    qh, sh, s32h, h = mx.bs_grouped_gemm_swiglu_nvfp4(go, dev(A), sa, dev(B), sbw, H, dev(ad), dev(b32), with_h=True)
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    hq, hs, hd = oracle.nvfp4_quantize(host(h))
    assert np.array_equal(host(qh), hq)
    assert np.array_equal(host(s32h).view(np.uint32), hd.view(np.uint32))
    sw = oracle.swizzle_scales(hs, offs)
    assert np.array_equal(host(sh)[: sw.size], sw)
    gq, gs, g32 = mx.nvfp4_quantize_per_token(h, group_offsets=go)
    assert torch.equal(gq, qh) and torch.equal(g32.view(torch.int32), s32h.view(torch.int32))
    assert torch.equal(gs[: sw.size], sh[: sw.size])
    qh2, sh2, s32h2 = mx.bs_grouped_gemm_swiglu_nvfp4(go, dev(A), sa, dev(B), sbw, H, dev(ad), dev(b32))
    assert torch.equal(qh2, qh) and torch.equal(sh2[: sw.size], sh[: sw.size])
    assert torch.equal(s32h2.view(torch.int32), s32h.view(torch.int32))


def test_swiglu_quantized_h_rejects_wide_ffn():
    """More than 8 h tiles per band (F > 1024) do not fit one cluster."""
    E, F, H = 2, 1152, 256
    go = torch.tensor([0, 10, 20], dtype=torch.int64, device="cuda")
    A = torch.zeros((20, H // 2), dtype=torch.uint8, device="cuda")
    SA = torch.zeros(mx.scale_bytes_grouped(mx.FMT_NVFP4, 20, E, H), dtype=torch.uint8, device="cuda")
    B = torch.zeros((E, 2 * F, H // 2), dtype=torch.uint8, device="cuda")
    SB = torch.zeros(mx.scale_bytes(mx.FMT_NVFP4, E * 2 * F, H), dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.Mx8Error) as ei:
        mx.bs_grouped_gemm_swiglu_nvfp4(go, A, SA, B, SB, H)
    assert ei.value.status == mx.ERR_UNSUPPORTED
