"""Parity of the MoE expert GEMMs at the exact shapes the benchmark runs,
against the oracle on sampled rows (every output column of each sampled row).

Qwen3-30B-A3B shape: 4096 tokens, top-8 of 128 experts (32768 dispatched
rows), hidden 2048, FFN 768.  DeepSeek-V3 shape: 16384 tokens, top-8 Zipf(1.1)
of 256 experts (131072 rows), hidden 7168, FFN 2048, 0.5% of activations
x100.  The layer runs as in the benchmark: tokens NVFP4-encoded once before
dispatch, per-expert weight quantization (gate|up joint), the gate|up grouped
GEMM with SwiGLU in the epilogue, per-token quantization of h, the down
grouped GEMM ("Miles Blackwell RL Cambia la Uniformidad BF16 por MXFP8 y
NVFP4 Nativos", sections "La Compatibilidad..." and "Un Cuantizador
Compartido..."; "Miles Blackwell MXFP8 / NVFP4 RL recipes", NVFP4 on MoE
experts).

The oracle quantizes the sampled token rows and every weight of the sampled
experts in full, and computes the FP64 GEMM references of those rows; h is
checked against silu(g) u of those references with the GEMM tolerance carried
through, and the down GEMM's input is the GPU's own h, quantized by the
oracle (codes and scales compared byte for byte first)."""
import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import ensure_built, gemm_tolerance_ok, grouped_padded_row, host, scale_offsets, swiglu_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _layer(d, E, F, topk):
    """The expert layer of the benchmark on the device; returns what the
    checks need (weights stay in bf16 for the oracle's per-expert copies)."""
    H = d["X"].shape[1]
    disp = inputs.dispatch(d["topk_ids"], E)
    go = disp.offsets
    dest = torch.argsort(disp.token_of_row, stable=True).to(torch.int64).contiguous()
    a4, sa4, a32 = mx.nvfp4_quantize_dispatch(d["X"], dest, topk, go, mx.DISPATCH_ROWS)
    Wgu = d["W_gu"].reshape(E * 2 * F, H)
    wgu4, swgu, wgu32 = mx.nvfp4_quantize_per_token(
        Wgu, mx.SCOPE_GROUP, torch.arange(E + 1, device="cuda", dtype=torch.int64) * (2 * F))
    h = mx.bs_grouped_gemm_fused(mx.FMT_NVFP4, go, a4, sa4, wgu4.view(E, 2 * F, H // 2), swgu, H, a32, wgu32,
                                 epilogue=mx.EPI_SWIGLU)
    h4, sh4, h32 = mx.nvfp4_quantize_per_token(h, group_offsets=go)
    Wd = d["W_d"].reshape(E * H, F)
    wd4, swd, wd32 = mx.nvfp4_quantize_per_token(
        Wd, mx.SCOPE_GROUP, torch.arange(E + 1, device="cuda", dtype=torch.int64) * H)
    out = mx.bs_grouped_gemm(mx.FMT_NVFP4, go, h4, sh4, wd4.view(E, H, F // 2), swd, F, h32, wd32,
                             out_dtype=torch.bfloat16)
    fused = None
    if F <= 1024:
        # the same gate|up GEMM with h quantized in its epilogue (one cluster per band)
        fused = mx.bs_grouped_gemm_swiglu_nvfp4(go, a4, sa4, wgu4.view(E, 2 * F, H // 2), swgu, H, a32, wgu32)
    torch.cuda.synchronize()
    return dict(offs=host(go).astype(np.int64), tor=host(disp.token_of_row).astype(np.int64), X=d["X"],
                W_gu=d["W_gu"], W_d=d["W_d"], h=h, h4=h4, sh4=sh4, h32=h32, out=out, H=H, F=F, fused=fused)


def _sample(offs, experts, rows_per_expert, rng):
    """Sampled dispatched rows of the given experts: random rows plus each
    expert's last row (the ragged end of its last 128-row tile)."""
    picked = {}
    for e in experts:
        lo, hi = offs[e], offs[e + 1]
        if hi == lo:
            continue
        r = rng.choice(np.arange(lo, hi), size=min(rows_per_expert, hi - lo), replace=False)
        picked[int(e)] = np.unique(np.append(r, hi - 1))
    return picked


def _check_swiglu(L, picked):
    """Every h column of the sampled rows against the FP64 gate and up
    references of the oracle's own quantization of those rows and experts."""
    H, F = L["H"], L["F"]
    hrows = host(L["h"][torch.from_numpy(np.concatenate(list(picked.values()))).cuda()])
    done = 0
    for e, rows in picked.items():
        xb = inputs.bits(L["X"][torch.from_numpy(L["tor"][rows]).cuda()])
        aq, as_, a32 = oracle.nvfp4_quantize(xb)                     # per token: the dispatched copies' bytes
        wq, ws, w32 = oracle.nvfp4_quantize(inputs.bits(L["W_gu"][e]), oracle.SCOPE_TENSOR)
        pg = np.array([(i, n) for i in range(rows.size) for n in range(F)])
        g, ag = oracle.gemm_ref(1, aq, as_, wq, ws, H, a32, w32, pairs=pg)
        u, au = oracle.gemm_ref(1, aq, as_, wq, ws, H, a32, w32, pairs=pg + np.array([0, F]))
        href, tol = swiglu_tolerance(g, ag, u, au, H)
        got = oracle.bf16_to_f32(hrows[done:done + rows.size]).astype(np.float64).ravel()
        done += rows.size
        bad = np.nonzero(np.abs(got - href) > tol)[0]
        assert bad.size == 0, (e, bad.size, got[bad[:4]], href[bad[:4]])


def _check_down(L, picked):
    """The GPU's h rows quantized by the oracle (byte for byte against the
    GPU's codes, block scales and S_dec), then every output column of the
    down GEMM for those rows against the FP64 reference."""
    H, F = L["H"], L["F"]
    pad = grouped_padded_row(L["offs"])
    h4, sh4, h32, out = host(L["h4"]), host(L["sh4"]), host(L["h32"]), L["out"]
    for e, rows in picked.items():
        hb = host(L["h"][torch.from_numpy(rows).cuda()])
        hq, hs, hd = oracle.nvfp4_quantize(hb)
        assert np.array_equal(h4[rows], hq)
        assert np.array_equal(h32[rows].view(np.uint32), hd.view(np.uint32))
        assert np.array_equal(sh4[scale_offsets(rows, F // 16, pad)], hs)
        wq, ws, w32 = oracle.nvfp4_quantize(inputs.bits(L["W_d"][e]), oracle.SCOPE_TENSOR)
        pairs = np.array([(i, n) for i in range(rows.size) for n in range(H)])
        ref, absref = oracle.gemm_ref(1, hq, hs, wq, ws, F, hd, w32, pairs=pairs)
        y = oracle.bf16_to_f32(host(out[torch.from_numpy(rows).cuda()])).astype(np.float64).ravel()
        ok, bad = gemm_tolerance_ok(y, ref, absref, bf16=True, K=F)
        assert ok, (e, bad.size, y[bad[:4]], ref[bad[:4]])


@pytest.fixture(scope="module")
def qwen():
    q = inputs.QWEN_SHAPE
    L = _layer(inputs.qwen_moe(seed=2, device="cuda"), q["experts"], q["ffn"], q["topk"])
    rng = np.random.default_rng(11)
    experts = np.sort(rng.choice(q["experts"], size=6, replace=False))
    L["picked"] = _sample(L["offs"], experts, 10, rng)
    return L


def test_qwen_gate_up_swiglu_full_shape(qwen):
    """Fused gate|up + SwiGLU at K = 2048, F = 768 (six 128-column h tiles per
    row), every h column of 66 sampled rows across 6 experts."""
    _check_swiglu(qwen, qwen["picked"])


def test_qwen_down_full_shape(qwen):
    """Per-token quantization of h (768 columns) and the down GEMM at
    K = 768, N = 2048, every output column of the sampled rows."""
    _check_down(qwen, qwen["picked"])


def test_qwen_quantized_h_full_shape(qwen):
    """The fused gate|up + SwiGLU + per-token NVFP4 of h at the Qwen shape
    (clusters of 6 CTAs, one per 128-column h tile): codes, block scales and
    S_dec of every dispatched row equal the separate quantizer's on the
    SwiGLU epilogue's h, byte for byte (that quantizer is checked against the
    oracle on the sampled rows in test_qwen_down_full_shape)."""
    qh, sh, s32h = qwen["fused"]
    assert torch.equal(qh, qwen["h4"])
    assert torch.equal(s32h.view(torch.int32), qwen["h32"].view(torch.int32))
    n = oracle.swizzled_bytes(qwen["h"].shape[0], qwen["F"] // 16, qwen["offs"])
    assert torch.equal(sh[:n], qwen["sh4"][:n])


@pytest.fixture(scope="module")
def dsv3():
    q = inputs.DSV3_SHAPE
    L = _layer(inputs.dsv3_moe(seed=3, device="cuda"), q["experts"], q["ffn"], q["topk"])
    rng = np.random.default_rng(12)
    # 2% of the 256 experts (5), chosen at random
    experts = np.sort(rng.choice(q["experts"], size=5, replace=False))
    L["picked"] = _sample(L["offs"], experts, 4, rng)
    return L


def test_dsv3_gate_up_swiglu_sampled(dsv3):
    """Fused gate|up + SwiGLU at K = 7168, F = 2048 on sampled rows of 5
    experts (every h column)."""
    _check_swiglu(dsv3, dsv3["picked"])


def test_dsv3_down_sampled(dsv3):
    """Per-token quantization of h (2048 columns) and the down GEMM at
    K = 2048, N = 7168 on the same rows (every output column)."""
    _check_down(dsv3, dsv3["picked"])
