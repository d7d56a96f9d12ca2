"""Full-size workload parity on the GPU, checked against the oracle on seeded
samples: the DeepSeek-V3-shaped NVFP4 MoE layer (2% of token rows and a few
experts, whose weights the oracle quantizes in full) and the quantizer
bandwidth sweep from 2^20 to 2^30 elements (sampled rows and 32-row slabs)."""
import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import ensure_built, gemm_tolerance_ok, grouped_padded_row, host, scale_offsets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_dsv3_moe_layer_sampled():
    """16384 tokens, hidden 7168, 256 routed experts, FFN 2048, top-8 Zipf(1.1),
    0.5% of activations x100: per-token quantization of the dispatched rows,
    per-expert quantization of gate|up, grouped gate|up GEMM."""
    E, H, F = 256, 7168, 2048
    d = inputs.dsv3_moe(device="cuda")
    disp = inputs.dispatch(d["topk_ids"], E)
    offs = host(disp.offsets).astype(np.int64)
    R = int(offs[-1])
    A = d["X"][disp.token_of_row].contiguous()
    del d["X"]
    Wgu = d.pop("W_gu").reshape(E * 2 * F, H)
    d.pop("W_d")
    go = disp.offsets
    eoffs = torch.arange(E + 1, device="cuda", dtype=torch.int64) * (2 * F)
    qa, sa, a32 = mx.nvfp4_quantize_per_token(A, group_offsets=go)
    qw, sw, w32 = mx.nvfp4_quantize_per_token(Wgu, mx.SCOPE_GROUP, eoffs)
    Y = mx.bs_grouped_gemm(mx.FMT_NVFP4, go, qa, sa, qw.view(E, 2 * F, H // 2), sw, H, a32, w32,
                           out_dtype=torch.float32)
    torch.cuda.synchronize()

    rng = np.random.default_rng(33)
    # 2% of the dispatched token rows: codes, block scales, FP32 scales
    rows = np.sort(rng.choice(R, size=R // 50, replace=False))
    Ab = inputs.bits(A[torch.from_numpy(rows).cuda()])
    oq, os_, o32 = oracle.nvfp4_quantize(Ab)
    assert np.array_equal(host(qa)[rows], oq)
    assert np.array_equal(host(a32)[rows].view(np.uint32), o32.view(np.uint32))
    sbuf = host(sa)
    assert np.array_equal(sbuf[scale_offsets(rows, H // 16, grouped_padded_row(offs))], os_)

    # a few experts (2% of 256 = 5), weights quantized in full by the oracle
    experts = np.sort(rng.choice(E, size=5, replace=False))
    swh, w32h = host(sw), host(w32)
    for e in experts:
        Wb = inputs.bits(Wgu[e * 2 * F:(e + 1) * 2 * F])
        wq, ws, w32e = oracle.nvfp4_quantize(Wb, oracle.SCOPE_TENSOR)
        assert np.array_equal(host(qw[e * 2 * F:(e + 1) * 2 * F]), wq)
        assert w32h[e].view(np.uint32) == w32e[0].view(np.uint32)
        er = np.arange(e * 2 * F, (e + 1) * 2 * F)
        assert np.array_equal(swh[scale_offsets(er, H // 16)], ws)
        # GEMM outputs of sampled rows routed to this expert
        erows = np.arange(offs[e], offs[e + 1])
        if erows.size == 0:
            continue
        pick = rng.choice(erows, size=min(erows.size, 24), replace=False)
        pq, ps, p32 = oracle.nvfp4_quantize(inputs.bits(A[torch.from_numpy(pick).cuda()]))
        ns = rng.integers(0, 2 * F, size=64)
        pairs = np.array([(i, n) for i in range(len(pick)) for n in ns])
        ref, absref = oracle.gemm_ref(1, pq, ps, wq, ws, H, p32, w32e, pairs=pairs)
        y = host(Y[torch.from_numpy(pick[pairs[:, 0]]).cuda(), torch.from_numpy(pairs[:, 1]).cuda()])
        ok, bad = gemm_tolerance_ok(y, ref, absref, K=H)
        assert ok, (e, bad[:5])


@pytest.mark.parametrize("numel,cols", [(1 << 20, 2048), (1 << 24, 4096), (1 << 27, 7168), (1 << 30, 2048)])
def test_quantizer_sweep_sampled(numel, cols):
    rows = max(128, (numel // cols) // 128 * 128)
    x = inputs.sweep(rows, cols, seed=4 + numel.bit_length(), device="cuda")
    q_r, s_r, q_c, s_c = mx.mx8_quantize(x)
    q4, s4, s32 = mx.nvfp4_quantize_per_token(x)
    torch.cuda.synchronize()
    rng = np.random.default_rng(numel.bit_length())
    # rowwise MXFP8 and per-token NVFP4 on sampled rows
    rs = np.sort(rng.choice(rows, size=64, replace=False))
    xb = inputs.bits(x[torch.from_numpy(rs).cuda()])
    oq, os_ = oracle.mxfp8_quantize_rowwise(xb)
    assert np.array_equal(host(q_r[torch.from_numpy(rs).cuda()]), oq)
    assert np.array_equal(host(s_r)[scale_offsets(rs, cols // 32)], os_)
    nq, ns, n32 = oracle.nvfp4_quantize(xb)
    assert np.array_equal(host(q4[torch.from_numpy(rs).cuda()]), nq)
    assert np.array_equal(host(s32)[rs].view(np.uint32), n32.view(np.uint32))
    assert np.array_equal(host(s4)[scale_offsets(rs, cols // 16)], ns)
    # columnwise MXFP8 on sampled 32-row slabs
    for b in rng.choice(rows // 32, size=4, replace=False):
        slab = inputs.bits(x[32 * b:32 * b + 32])
        cq, cs = oracle.mxfp8_quantize_colwise(slab)
        assert np.array_equal(host(q_c[:, 32 * b:32 * b + 32]), cq)
        got = host(s_c)[scale_offsets(np.arange(cols), rows // 32)][:, b]
        assert np.array_equal(got, cs[:, 0])
