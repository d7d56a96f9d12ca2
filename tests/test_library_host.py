"""Host-side checks of the C-ABI library that need no GPU: it builds for
sm_103a, loads, exports every symbol the header declares, sizes its buffers
as documented, and rejects bad arguments before any device work."""
import ctypes
import re

import pytest

from tests._lib import ROOT, ensure_built


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import moe_mx8_quantize_gb300 as m
    return m.load()


def _header_functions():
    src = open(f"{ROOT}/include/mx8q.h").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b([a-z_0-9]+)\s*\(", src)) - {"sizeof"}


def test_exports_every_declared_symbol(lib):
    import moe_mx8_quantize_gb300 as m
    declared = _header_functions()
    assert declared == set(m.EXPORTS), declared ^ set(m.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_scale_and_workspace_sizes(lib):
    import moe_mx8_quantize_gb300 as m
    # [R, C/32] padded to 128 x 4
    assert m.scale_bytes(m.FMT_MXFP8, 2048, 2048) == 2048 * 64
    assert m.scale_bytes(m.FMT_MXFP8, 130, 160) == 256 * 8
    assert m.scale_bytes(m.FMT_NVFP4, 1, 16) == 128 * 4
    assert m.scale_bytes(m.FMT_NVFP4, 4096, 2048) == 4096 * 128
    assert m.scale_bytes_grouped(m.FMT_NVFP4, 300, 4, 256) == (3 + 4) * 128 * 16
    # MXFP4 blocks are 32 wide like MXFP8
    assert m.scale_bytes(m.FMT_MXFP4, 130, 160) == 256 * 8
    assert m.scale_bytes(m.FMT_MXFP4, 2048, 2048) == 2048 * 64
    assert m.scale_bytes_grouped(m.FMT_MXFP4, 300, 4, 256) == (3 + 4) * 128 * 8
    assert m.workspace_bytes(1) >= 16 and m.workspace_bytes(256) >= 256 + 1024


def test_invalid_arguments_rejected_on_host(lib):
    import moe_mx8_quantize_gb300 as m
    p = ctypes.c_void_p(16)      # never dereferenced: validation fails first
    # cols not a multiple of 32
    assert lib.mx8_quantize(p, 64, 48, 48, m.ROWWISE, p, p, None, None, p, 4096, None) == m.ERR_INVALID_ARG
    # colwise needs rows % 32 == 0
    assert lib.mx8_quantize(p, 40, 64, 64, m.COLWISE, None, None, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    # no copy requested / unknown flag
    assert lib.mx8_quantize(p, 64, 64, 64, 0, p, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.mx8_quantize(p, 64, 64, 64, 8, p, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    # ld < cols
    assert lib.mx8_quantize(p, 64, 64, 32, m.ROWWISE, p, p, None, None, p, 4096, None) == m.ERR_INVALID_ARG
    # misaligned input pointer
    q = ctypes.c_void_p(24)
    assert lib.mx8_quantize(q, 64, 64, 64, m.ROWWISE, p, p, None, None, p, 4096, None) == m.ERR_ALIGNMENT
    # NVFP4: cols % 16, group scope without offsets, bad scope
    assert lib.nvfp4_quantize_per_token(p, 4, 24, 24, 0, None, 0, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token(p, 4, 32, 32, 1, None, 0, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token(p, 4, 32, 32, 7, None, 0, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    # MXFP4: same rules as MXFP8
    assert lib.mxfp4_quantize(p, 64, 48, 48, m.ROWWISE, p, p, None, None, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.mxfp4_quantize(p, 40, 64, 64, m.COLWISE, None, None, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.mxfp4_quantize(p, 64, 64, 64, 0, p, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.mxfp4_quantize(q, 64, 64, 64, m.ROWWISE, p, p, None, None, p, 4096, None) == m.ERR_ALIGNMENT
    assert lib.mxfp4_quantize(p, 64, 64, 64, m.ROWWISE, p, p, None, None, None, 0, None) == m.ERR_WORKSPACE
    assert lib.mxfp4_quantize(None, 0, 64, 64, m.ROWWISE, None, None, None, None, None, 0, None) == m.OK
    # workspace missing or too small
    assert lib.nvfp4_quantize_per_token(p, 4, 32, 32, 0, None, 0, p, p, p, None, 0, None) == m.ERR_WORKSPACE
    # GEMM: K % 32, ldc < N, accumulate into bf16, bad scale modes
    assert lib.bs_gemm(0, 8, 8, 48, p, p, None, 0, p, p, None, 0, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bs_gemm(0, 8, 16, 64, p, p, None, 0, p, p, None, 0, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bs_gemm(0, 8, 8, 64, p, p, None, 0, p, p, None, 0, 1, p, 8, 1, p, 4096, None) == m.ERR_UNSUPPORTED
    assert lib.bs_gemm(1, 8, 8, 64, p, p, None, 1, p, p, None, 0, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bs_gemm(0, 8, 8, 64, p, p, None, 0, p, p, None, 0, 0, p, 12, 0, p, 4096, None) == m.ERR_ALIGNMENT
    # unknown format; MXFP4 K % 32
    assert lib.bs_gemm(3, 8, 8, 64, p, p, None, 0, p, p, None, 0, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bs_gemm(2, 8, 8, 48, p, p, None, 0, p, p, None, 0, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    # grouped: group count out of range
    assert lib.bs_grouped_gemm(1, 0, p, 8, 8, 64, p, p, None, p, p, None, 0, p, 8, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm(1, 5000, p, 8, 8, 64, p, p, None, p, p, None, 0, p, 8, p, 1 << 20, None) == m.ERR_INVALID_ARG
    # dequantize: MXFP8 takes no FP32 scale, bad dtype
    assert lib.dequantize(0, p, p, p, 1, None, 0, 4, 32, 0, p, None) == m.ERR_INVALID_ARG
    assert lib.dequantize(1, p, p, None, 0, None, 0, 4, 32, 5, p, None) == m.ERR_INVALID_ARG
    # MXFP4: blocks of 32, no FP32 scale; unknown format
    assert lib.dequantize(2, p, p, None, 0, None, 0, 4, 16, 0, p, None) == m.ERR_INVALID_ARG
    assert lib.dequantize(2, p, p, p, 2, None, 0, 4, 32, 0, p, None) == m.ERR_INVALID_ARG
    assert lib.dequantize(3, p, p, None, 0, None, 0, 4, 32, 0, p, None) == m.ERR_INVALID_ARG
    # BF16 GEMM: K % 8, lda < K, misaligned stride, accumulate into bf16, empty
    assert lib.bf16_gemm(8, 8, 12, p, 16, p, 16, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bf16_gemm(8, 8, 64, p, 32, p, 64, 0, p, 8, 0, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.bf16_gemm(8, 8, 64, p, 68, p, 64, 0, p, 8, 0, p, 4096, None) == m.ERR_ALIGNMENT
    assert lib.bf16_gemm(8, 8, 64, p, 64, p, 64, 1, p, 8, 1, p, 4096, None) == m.ERR_UNSUPPORTED
    assert lib.bf16_gemm(0, 8, 64, None, 64, None, 64, 0, None, 8, 0, None, 0, None) == m.OK
    # quantize before dispatch: topk range, missing offsets, cols % 16
    assert lib.nvfp4_quantize_dispatch(p, 4, 32, 32, p, 0, p, 2, 1, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_dispatch(p, 4, 32, 32, p, 17, p, 2, 1, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_dispatch(p, 4, 32, 32, p, 2, None, 2, 1, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_dispatch(p, 4, 24, 24, p, 2, p, 2, 1, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_dispatch(p, 4, 32, 32, p, 2, p, 2, 7, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    # 2-D block-scaled NVFP4: rows and cols % 32, flags
    assert lib.nvfp4_quantize_2d(p, 48, 64, 64, 3, p, p, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_2d(p, 64, 48, 48, 3, p, p, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_2d(p, 64, 64, 64, 0, p, p, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_2d(p, 64, 64, 64, 3, p, p, p, p, None, p, 4096, None) == m.ERR_INVALID_ARG
    # RHT columnwise: rows % 32, cols % 8, a sign mask of 16 bits
    assert lib.nvfp4_quantize_rht_colwise(p, 48, 64, 64, 0, 0, 0, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_rht_colwise(p, 64, 12, 12, 0, 0, 0, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_rht_colwise(p, 64, 64, 64, 0x10000, 0, 0, p, p, p, p, 4096, None) == m.ERR_INVALID_ARG
    # stochastic per-token: cols % 16, misaligned stride
    assert lib.nvfp4_quantize_per_token_sr(p, 4, 24, 24, 1, p, p, p, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token_sr(p, 4, 32, 36, 1, p, p, p, None) == m.ERR_ALIGNMENT
    # MoE combine: hidden % 8, topk range, bad dtype
    assert lib.mx8_moe_combine(p, 8, 12, p, p, 4, 12, 2, 1, p, 12, None) == m.ERR_INVALID_ARG
    assert lib.mx8_moe_combine(p, 8, 16, p, p, 4, 16, 0, 1, p, 16, None) == m.ERR_INVALID_ARG
    assert lib.mx8_moe_combine(p, 8, 16, p, p, 4, 16, 2, 7, p, 16, None) == m.ERR_INVALID_ARG
    # fused MoE GEMM: bad epilogue, SwiGLU needs N % 256 and bf16, formats other than NVFP4
    assert lib.bs_grouped_gemm_fused(1, 2, p, 8, 256, 64, p, p, None, None, 0, p, p, None, 5, 1, p, 128, p, 4096,
                                     None) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_fused(1, 2, p, 8, 384, 64, p, p, None, None, 0, p, p, None, 1, 1, p, 192, p, 4096,
                                     None) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_fused(1, 2, p, 8, 256, 64, p, p, None, None, 0, p, p, None, 1, 0, p, 128, p, 4096,
                                     None) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_fused(1, 2, p, 8, 256, 64, p, p, None, p, 0, p, p, None, 0, 1, p, 256, p, 4096,
                                     None) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_fused(0, 2, p, 8, 256, 64, p, p, None, None, 0, p, p, None, 0, 1, p, 256, p, 4096,
                                     None) == m.ERR_UNSUPPORTED
    # empty problems are no-ops
    assert lib.mx8_quantize(None, 0, 64, 64, m.ROWWISE, None, None, None, None, None, 0, None) == m.OK
    assert lib.bs_gemm(0, 0, 8, 64, None, None, None, 0, None, None, None, 0, 0, None, 8, 0, None, 0, None) == m.OK


def test_status_strings(lib):
    import moe_mx8_quantize_gb300 as m
    for s in range(7):
        assert m.status_string(s)
    assert m.status_string(m.ERR_TIMEOUT) == "a bounded device wait ran out"


def test_quantize_batch_rejects_bad_counts(lib):
    import moe_mx8_quantize_gb300 as m
    items = (m.QuantizeItem * 5)()
    for n in (0, 5, -1):
        assert lib.mx8_quantize_batch(m.FMT_MXFP8, ctypes.cast(items, ctypes.c_void_p), n, m.ROWWISE, None, 0,
                                      None) == m.ERR_INVALID_ARG
    assert lib.mx8_quantize_batch(m.FMT_NVFP4, ctypes.cast(items, ctypes.c_void_p), 1, m.ROWWISE, None, 0,
                                  None) == m.ERR_INVALID_ARG
    # one item with cols % 32 != 0 fails the whole call before any launch
    items[0] = m.QuantizeItem(16, 64, 48, 48, 16, 16, None, None)
    assert lib.mx8_quantize_batch(m.FMT_MXFP8, ctypes.cast(items, ctypes.c_void_p), 1, m.ROWWISE, None, 0,
                                  None) == m.ERR_INVALID_ARG


def test_fused_swiglu_noalloc_and_selftest_arguments_rejected_on_host(lib):
    """The entries the other host checks do not reach: argument errors come
    back before any device work (no GPU in this process)."""
    import moe_mx8_quantize_gb300 as m
    p = ctypes.c_void_p(16)      # never dereferenced
    odd = ctypes.c_void_p(18)    # not 4-byte aligned
    # SwiGLU: ffn % 8, ld_gate_up < 2 ffn, ld_h < ffn, misaligned, empty
    assert lib.mx8_swiglu(p, 4, 12, 24, p, 12, None) == m.ERR_INVALID_ARG
    assert lib.mx8_swiglu(p, 4, 64, 96, p, 64, None) == m.ERR_INVALID_ARG
    assert lib.mx8_swiglu(p, 4, 64, 128, p, 32, None) == m.ERR_INVALID_ARG
    assert lib.mx8_swiglu(odd, 4, 64, 128, p, 64, None) == m.ERR_ALIGNMENT
    assert lib.mx8_swiglu(None, 0, 64, 128, None, 64, None) == m.OK
    # gate|up GEMM with h quantized: group count, N % 256, F / 128 above the
    # cluster limit, K % 32, missing outputs, misaligned S_dec, no workspace
    args = lambda G, N, K, qh=p, s32=p, ws=p, wsb=1 << 20: (G, p, 256, N, K, p, p, None, p, p, None, qh, p, s32,
                                                            None, 0, ws, wsb, None)
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(0, 512, 64)) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(2, 384, 64)) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(2, 2304, 64)) == m.ERR_UNSUPPORTED
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(2, 512, 48)) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(2, 512, 64, qh=None)) == m.ERR_INVALID_ARG
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(2, 512, 64, s32=odd)) == m.ERR_ALIGNMENT
    assert lib.bs_grouped_gemm_swiglu_nvfp4(*args(2, 512, 64, ws=None, wsb=0)) == m.ERR_WORKSPACE
    # the no-allocation quantizer: scope, cols % 16, group scope without
    # offsets, group count, misaligned, empty
    assert lib.nvfp4_quantize_per_token_noalloc(p, 4, 32, 32, 7, None, 0, p, p, p, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token_noalloc(p, 4, 24, 24, 0, None, 0, p, p, p, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token_noalloc(p, 4, 32, 32, 1, None, 0, p, p, p, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token_noalloc(p, 4, 32, 32, 1, p, 0, p, p, p, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token_noalloc(odd, 4, 32, 32, 0, None, 0, p, p, p, None) == m.ERR_ALIGNMENT
    assert lib.nvfp4_quantize_per_token_noalloc(None, 0, 0, 0, 0, None, 0, None, None, None, None) == m.OK
    # the bounded-wait self test: workspace, wait limit
    assert lib.mx8_selftest_bounded_wait(None, 1000, None) == m.ERR_WORKSPACE
    assert lib.mx8_selftest_bounded_wait(p, 0, None) == m.ERR_INVALID_ARG
    assert lib.mx8_selftest_bounded_wait(p, 3000000000, None) == m.ERR_INVALID_ARG
