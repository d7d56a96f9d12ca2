"""GPU parity of the quantizers and the dequantizer against the CPU oracle:
bit-exact codes, scales (every byte of the tensor-core tile buffers, padding
included) and FP32 decode scales, on the workloads' shapes, ragged tails and
edge-case inputs."""
import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import dev, ensure_built, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _mx8_check(xb, flags=mx.ROWWISE | mx.COLWISE):
    x = dev(xb)
    q_row, s_row, q_col, s_col = mx.mx8_quantize(x, flags)
    torch.cuda.synchronize()
    R, C = xb.shape
    if flags & mx.ROWWISE:
        q, s = oracle.mxfp8_quantize_rowwise(xb)
        assert np.array_equal(host(q_row), q), "rowwise codes"
        sw = oracle.swizzle_scales(s)
        assert np.array_equal(host(s_row)[: sw.size], sw), "rowwise scales"
    if flags & mx.COLWISE:
        qT, sT = oracle.mxfp8_quantize_colwise(xb)
        assert np.array_equal(host(q_col), qT), "colwise codes"
        sw = oracle.swizzle_scales(sT)
        assert np.array_equal(host(s_col)[: sw.size], sw), "colwise scales"


def test_mxfp8_pr1():
    d = inputs.pr1()
    _mx8_check(inputs.bits(d["X"]))
    _mx8_check(inputs.bits(d["W"]))


@pytest.mark.parametrize("shape,flags", [
    ((96, 160), mx.ROWWISE | mx.COLWISE),     # ragged rows and columns of the 128x128 tile
    ((32, 32), mx.ROWWISE | mx.COLWISE),
    ((1, 32), mx.ROWWISE),
    ((200, 96), mx.ROWWISE),
    ((33, 4096), mx.ROWWISE),
    ((256, 544), mx.COLWISE),
    ((640, 384), mx.ROWWISE | mx.COLWISE),
])
def test_mxfp8_ragged_and_sweep_mix(shape, flags):
    _mx8_check(inputs.bits(inputs.sweep(*shape, seed=11 + shape[0])), flags)


def test_mxfp8_edge_values():
    xb = np.zeros((64, 64), np.uint16)
    xb[0, 0] = 0x7F7F           # +bf16 max
    xb[1, 5] = 0xFF7F           # -bf16 max
    xb[2, :] = 0x0001           # smallest subnormal
    xb[3, 7] = 0x8000           # -0
    xb[4, 3] = 0x8001           # negative subnormal
    xb[5, :32] = 0x3F80         # all equal blocks (1.0)
    xb[6, 32:] = 0xC3E0         # -448
    _mx8_check(xb)


def test_mxfp8_linear_full_size():
    d = inputs.linear(device="cuda")
    for name in ("X", "W", "dY"):
        _mx8_check(inputs.bits(d[name]))


def test_mxfp8_strided_input():
    xb = inputs.bits(inputs.sweep(128, 256, seed=3))
    big = torch.zeros((128, 320), dtype=torch.bfloat16, device="cuda")
    big[:, :256] = dev(xb)
    view = big[:, :256]
    q_row, s_row, q_col, s_col = mx.mx8_quantize(view)
    q, s = oracle.mxfp8_quantize_rowwise(xb)
    assert np.array_equal(host(q_row), q)
    qT, _ = oracle.mxfp8_quantize_colwise(xb)
    assert np.array_equal(host(q_col), qT)


def test_mxfp8_empty():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    mx.mx8_quantize(x, mx.ROWWISE)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ NVFP4
def _nv_check(xb, scope=mx.SCOPE_TOKEN, offs=None):
    x = dev(xb)
    go = None if offs is None else torch.tensor(offs, dtype=torch.int64, device="cuda")
    q, s, s32 = mx.nvfp4_quantize_per_token(x, scope, go)
    torch.cuda.synchronize()
    oq, os_, o32 = oracle.nvfp4_quantize(xb, scope, offs)
    assert np.array_equal(host(q), oq), "codes"
    assert np.array_equal(host(s32).view(np.uint32), o32.view(np.uint32)), "fp32 scales"
    sw = oracle.swizzle_scales(os_, offs)
    assert np.array_equal(host(s)[: sw.size], sw), "block scales"
    return q, s, s32


def test_nvfp4_pr1():
    d = inputs.pr1()
    _nv_check(inputs.bits(d["X"]))
    _nv_check(inputs.bits(d["W"]), mx.SCOPE_TENSOR)


@pytest.mark.parametrize("shape", [(5, 16), (7, 48), (130, 80), (64, 208), (300, 768), (9, 4096), (33, 7168), (5, 8448),
                                   (7, 256), (131, 768), (1, 768)])
def test_nvfp4_ragged(shape):
    rows, cols = shape
    wide = inputs.sweep(rows, (cols + 31) // 32 * 32, seed=rows)
    _nv_check(inputs.bits(wide[:, :cols]))


def test_nvfp4_edge_values():
    xb = np.zeros((8, 64), np.uint16)
    xb[1, 3] = 0x0001
    xb[1, 9] = 0x8001
    xb[2, :] = 0x7F7F
    xb[3, ::2] = 0xFF7F
    xb[4, 5] = 0x8000
    xb[5, :] = 0x3F80
    xb[6, 0] = 0x4528           # 2688
    xb[6, 1:16] = 0x4100        # 8
    xb[7, :16] = 0x0080         # smallest normal bf16 (2^-126)
    _nv_check(xb)
    _nv_check(xb, mx.SCOPE_TENSOR)


def test_nvfp4_qwen_activation_full_size():
    d = inputs.qwen_moe(device="cuda", with_weights=False)
    _nv_check(inputs.bits(d["X"]))


def test_nvfp4_group_scope_and_grouped_layout():
    xb = inputs.bits(inputs.sweep(700, 256, seed=21))
    offs = [0, 130, 130, 131, 400, 700]
    _nv_check(xb, mx.SCOPE_GROUP, offs)
    _nv_check(xb, mx.SCOPE_TOKEN, offs)
    _nv_check(xb, mx.SCOPE_TENSOR, offs)


def test_nvfp4_expert_weights_group_scope():
    # gate|up of 4 experts stored jointly [E*2F, H], one FP32 scale per expert
    d = inputs.qwen_moe(with_weights=True, tokens=8, hidden=256, experts=4, ffn=96)
    W = inputs.bits(d["W_gu"]).reshape(4 * 192, 256)
    _nv_check(W, mx.SCOPE_GROUP, [0, 192, 384, 576, 768])


def test_nvfp4_group_scope_interleaved_work_order():
    """24 experts of Qwen3-30B-A3B gate|up shape ([1536, 2048] bf16, 6 MB each):
    enough data that the fused group-scope kernel interleaves the amax work of
    later experts with the encode work of earlier ones."""
    g = torch.Generator(device="cuda").manual_seed(17)
    W = inputs.normal_bf16((24 * 1536, 2048), 0.02, g, "cuda", 0.001, 30.0)
    _nv_check(inputs.bits(W), mx.SCOPE_GROUP, list(range(0, 24 * 1536 + 1, 1536)))


@pytest.mark.parametrize("cols", [256, 768])
def test_nvfp4_paired_rows_group_and_token_scopes(cols):
    """Rows of 256 or 768 columns are encoded two per warp: group scope over
    ragged groups (odd sizes, empty groups, groups ending inside a row pair)
    and token scope with the grouped layout, bit-exact."""
    xb = inputs.bits(inputs.sweep(517, cols, seed=cols))
    offs = [0, 3, 3, 130, 257, 258, 517]
    _nv_check(xb, mx.SCOPE_GROUP, offs)
    _nv_check(xb, mx.SCOPE_TOKEN, offs)
    _nv_check(xb, mx.SCOPE_TENSOR)
    W = inputs.bits(inputs.normal_bf16((8 * 256, cols), 0.02, torch.Generator().manual_seed(cols), "cpu"))
    _nv_check(W, mx.SCOPE_GROUP, list(range(0, 8 * 256 + 1, 256)))


def test_nvfp4_group_scope_one_large_group():
    """One group of 8192 x 2048 bf16 (32 MB) among small ones: its amax items
    span many blocks before any of its encode items can run."""
    g = torch.Generator(device="cuda").manual_seed(19)
    W = inputs.normal_bf16((8192 + 300, 2048), 0.02, g, "cuda", 0.001, 30.0)
    _nv_check(inputs.bits(W), mx.SCOPE_GROUP, [0, 100, 100, 8292, 8492])


def test_nvfp4_group_scope_ragged_groups_resident():
    """Ragged groups (empty, one row, 129 rows, several chunks) with columns
    that are not a multiple of 512: the resident kernel's chunking, its
    padding scale rows and the empty groups' zero decode scales."""
    xb = inputs.bits(inputs.sweep(1200, 800, seed=23))
    _nv_check(xb, mx.SCOPE_GROUP, [0, 0, 1, 130, 130, 700, 1200])
    _nv_check(xb[:300], mx.SCOPE_TENSOR)


@pytest.mark.parametrize("cols", [2560, 7168, 9216])
def test_nvfp4_group_scope_long_rows(cols):
    """Rows longer than 2048 values (the DeepSeek-V3 hidden size among them)
    are streamed four 512-value chunks at a time: ragged groups, a tail chunk
    shorter than 512, empty groups and tensor scope, bit-exact."""
    xb = inputs.bits(inputs.sweep(260, cols, seed=cols))
    _nv_check(xb, mx.SCOPE_GROUP, [0, 1, 1, 129, 200, 260])
    _nv_check(xb, mx.SCOPE_TENSOR)


def test_nvfp4_tensor_scope_large():
    g = torch.Generator(device="cuda").manual_seed(18)
    W = inputs.normal_bf16((8192, 2048), 0.02, g, "cuda")
    _nv_check(inputs.bits(W), mx.SCOPE_TENSOR)


def test_nvfp4_per_token_batch_invariance_on_gpu():
    xb = inputs.bits(inputs.qwen_moe(with_weights=False, tokens=256, hidden=512)["X"])
    qa, sa, s32a = mx.nvfp4_quantize_per_token(dev(xb))
    perm = np.random.default_rng(1).permutation(256)[:100]
    qb, sb, s32b = mx.nvfp4_quantize_per_token(dev(xb[perm]))
    assert np.array_equal(host(qa)[perm], host(qb))
    assert np.array_equal(host(s32a)[perm], host(s32b))


# ------------------------------------------------------------------ dequantize
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_dequant_mxfp8(out_dtype):
    xb = inputs.bits(inputs.sweep(160, 320, seed=31))
    q, s = oracle.mxfp8_quantize_rowwise(xb)
    ref = oracle.dequant_mxfp8(q, s)
    out = mx.dequantize(mx.FMT_MXFP8, dev(q), dev(oracle.swizzle_scales(s)), out_dtype=out_dtype)
    got = host(out)
    if out_dtype == torch.float32:
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(got, oracle.f32_to_bf16(ref))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_dequant_nvfp4(out_dtype):
    xb = inputs.bits(inputs.pr1()["X"])
    q, s, s32 = oracle.nvfp4_quantize(xb)
    ref = oracle.dequant_nvfp4(q, s, s32, oracle.S32_ROW)
    out = mx.dequantize(mx.FMT_NVFP4, dev(q), dev(oracle.swizzle_scales(s)), dev(s32), out_dtype=out_dtype)
    got = host(out)
    if out_dtype == torch.float32:
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(got, oracle.f32_to_bf16(ref))


def test_dequant_nvfp4_grouped_group_scale():
    xb = inputs.bits(inputs.sweep(300, 128, seed=41))
    offs = [0, 100, 100, 300]
    q, s, s32 = oracle.nvfp4_quantize(xb, oracle.SCOPE_GROUP, offs)
    ref = oracle.dequant_nvfp4(q, s, s32, oracle.S32_GROUP, offs)
    go = torch.tensor(offs, dtype=torch.int64, device="cuda")
    out = mx.dequantize(mx.FMT_NVFP4, dev(q), dev(oracle.swizzle_scales(s, offs)), dev(s32),
                        s32_mode=mx.S32_GROUP, group_offsets=go)
    assert np.array_equal(host(out).view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ bounded waits
def test_bounded_wait_times_out_and_reports():
    ws = mx.new_workspace()
    assert mx.check_device_error(ws) == mx.OK
    mx.selftest_bounded_wait(ws, 5_000_000)        # 5 ms
    assert mx.check_device_error(ws) == mx.ERR_TIMEOUT
    assert mx.check_device_error(ws) == mx.OK      # cleared
    # the context is still usable
    x = torch.ones((32, 32), dtype=torch.bfloat16, device="cuda")
    q, s, _, _ = mx.mx8_quantize(x, mx.ROWWISE, ws=ws)
    oq, _ = oracle.mxfp8_quantize_rowwise(host(x))
    assert np.array_equal(host(q), oq)
    assert mx.check_device_error(ws) == mx.OK


# ------------------------------------------------------------------ SwiGLU
def _bf16_ulps(a, b):
    def ordered(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def test_swiglu_within_one_bf16_unit_of_oracle():
    """silu uses CUDA's expf in FP32; the oracle evaluates in double.  Both
    round to bf16 once, so results agree to one bf16 unit and almost always
    exactly."""
    g = torch.Generator().manual_seed(5)
    gu = inputs.bits(inputs.normal_bf16((512, 2 * 768), 2.0, g, "cpu", 0.01, 20.0))
    got = host(mx.swiglu(dev(gu)))
    ref = oracle.swiglu(gu)
    ulps = _bf16_ulps(got, ref)
    assert ulps.max() <= 1
    assert (ulps == 0).mean() >= 0.999


def _alloc_copies(fmt, R, C, flags):
    """Output buffers of one rowwise / columnwise quantization (zeroed, so
    every byte the kernel must write is compared)."""
    packed = fmt == mx.FMT_MXFP4
    z = lambda n: torch.zeros(max(n, 16), dtype=torch.uint8, device="cuda")
    qr = z(R * C // (2 if packed else 1)) if flags & mx.ROWWISE else None
    sr = z(mx.scale_bytes(fmt, R, C)) if flags & mx.ROWWISE else None
    qc = z(R * C // (2 if packed else 1)) if flags & mx.COLWISE else None
    sc = z(mx.scale_bytes(fmt, C, R)) if flags & mx.COLWISE else None
    return qr, sr, qc, sc


@pytest.mark.parametrize("fmt", [mx.FMT_MXFP8, mx.FMT_MXFP4])
@pytest.mark.parametrize("flags", [mx.ROWWISE | mx.COLWISE, mx.ROWWISE, mx.COLWISE])
def test_quantize_batch_equals_separate_calls(fmt, flags):
    """One launch over the X, W and dY of the 2048 x 2048 -> 8192 linear layer
    plus a ragged 96 x 160 tensor (partial 128 x 128 tiles): every output byte
    equals the separate single-tensor calls; the ragged tensor also against
    the oracle."""
    lin = inputs.linear(seed=1, device="cuda")
    rag = inputs.sweep(96, 160, seed=21, device="cuda")
    xs = [lin["X"], lin["W"], lin["dY"], rag]
    batch = [(x, *_alloc_copies(fmt, *x.shape, flags)) for x in xs]
    one = [(x, *_alloc_copies(fmt, *x.shape, flags)) for x in xs]
    mx.mx8_quantize_batch_into(fmt, batch, flags)
    single = mx.mx8_quantize_into if fmt == mx.FMT_MXFP8 else mx.mxfp4_quantize_into
    for x, qr, sr, qc, sc in one:
        single(x, qr, sr, qc, sc, flags)
    torch.cuda.synchronize()
    for b, o in zip(batch, one):
        for tb, to in zip(b[1:], o[1:]):
            if tb is not None:
                assert torch.equal(tb, to)
    xb = inputs.bits(rag)
    x, qr, sr, qc, sc = batch[3]
    if fmt == mx.FMT_MXFP8:
        rq, rs = oracle.mxfp8_quantize_rowwise(xb)
        cq, cs = oracle.mxfp8_quantize_colwise(xb)
    else:
        rq, rs = oracle.mxfp4_quantize_rowwise(xb)
        cq, cs = oracle.mxfp4_quantize_colwise(xb)
    if flags & mx.ROWWISE:
        assert np.array_equal(host(qr)[: rq.size], rq.ravel())
        sw = oracle.swizzle_scales(rs)
        assert np.array_equal(host(sr)[: sw.size], sw)
    if flags & mx.COLWISE:
        assert np.array_equal(host(qc)[: cq.size], cq.ravel())
        sw = oracle.swizzle_scales(cs)
        assert np.array_equal(host(sc)[: sw.size], sw)


def test_quantize_batch_skips_empty_items():
    x = inputs.sweep(64, 96, seed=3, device="cuda")
    empty = torch.empty((0, 96), dtype=torch.bfloat16, device="cuda")
    a = _alloc_copies(mx.FMT_MXFP8, 64, 96, mx.ROWWISE | mx.COLWISE)
    mx.mx8_quantize_batch_into(mx.FMT_MXFP8, [(empty, None, None, None, None), (x, *a)])
    q, s = oracle.mxfp8_quantize_rowwise(inputs.bits(x))
    torch.cuda.synchronize()
    assert np.array_equal(host(a[0])[: q.size], q.ravel())
