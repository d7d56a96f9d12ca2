"""The allocation-free NVFP4 quantizer entry point, for callers that cannot
allocate device memory (code running inside a host application that owns
every allocation), so cannot hand the library a workspace: its scratch is a
fixed array inside the library.  Every case is called twice in a row through
the C ABI with different data (amax scratch left over from the first call
would show in the second) and compared byte for byte with the oracle and with
the regular entry point.  Cases: group scope with ragged and empty groups,
1024 groups (the array's limit; most of them empty), tensor scope on a small
tensor (amax launch + token kernel) and on one over 64 MB (the ticket
kernel, which uses the array's amax, count and ticket words), and token
scope.  Kept in a file that runs last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import ensure_built, host

pytestmark = pytest.mark.gpu


def _outputs(R, C, scope, G):
    dev = "cuda"
    q = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
    sb = torch.zeros(mx.scale_bytes_grouped(mx.FMT_NVFP4, R, G, C), dtype=torch.uint8, device=dev)
    n32 = R if scope == mx.SCOPE_TOKEN else (G if scope == mx.SCOPE_GROUP else 1)
    s32 = torch.empty(n32, dtype=torch.float32, device=dev)
    return q, sb, s32


def _offs_args(offs):
    return (ctypes.c_void_p(offs.data_ptr()), offs.numel() - 1) if offs is not None else (None, 0)


def _call_noalloc(lib, x, scope, offs, q, sb, s32):
    R, C = x.shape
    st = lib.nvfp4_quantize_per_token_noalloc(
        ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), scope, *_offs_args(offs),
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(s32.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mx.OK, mx.status_string(st)


def _call_regular(lib, x, scope, offs, q, sb, s32):
    R, C = x.shape
    ws = mx.new_workspace(offs.numel() - 1 if offs is not None else 1)
    st = lib.nvfp4_quantize_per_token(
        ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), scope, *_offs_args(offs),
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(s32.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mx.OK, mx.status_string(st)


def _oracle(xb, scope, offs_np):
    q, s, s32 = oracle.nvfp4_quantize(xb, scope, offs_np)
    return q, oracle.swizzle_scales(s, offs_np), s32


def _run_twice(lib, shape, stds, scope, offs_np, seed):
    ensure_built()
    offs = torch.tensor(offs_np, dtype=torch.int64, device="cuda") if offs_np is not None else None
    G = len(offs_np) - 1 if offs_np is not None else 1
    R, C = shape
    # two calls in a row; the first sees much larger values than the second
    for i, std in enumerate(stds):
        x = inputs.normal_bf16(shape, std, torch.Generator(device="cuda").manual_seed(seed + i), "cuda",
                               0.001, 40.0)
        got = _outputs(R, C, scope, G)
        want = _outputs(R, C, scope, G)
        _call_noalloc(lib, x, scope, offs, *got)
        _call_regular(lib, x, scope, offs, *want)
        torch.cuda.synchronize()
        assert lib.nvfp4_noalloc_check_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == mx.OK
        for a, b in zip(got, want):
            assert torch.equal(a.view(torch.uint8).reshape(-1), b.view(torch.uint8).reshape(-1))
        oq, os_, o32 = _oracle(inputs.bits(x), scope, offs_np)
        assert np.array_equal(host(got[0]), oq)
        assert np.array_equal(host(got[1])[: os_.size], os_)
        assert np.array_equal(host(got[2]).view(np.uint32), o32.view(np.uint32))


@pytest.mark.parametrize("scope", [mx.SCOPE_GROUP, mx.SCOPE_TENSOR, mx.SCOPE_TOKEN])
def test_noalloc_ragged_groups_twice(scope):
    _run_twice(mx.load(), (512, 768), (50.0, 0.5), scope, np.array([0, 100, 100, 357, 512]), 1)


def test_noalloc_1024_groups_twice():
    """The largest group count the array serves: 1024 groups over 600 rows,
    most of them empty (their decode scale is zero)."""
    rng = np.random.default_rng(3)
    offs = np.concatenate([[0], np.sort(rng.integers(0, 601, 1023)), [600]]).astype(np.int64)
    _run_twice(mx.load(), (600, 256), (3.0, 0.01), mx.SCOPE_GROUP, offs, 5)


def test_noalloc_large_tensor_scope_twice():
    """Tensor scope on a 16384 x 2176 bf16 tensor (71 MB, above the size the
    amax launch + token kernel path takes), so the ticket kernel runs on the
    array's amax, count and ticket words."""
    _run_twice(mx.load(), (16384, 2176), (2.0, 0.03), mx.SCOPE_TENSOR, None, 9)


def test_noalloc_rejects_too_many_groups():
    ensure_built()
    lib = mx.load()
    offs = torch.zeros(1026, dtype=torch.int64, device="cuda")    # 1025 groups
    x = torch.zeros((16, 32), dtype=torch.bfloat16, device="cuda")
    q, sb, s32 = _outputs(16, 32, mx.SCOPE_GROUP, 1025)
    st = lib.nvfp4_quantize_per_token_noalloc(
        ctypes.c_void_p(x.data_ptr()), 16, 32, 32, mx.SCOPE_GROUP, ctypes.c_void_p(offs.data_ptr()), 1025,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(s32.data_ptr()), None)
    assert st == mx.ERR_INVALID_ARG
