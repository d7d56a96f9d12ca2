"""The allocation-free NVFP4 quantizer entry point (for callers that cannot
allocate device memory, so cannot hand the library a workspace) must give the
same bytes as the regular entry point.  Called twice in a row through the C
ABI with different data, so amax scratch left over from the first call would
show up in the second.  Kept in a file that runs last."""
import ctypes

import numpy as np
import pytest
import torch

import moe_mx8_quantize_gb300 as mx
from moe_mx8_quantize_gb300 import inputs
from tests._lib import ensure_built

pytestmark = pytest.mark.gpu


def _outputs(R, C, scope, G):
    dev = "cuda"
    q = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
    sb = torch.zeros(mx.scale_bytes_grouped(mx.FMT_NVFP4, R, G, C), dtype=torch.uint8, device=dev)
    n32 = R if scope == mx.SCOPE_TOKEN else (G if scope == mx.SCOPE_GROUP else 1)
    s32 = torch.empty(n32, dtype=torch.float32, device=dev)
    return q, sb, s32


def _call_noalloc(lib, x, scope, offs, q, sb, s32):
    R, C = x.shape
    G = offs.numel() - 1
    st = lib.nvfp4_quantize_per_token_noalloc(
        ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), scope, ctypes.c_void_p(offs.data_ptr()), G,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(s32.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mx.OK, mx.status_string(st)


def _call_regular(lib, x, scope, offs, q, sb, s32):
    R, C = x.shape
    G = offs.numel() - 1
    ws = mx.new_workspace(G)
    st = lib.nvfp4_quantize_per_token(
        ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), scope, ctypes.c_void_p(offs.data_ptr()), G,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(s32.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mx.OK, mx.status_string(st)


@pytest.mark.parametrize("scope", [mx.SCOPE_GROUP, mx.SCOPE_TENSOR])
def test_noalloc_matches_regular_entry_point_twice(scope):
    ensure_built()
    lib = mx.load()
    offs = torch.tensor([0, 100, 100, 357, 512], dtype=torch.int64, device="cuda")
    G = offs.numel() - 1
    # two calls in a row; the first sees much larger values than the second
    xs = [inputs.normal_bf16((512, 768), 50.0, torch.Generator().manual_seed(1), "cpu").cuda(),
          inputs.normal_bf16((512, 768), 0.5, torch.Generator().manual_seed(2), "cpu").cuda()]
    for x in xs:
        got = _outputs(512, 768, scope, G)
        want = _outputs(512, 768, scope, G)
        _call_noalloc(lib, x, scope, offs, *got)
        _call_regular(lib, x, scope, offs, *want)
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a.cpu().view(torch.uint8).reshape(-1), b.cpu().view(torch.uint8).reshape(-1))


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
