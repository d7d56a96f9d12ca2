"""GB300-native microscaling quantization (MXFP8, per-token NVFP4, MXFP4) and the
block-scaled tcgen05 GEMM it feeds.

This package is a thin ctypes binding over the C ABI of ``_build/libmx8q.so``
(declared in ``include/mx8q.h``): it marshals torch tensors into device
pointers, sizes and the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no CPU fallback.  Importing the
package does not load the library; the first call does, and raises if the
library has not been built (``python -m moe_mx8_quantize_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmx8q.so")

# ---------------------------------------------------------------- constants
OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(7)
ROWWISE, COLWISE = 1, 2
SCOPE_TOKEN, SCOPE_GROUP, SCOPE_TENSOR = 0, 1, 2
FMT_MXFP8, FMT_NVFP4, FMT_MXFP4 = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1
EPI_NONE, EPI_SWIGLU = 0, 1
DISPATCH_TOKENS, DISPATCH_ROWS = 0, 1
S32_NONE, S32_ROW, S32_TENSOR, S32_GROUP = 0, 1, 2, 3

# every C symbol the header declares
EXPORTS = ("mx8_scale_bytes", "mx8_scale_bytes_grouped", "mx8_workspace_bytes",
           "mx8_device_sm_count", "mx8_quantize", "mxfp4_quantize", "mx8_quantize_batch", "nvfp4_quantize_per_token",
           "nvfp4_quantize_dispatch", "nvfp4_quantize_2d", "nvfp4_quantize_rht_colwise",
           "nvfp4_quantize_per_token_sr",
           "nvfp4_quantize_per_token_noalloc", "nvfp4_noalloc_check_error", "dequantize",
           "bs_gemm", "bs_grouped_gemm", "bs_grouped_gemm_fused", "bs_grouped_gemm_swiglu_nvfp4", "bf16_gemm", "mx8_moe_combine", "mx8_swiglu", "mx8_check_device_error", "mx8_selftest_bounded_wait",
           "mx8_status_string")


class Mx8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i = ctypes.c_int
_sz = ctypes.c_size_t


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the CUDA library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"mx8q CUDA library not built: {path} is missing "
                           "(run python -m moe_mx8_quantize_gb300.build)")
    lib = ctypes.CDLL(path)
    lib.mx8_scale_bytes.restype = _sz
    lib.mx8_scale_bytes.argtypes = [_i, _i64, _i64]
    lib.mx8_scale_bytes_grouped.restype = _sz
    lib.mx8_scale_bytes_grouped.argtypes = [_i, _i64, _i, _i64]
    lib.mx8_workspace_bytes.restype = _sz
    lib.mx8_workspace_bytes.argtypes = [_i]
    lib.mx8_device_sm_count.restype = _i
    lib.mx8_device_sm_count.argtypes = []
    lib.mx8_quantize.restype = _i
    lib.mx8_quantize.argtypes = [_p, _i64, _i64, _i64, _i, _p, _p, _p, _p, _p, _sz, _p]
    lib.mx8_quantize_batch.restype = _i
    lib.mx8_quantize_batch.argtypes = [_i, _p, _i, _i, _p, _sz, _p]
    lib.mxfp4_quantize.restype = _i
    lib.mxfp4_quantize.argtypes = [_p, _i64, _i64, _i64, _i, _p, _p, _p, _p, _p, _sz, _p]
    lib.nvfp4_quantize_per_token.restype = _i
    lib.nvfp4_quantize_per_token.argtypes = [_p, _i64, _i64, _i64, _i, _p, _i, _p, _p, _p, _p, _sz, _p]
    lib.nvfp4_quantize_per_token_noalloc.restype = _i
    lib.nvfp4_quantize_per_token_noalloc.argtypes = [_p, _i64, _i64, _i64, _i, _p, _i, _p, _p, _p, _p]
    lib.nvfp4_noalloc_check_error.restype = _i
    lib.nvfp4_noalloc_check_error.argtypes = [_p]
    lib.dequantize.restype = _i
    lib.dequantize.argtypes = [_i, _p, _p, _p, _i, _p, _i, _i64, _i64, _i, _p, _p]
    lib.bs_gemm.restype = _i
    lib.bs_gemm.argtypes = [_i, _i64, _i64, _i64, _p, _p, _p, _i, _p, _p, _p, _i, _i, _p, _i64, _i,
                            _p, _sz, _p]
    lib.bs_grouped_gemm.restype = _i
    lib.bs_grouped_gemm.argtypes = [_i, _i, _p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _i, _p,
                                    _i64, _p, _sz, _p]
    lib.nvfp4_quantize_dispatch.restype = _i
    lib.nvfp4_quantize_dispatch.argtypes = [_p, _i64, _i64, _i64, _p, _i, _p, _i, _i, _p, _p, _p, _p, _sz, _p]
    lib.nvfp4_quantize_2d.restype = _i
    lib.nvfp4_quantize_2d.argtypes = [_p, _i64, _i64, _i64, _i, _p, _p, _p, _p, _p, _p, _sz, _p]
    lib.nvfp4_quantize_rht_colwise.restype = _i
    lib.nvfp4_quantize_rht_colwise.argtypes = [_p, _i64, _i64, _i64, ctypes.c_uint32, _i, ctypes.c_uint64, _p, _p,
                                               _p, _p, _sz, _p]
    lib.nvfp4_quantize_per_token_sr.restype = _i
    lib.nvfp4_quantize_per_token_sr.argtypes = [_p, _i64, _i64, _i64, ctypes.c_uint64, _p, _p, _p, _p]
    lib.bs_grouped_gemm_fused.restype = _i
    lib.bs_grouped_gemm_fused.argtypes = [_i, _i, _p, _i64, _i64, _i64, _p, _p, _p, _p, _i64, _p, _p, _p, _i,
                                          _i, _p, _i64, _p, _sz, _p]
    lib.bs_grouped_gemm_swiglu_nvfp4.restype = _i
    lib.bs_grouped_gemm_swiglu_nvfp4.argtypes = [_i, _p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                                 _i64, _p, _sz, _p]
    lib.mx8_moe_combine.restype = _i
    lib.mx8_moe_combine.argtypes = [_p, _i64, _i64, _p, _p, _i64, _i64, _i, _i, _p, _i64, _p]
    lib.bf16_gemm.restype = _i
    lib.bf16_gemm.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64, _i, _p, _i64, _i, _p, _sz, _p]
    lib.mx8_swiglu.restype = _i
    lib.mx8_swiglu.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
    lib.mx8_check_device_error.restype = _i
    lib.mx8_check_device_error.argtypes = [_p, _p]
    lib.mx8_selftest_bounded_wait.restype = _i
    lib.mx8_selftest_bounded_wait.argtypes = [_p, ctypes.c_uint64, _p]
    lib.mx8_status_string.restype = ctypes.c_char_p
    lib.mx8_status_string.argtypes = [_i]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().mx8_status_string(status).decode()


def _check(status: int, what: str):
    if status != OK:
        raise Mx8Error(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------- sizes
def scale_bytes(fmt: int, rows: int, cols: int) -> int:
    return int(load().mx8_scale_bytes(fmt, rows, cols))


def scale_bytes_grouped(fmt: int, total_rows: int, num_groups: int, cols: int) -> int:
    return int(load().mx8_scale_bytes_grouped(fmt, total_rows, num_groups, cols))


def workspace_bytes(num_groups: int = 1) -> int:
    return int(load().mx8_workspace_bytes(num_groups))


def new_workspace(num_groups: int = 1, device=None) -> torch.Tensor:
    """Zero-filled workspace (error word + scratch) for calls with up to
    num_groups groups."""
    return torch.zeros(workspace_bytes(num_groups), dtype=torch.uint8, device=device or "cuda")


_default_ws = {}


def _ws(ws, num_groups, device):
    if ws is not None:
        return ws
    key = (device, num_groups)
    w = _default_ws.get(key)
    if w is None or w.numel() < workspace_bytes(num_groups):
        w = new_workspace(num_groups, device)
        _default_ws[key] = w
    return w


def _u8(n, device):
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- MXFP8
def mx8_quantize_into(x, q_row, s_row, q_col, s_col, flags=ROWWISE | COLWISE, ws=None, stream=None):
    """In-place form of :func:`mx8_quantize` (outputs pre-allocated)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    ws = _ws(ws, 1, x.device)
    _check(load().mx8_quantize(_ptr(x), R, C, x.stride(0), flags, _ptr(q_row), _ptr(s_row),
                               _ptr(q_col), _ptr(s_col), _ptr(ws), ws.numel(), _stream(stream)),
           "mx8_quantize")


def mx8_quantize(x: torch.Tensor, flags: int = ROWWISE | COLWISE, ws=None, stream=None):
    """MXFP8 rowwise and/or columnwise quantization of a bf16 [R, C] matrix.

    Returns (q_row [R,C] u8, s_row u8 tiles, q_col [C,R] u8, s_col u8 tiles);
    the copies not requested are None.
    """
    R, C = x.shape
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if flags & ROWWISE:
        q_row = torch.empty((R, C), dtype=torch.uint8, device=dev)
        s_row = _u8(scale_bytes(FMT_MXFP8, R, C), dev)
    if flags & COLWISE:
        q_col = torch.empty((C, R), dtype=torch.uint8, device=dev)
        s_col = _u8(scale_bytes(FMT_MXFP8, C, R), dev)
    mx8_quantize_into(x, q_row, s_row, q_col, s_col, flags, ws, stream)
    return q_row, s_row, q_col, s_col


# ---------------------------------------------------------------- MXFP4
class QuantizeItem(ctypes.Structure):
    """One input of mx8_quantize_batch (the C struct mx8_quantize_item)."""
    _fields_ = [("x", _p), ("rows", _i64), ("cols", _i64), ("ld", _i64),
                ("q_row", _p), ("s_row", _p), ("q_col", _p), ("s_col", _p)]


BATCH_MAX = 4


def mx8_quantize_batch_into(fmt, items, flags=ROWWISE | COLWISE, ws=None, stream=None):
    """MXFP8 (fmt FMT_MXFP8) or MXFP4 (FMT_MXFP4) quantization of up to
    BATCH_MAX tensors in one launch.  items: sequence of (x, q_row, s_row,
    q_col, s_col) with pre-allocated outputs (None for a copy not in flags);
    the bytes equal those of one mx8_quantize_into / mxfp4_quantize_into call
    per tensor."""
    arr = (QuantizeItem * len(items))()
    for i, (x, qr, sr, qc, sc) in enumerate(items):
        assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
        arr[i] = QuantizeItem(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0),
                              *(t.data_ptr() if t is not None else None for t in (qr, sr, qc, sc)))
    ws = _ws(ws, 1, items[0][0].device)
    _check(load().mx8_quantize_batch(fmt, ctypes.cast(arr, _p), len(items), flags, _ptr(ws), ws.numel(),
                                     _stream(stream)), "mx8_quantize_batch")


def mxfp4_quantize_into(x, q_row, s_row, q_col, s_col, flags=ROWWISE | COLWISE, ws=None, stream=None):
    """In-place form of :func:`mxfp4_quantize` (outputs pre-allocated)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    ws = _ws(ws, 1, x.device)
    _check(load().mxfp4_quantize(_ptr(x), R, C, x.stride(0), flags, _ptr(q_row), _ptr(s_row),
                                 _ptr(q_col), _ptr(s_col), _ptr(ws), ws.numel(), _stream(stream)),
           "mxfp4_quantize")


def mxfp4_quantize(x: torch.Tensor, flags: int = ROWWISE | COLWISE, ws=None, stream=None):
    """MXFP4 rowwise and/or columnwise quantization of a bf16 [R, C] matrix.

    Returns (q_row [R,C/2] u8, s_row u8 tiles, q_col [C,R/2] u8, s_col u8
    tiles); the copies not requested are None.
    """
    R, C = x.shape
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if flags & ROWWISE:
        q_row = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
        s_row = _u8(scale_bytes(FMT_MXFP4, R, C), dev)
    if flags & COLWISE:
        q_col = torch.empty((C, R // 2), dtype=torch.uint8, device=dev)
        s_col = _u8(scale_bytes(FMT_MXFP4, C, R), dev)
    mxfp4_quantize_into(x, q_row, s_row, q_col, s_col, flags, ws, stream)
    return q_row, s_row, q_col, s_col


# ---------------------------------------------------------------- NVFP4
def nvfp4_quantize_into(x, q, s_blk, s32, scope=SCOPE_TOKEN, group_offsets=None, ws=None,
                        stream=None):
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    G = 0 if group_offsets is None else group_offsets.numel() - 1
    ws = _ws(ws, max(G, 1), x.device)
    _check(load().nvfp4_quantize_per_token(_ptr(x), R, C, x.stride(0), scope, _ptr(group_offsets), G,
                                           _ptr(q), _ptr(s_blk), _ptr(s32), _ptr(ws), ws.numel(),
                                           _stream(stream)),
           "nvfp4_quantize_per_token")


def nvfp4_quantize_per_token(x: torch.Tensor, scope: int = SCOPE_TOKEN, group_offsets=None,
                             ws=None, stream=None):
    """Two-level NVFP4 quantization with an FP32 scale per token (or group /
    tensor).  Returns (q [R, C/2] u8, s_blk u8 tiles, s32 f32 decode scales).
    group_offsets (device int64 [G+1]) selects the grouped scale layout."""
    R, C = x.shape
    dev = x.device
    G = 0 if group_offsets is None else group_offsets.numel() - 1
    q = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
    if group_offsets is None:
        s_blk = _u8(scale_bytes(FMT_NVFP4, R, C), dev)
    else:
        s_blk = _u8(scale_bytes_grouped(FMT_NVFP4, R, G, C), dev)
    n32 = R if scope == SCOPE_TOKEN else (G if scope == SCOPE_GROUP else 1)
    s32 = torch.empty(max(n32, 1), dtype=torch.float32, device=dev)
    nvfp4_quantize_into(x, q, s_blk, s32, scope, group_offsets, ws, stream)
    return q, s_blk, s32[:n32]


def nvfp4_quantize_dispatch_into(x, dest_rows, topk, group_offsets, q, s_blk, s32, layout=DISPATCH_ROWS,
                                 ws=None, stream=None):
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    T, C = x.shape
    G = group_offsets.numel() - 1
    ws = _ws(ws, G, x.device)
    _check(load().nvfp4_quantize_dispatch(_ptr(x), T, C, x.stride(0), _ptr(dest_rows), topk, _ptr(group_offsets),
                                          G, layout, _ptr(q), _ptr(s_blk), _ptr(s32), _ptr(ws), ws.numel(),
                                          _stream(stream)),
           "nvfp4_quantize_dispatch")


def nvfp4_quantize_dispatch(x, dest_rows, topk, group_offsets, layout=DISPATCH_ROWS, ws=None, stream=None):
    """Per-token NVFP4 of MoE tokens, encoded once before dispatch.  Returns
    (q, s_blk, s32): s_blk holds the dispatched rows' scales in the grouped
    layout; q [rows, C/2] and s32 [rows] are in dispatched-row order
    (DISPATCH_ROWS) or token-major [T, C/2], [T] (DISPATCH_TOKENS)."""
    T, C = x.shape
    G = group_offsets.numel() - 1
    n = T * topk if layout == DISPATCH_ROWS else T
    q = torch.empty((n, C // 2), dtype=torch.uint8, device=x.device)
    s_blk = _u8(scale_bytes_grouped(FMT_NVFP4, T * topk, G, C), x.device)
    s32 = torch.empty(max(n, 1), dtype=torch.float32, device=x.device)
    nvfp4_quantize_dispatch_into(x, dest_rows, topk, group_offsets, q, s_blk, s32, layout, ws, stream)
    return q, s_blk, s32[:n]


def nvfp4_quantize_2d_into(x, q_row, s_row, q_col, s_col, s32, flags=ROWWISE | COLWISE, ws=None, stream=None):
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    ws = _ws(ws, 1, x.device)
    _check(load().nvfp4_quantize_2d(_ptr(x), R, C, x.stride(0), flags, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                    _ptr(s_col), _ptr(s32), _ptr(ws), ws.numel(), _stream(stream)),
           "nvfp4_quantize_2d")


def nvfp4_quantize_2d(x, flags=ROWWISE | COLWISE, ws=None, stream=None):
    """NVFP4 weights with 16x16 block scales: (q_row [R,C/2], s_row tiles,
    q_col [C,R/2], s_col tiles, s32 [1]); copies not requested are None."""
    R, C = x.shape
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if flags & ROWWISE:
        q_row = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
        s_row = _u8(scale_bytes(FMT_NVFP4, R, C), dev)
    if flags & COLWISE:
        q_col = torch.empty((C, R // 2), dtype=torch.uint8, device=dev)
        s_col = _u8(scale_bytes(FMT_NVFP4, C, R), dev)
    s32 = torch.empty(1, dtype=torch.float32, device=dev)
    nvfp4_quantize_2d_into(x, q_row, s_row, q_col, s_col, s32, flags, ws, stream)
    return q_row, s_row, q_col, s_col, s32


def nvfp4_quantize_rht_colwise_into(x, sign_mask, q_col, s_col, s32, stochastic=False, seed=0, ws=None,
                                    stream=None):
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    ws = _ws(ws, 1, x.device)
    _check(load().nvfp4_quantize_rht_colwise(_ptr(x), R, C, x.stride(0), int(sign_mask), int(bool(stochastic)),
                                             int(seed), _ptr(q_col), _ptr(s_col), _ptr(s32), _ptr(ws), ws.numel(),
                                             _stream(stream)),
           "nvfp4_quantize_rht_colwise")


def nvfp4_quantize_rht_colwise(x, sign_mask, stochastic=False, seed=0, ws=None, stream=None):
    """Transposed NVFP4 copy of a Wgrad input [R, C] with the 16x16 random
    Hadamard transform along R: (q_col [C, R/2], s_col tiles, s32 [1]);
    stochastic rounding of the codes for gradient inputs."""
    R, C = x.shape
    q_col = torch.empty((C, R // 2), dtype=torch.uint8, device=x.device)
    s_col = _u8(scale_bytes(FMT_NVFP4, C, R), x.device)
    s32 = torch.empty(1, dtype=torch.float32, device=x.device)
    nvfp4_quantize_rht_colwise_into(x, sign_mask, q_col, s_col, s32, stochastic, seed, ws, stream)
    return q_col, s_col, s32


def nvfp4_quantize_per_token_sr_into(x, seed, q, s_blk, s32, stream=None):
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    _check(load().nvfp4_quantize_per_token_sr(_ptr(x), R, C, x.stride(0), int(seed), _ptr(q), _ptr(s_blk),
                                              _ptr(s32), _stream(stream)),
           "nvfp4_quantize_per_token_sr")


def nvfp4_quantize_per_token_sr(x, seed, stream=None):
    """Per-token NVFP4 of a gradient with stochastically rounded codes:
    (q [R, C/2], s_blk tiles, s32 [R])."""
    R, C = x.shape
    q = torch.empty((R, C // 2), dtype=torch.uint8, device=x.device)
    s_blk = _u8(scale_bytes(FMT_NVFP4, R, C), x.device)
    s32 = torch.empty(max(R, 1), dtype=torch.float32, device=x.device)
    nvfp4_quantize_per_token_sr_into(x, seed, q, s_blk, s32, stream)
    return q, s_blk, s32[:R]


# ---------------------------------------------------------------- dequantize
def dequantize_into(fmt, q, s, out, s32=None, s32_mode=S32_NONE, group_offsets=None, stream=None):
    R = q.shape[0]
    C = q.shape[1] if fmt == FMT_MXFP8 else q.shape[1] * 2
    G = 0 if group_offsets is None else group_offsets.numel() - 1
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _check(load().dequantize(fmt, _ptr(q), _ptr(s), _ptr(s32), s32_mode, _ptr(group_offsets), G, R, C,
                             od, _ptr(out), _stream(stream)), "dequantize")


def dequantize(fmt, q, s, s32=None, s32_mode=None, group_offsets=None, out_dtype=torch.float32,
               stream=None):
    R = q.shape[0]
    C = q.shape[1] if fmt == FMT_MXFP8 else q.shape[1] * 2
    if s32_mode is None:
        if s32 is None:
            s32_mode = S32_NONE
        elif s32.numel() == R and R != 1:
            s32_mode = S32_ROW
        else:
            s32_mode = S32_TENSOR
    out = torch.empty((R, C), dtype=out_dtype, device=q.device)
    dequantize_into(fmt, q, s, out, s32, s32_mode, group_offsets, stream)
    return out


# ---------------------------------------------------------------- BF16 GEMM
def bf16_gemm_into(A, B, out, accumulate=False, ws=None, stream=None):
    """out (+)= A @ B^T for bf16 A [M, K], B [N, K] (rows K-contiguous, any
    row stride that is a multiple of 8); out f32 or bf16 [M, N]."""
    assert A.dtype == torch.bfloat16 and B.dtype == torch.bfloat16
    assert A.stride(1) == 1 and B.stride(1) == 1 and out.stride(1) == 1
    (M, K), N = A.shape, B.shape[0]
    assert B.shape[1] == K and out.shape == (M, N)
    ws = _ws(ws, 1, A.device)
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _check(load().bf16_gemm(M, N, K, _ptr(A), A.stride(0), _ptr(B), B.stride(0), od, _ptr(out), out.stride(0),
                            int(accumulate), _ptr(ws), ws.numel(), _stream(stream)), "bf16_gemm")


def bf16_gemm(A, B, out_dtype=torch.float32, ws=None, stream=None):
    """Dense BF16 GEMM A @ B^T on the tensor cores (the dequantized-backward
    mode's Dgrad / Wgrad)."""
    out = torch.empty((A.shape[0], B.shape[0]), dtype=out_dtype, device=A.device)
    bf16_gemm_into(A, B, out, False, ws, stream)
    return out


# ---------------------------------------------------------------- GEMM
def _mode(v, n):
    if v is None:
        return S32_NONE
    return S32_TENSOR if (v.numel() == 1 and n != 1) else S32_ROW


def bs_gemm_into(fmt, A, SA, B, SB, K, out, A32=None, B32=None, accumulate=False, ws=None,
                 stream=None, a32_mode=None, b32_mode=None):
    M, N = A.shape[0], B.shape[0]
    ws = _ws(ws, 1, A.device)
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    am = _mode(A32, M) if a32_mode is None else a32_mode
    bm = _mode(B32, N) if b32_mode is None else b32_mode
    _check(load().bs_gemm(fmt, M, N, K, _ptr(A), _ptr(SA), _ptr(A32), am, _ptr(B), _ptr(SB), _ptr(B32),
                          bm, od, _ptr(out), out.stride(0), int(accumulate), _ptr(ws), ws.numel(),
                          _stream(stream)), "bs_gemm")


def bs_gemm(fmt, A, SA, B, SB, K, A32=None, B32=None, out_dtype=torch.float32, ws=None, stream=None):
    """C[M, N] = A32[m] * B32[n] * sum_k A^[m,k] B^[n,k] on the tensor cores.
    A: [M, K] (MXFP8) or [M, K/2] (NVFP4) u8 with K contiguous; SA/SB the
    scale tiles; A32/B32 optional FP32 decode scales (per row or [1])."""
    out = torch.empty((A.shape[0], B.shape[0]), dtype=out_dtype, device=A.device)
    bs_gemm_into(fmt, A, SA, B, SB, K, out, A32, B32, False, ws, stream)
    return out


def bs_grouped_gemm_into(fmt, group_offsets, A, SA, B, SB, K, out, A32=None, B32=None, ws=None,
                         stream=None):
    G = group_offsets.numel() - 1
    rows = A.shape[0]
    N = B.shape[1]
    ws = _ws(ws, G, A.device)
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _check(load().bs_grouped_gemm(fmt, G, _ptr(group_offsets), rows, N, K, _ptr(A), _ptr(SA), _ptr(A32),
                                  _ptr(B), _ptr(SB), _ptr(B32), od, _ptr(out), out.stride(0), _ptr(ws),
                                  ws.numel(), _stream(stream)), "bs_grouped_gemm")


def bs_grouped_gemm(fmt, group_offsets, A, SA, B, SB, K, A32=None, B32=None,
                    out_dtype=torch.bfloat16, ws=None, stream=None):
    """MoE routed-expert GEMM: rows [off[g], off[g+1]) of A times B[g]^T.
    B: [G, N, K] (or [G, N, K/2]) u8; SB the [G*N, K/bs] scale tiles."""
    out = torch.empty((A.shape[0], B.shape[1]), dtype=out_dtype, device=A.device)
    bs_grouped_gemm_into(fmt, group_offsets, A, SA, B, SB, K, out, A32, B32, ws, stream)
    return out


def bs_grouped_gemm_fused_into(fmt, group_offsets, total_rows, A, SA, B, SB, K, out, A32=None, B32=None,
                               a_rows=None, epilogue=EPI_NONE, ws=None, stream=None):
    """In-place form of :func:`bs_grouped_gemm_fused`."""
    G = group_offsets.numel() - 1
    N = B.shape[1]
    ws = _ws(ws, G, A.device)
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    src_rows = A.shape[0] if a_rows is not None else 0
    _check(load().bs_grouped_gemm_fused(fmt, G, _ptr(group_offsets), total_rows, N, K, _ptr(A), _ptr(SA),
                                        _ptr(A32), _ptr(a_rows), src_rows, _ptr(B), _ptr(SB), _ptr(B32),
                                        epilogue, od, _ptr(out), out.stride(0), _ptr(ws), ws.numel(),
                                        _stream(stream)), "bs_grouped_gemm_fused")


def bs_grouped_gemm_fused(fmt, group_offsets, A, SA, B, SB, K, A32=None, B32=None, a_rows=None,
                          epilogue=EPI_NONE, out_dtype=torch.bfloat16, ws=None, stream=None):
    """MoE expert GEMM with the dispatch gather and / or the SwiGLU fused in.

    a_rows (device int64 [rows]): token of each dispatched row; A, SA, A32
    are then the token-major quantize output (plain scale layout).
    epilogue=EPI_SWIGLU: B holds gate rows [0, F) and up rows [F, 2F) per
    expert; returns h [rows, F] bf16 instead of the gate|up output."""
    rows = a_rows.numel() if a_rows is not None else A.shape[0]
    n_out = B.shape[1] // 2 if epilogue == EPI_SWIGLU else B.shape[1]
    out = torch.empty((rows, n_out), dtype=out_dtype, device=A.device)
    bs_grouped_gemm_fused_into(fmt, group_offsets, rows, A, SA, B, SB, K, out, A32, B32, a_rows, epilogue,
                               ws, stream)
    return out


# ---------------------------------------------------------------- MoE combine
def bs_grouped_gemm_swiglu_nvfp4_into(group_offsets, total_rows, A, SA, B, SB, K, q_h, s_h, s32_h, A32=None,
                                      B32=None, h=None, ws=None, stream=None):
    """In-place form of :func:`bs_grouped_gemm_swiglu_nvfp4`."""
    G = group_offsets.numel() - 1
    N = B.shape[1]
    ws = _ws(ws, G, A.device)
    _check(load().bs_grouped_gemm_swiglu_nvfp4(G, _ptr(group_offsets), total_rows, N, K, _ptr(A), _ptr(SA),
                                               _ptr(A32), _ptr(B), _ptr(SB), _ptr(B32), _ptr(q_h), _ptr(s_h),
                                               _ptr(s32_h), _ptr(h), h.stride(0) if h is not None else 0,
                                               _ptr(ws), ws.numel(), _stream(stream)),
           "bs_grouped_gemm_swiglu_nvfp4")


def bs_grouped_gemm_swiglu_nvfp4(group_offsets, A, SA, B, SB, K, A32=None, B32=None, with_h=False, ws=None,
                                 stream=None):
    """gate|up expert GEMM + SwiGLU + per-token NVFP4 of h in one kernel.
    B: [G, 2F, K/2] (gate rows, then up rows).  Returns (q_h [R, F/2],
    s_h grouped scale tiles, s32_h [R]) and, with with_h, the bf16 h too."""
    G = group_offsets.numel() - 1
    R = A.shape[0]
    F = B.shape[1] // 2
    q_h = torch.empty((R, F // 2), dtype=torch.uint8, device=A.device)
    s_h = _u8(scale_bytes_grouped(FMT_NVFP4, R, G, F), A.device)
    s32_h = torch.empty(max(R, 1), dtype=torch.float32, device=A.device)
    h = torch.empty((R, F), dtype=torch.bfloat16, device=A.device) if with_h else None
    bs_grouped_gemm_swiglu_nvfp4_into(group_offsets, R, A, SA, B, SB, K, q_h, s_h, s32_h, A32, B32, h, ws, stream)
    return (q_h, s_h, s32_h, h) if with_h else (q_h, s_h, s32_h)


def moe_combine_into(y, rows_of_slot, weights, out, stream=None):
    """out [T, H] = sum_j weights[t, j] * y[rows_of_slot[t, j]] (binary32, j
    in order); y bf16 [R, H]; out f32 or bf16."""
    assert y.dtype == torch.bfloat16 and y.stride(1) == 1 and out.stride(1) == 1
    T, k = rows_of_slot.shape
    od = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    _check(load().mx8_moe_combine(_ptr(y), y.shape[0], y.stride(0), _ptr(rows_of_slot), _ptr(weights), T,
                                  y.shape[1], k, od, _ptr(out), out.stride(0), _stream(stream)),
           "mx8_moe_combine")


def moe_combine(y, rows_of_slot, weights, out_dtype=torch.bfloat16, stream=None):
    out = torch.empty((rows_of_slot.shape[0], y.shape[1]), dtype=out_dtype, device=y.device)
    moe_combine_into(y, rows_of_slot, weights, out, stream)
    return out


# ---------------------------------------------------------------- SwiGLU
def swiglu_into(gate_up, h, stream=None):
    R, F2 = gate_up.shape
    _check(load().mx8_swiglu(_ptr(gate_up), R, F2 // 2, gate_up.stride(0), _ptr(h), h.stride(0),
                             _stream(stream)), "mx8_swiglu")


def swiglu(gate_up, stream=None):
    """h = silu(gate) * up for a bf16 [R, 2F] gate|up matrix -> bf16 [R, F]."""
    R, F2 = gate_up.shape
    h = torch.empty((R, F2 // 2), dtype=torch.bfloat16, device=gate_up.device)
    swiglu_into(gate_up, h, stream)
    return h


# ---------------------------------------------------------------- errors
def check_device_error(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error
    status of the workspace: OK or ERR_TIMEOUT."""
    return int(load().mx8_check_device_error(_ptr(ws), _stream(stream)))


def selftest_bounded_wait(ws, limit_ns: int, stream=None):
    _check(load().mx8_selftest_bounded_wait(_ptr(ws), limit_ns, _stream(stream)), "selftest")
