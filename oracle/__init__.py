"""CPU oracle for MXFP8 / per-token NVFP4 / MXFP4 quantization, the
block-scaled GEMM and the dequantized-backward BF16 GEMM.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the library's product path
never imports this package.  The arithmetic lives in ``mx8q_oracle.c`` (plain
scalar C, built by :func:`build`); this module only marshals numpy arrays.

Every function cites the passage it follows in the C source.  Inputs are bf16
bit patterns held in ``numpy.uint16`` arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx8q_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmx8q_oracle.so")

# gcc flags: -ffp-contract=off keeps every float operation a single IEEE
# round-to-nearest step (no fused multiply-add, no fast-math).
_CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
           "-fno-fast-math", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library in-tree; returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None
_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.or_bf16_to_f32.restype = ctypes.c_float
        lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.or_f32_to_bf16.restype = ctypes.c_uint16
        lib.or_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.or_e4m3_decode.restype = ctypes.c_double
        lib.or_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_e4m3_encode.argtypes = [ctypes.c_float]
        lib.or_e2m1_decode.restype = ctypes.c_double
        lib.or_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.or_e2m1_encode.restype = ctypes.c_uint8
        lib.or_e2m1_encode.argtypes = [ctypes.c_float]
        lib.or_e8m0_decode.restype = ctypes.c_double
        lib.or_e8m0_decode.argtypes = [ctypes.c_uint8]
        lib.or_mxfp8_block_exp.restype = ctypes.c_int
        lib.or_mxfp8_block_exp.argtypes = [ctypes.c_float]
        lib.or_mxfp8_quantize_rowwise.argtypes = [_p, _i64, _i64, _i64, _p, _p]
        lib.or_mxfp8_quantize_colwise.argtypes = [_p, _i64, _i64, _i64, _p, _p]
        lib.or_dequant_mxfp8.argtypes = [_p, _p, _i64, _i64, _p]
        lib.or_mxfp4_block_exp.restype = ctypes.c_int
        lib.or_mxfp4_block_exp.argtypes = [ctypes.c_float]
        lib.or_mxfp4_quantize_rowwise.argtypes = [_p, _i64, _i64, _i64, _p, _p]
        lib.or_mxfp4_quantize_colwise.argtypes = [_p, _i64, _i64, _i64, _p, _p]
        lib.or_dequant_mxfp4.argtypes = [_p, _p, _i64, _i64, _p]
        lib.or_nvfp4_quantize.argtypes = [_p, _i64, _i64, _i64, ctypes.c_int, _p,
                                          ctypes.c_int, _p, _p, _p]
        lib.or_dequant_nvfp4.argtypes = [_p, _p, _p, ctypes.c_int, _p, ctypes.c_int,
                                         _i64, _i64, _p]
        lib.or_swizzled_bytes.restype = _i64
        lib.or_swizzled_bytes.argtypes = [_i64, _i64, _p, ctypes.c_int]
        lib.or_swizzle_scales.argtypes = [_p, _i64, _i64, _p, ctypes.c_int, _p]
        lib.or_gemm_ref.argtypes = [ctypes.c_int, _i64, _i64, _i64,
                                    _p, _p, _p, ctypes.c_int,
                                    _p, _p, _p, ctypes.c_int,
                                    _p, _i64, _p, _p, _p]
        lib.or_grouped_gemm_ref.argtypes = [ctypes.c_int, ctypes.c_int, _p, _i64, _i64,
                                            _p, _p, _p, _p, _p, _p,
                                            _p, _i64, _p, _p, _p]
        lib.or_swiglu.argtypes = [_p, _i64, _i64, _p]
        lib.or_nvfp4_quantize_2d.argtypes = [_p, _i64, _i64, _i64, _p, _p, _p, _p, _p]
        lib.or_rht16.argtypes = [_p, ctypes.c_uint, _p]
        lib.or_nvfp4_quantize_rht_colwise.argtypes = [_p, _i64, _i64, _i64, ctypes.c_uint, ctypes.c_int,
                                                      ctypes.c_uint64, _p, _p, _p]
        lib.or_philox4x32_10.argtypes = [_p, _p, _p]
        lib.or_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.or_sr_bits.restype = ctypes.c_uint32
        lib.or_e2m1_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        lib.or_e2m1_sr.restype = ctypes.c_uint8
        lib.or_nvfp4_quantize_sr.argtypes = [_p, _i64, _i64, _i64, ctypes.c_uint64, _p, _p, _p]
        lib.or_moe_combine.argtypes = [_p, _i64, _i64, _p, _p, _i64, ctypes.c_int, _p]
        lib.or_bf16_gemm_ref.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _p]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- codecs
def bf16_to_f32(bits):
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x):
    """Round-to-nearest-even narrowing of float32 to bf16 bit patterns."""
    L = _L()
    x = np.asarray(x, dtype=np.float32)
    return np.array([L.or_f32_to_bf16(float(v)) for v in x.ravel()],
                    dtype=np.uint16).reshape(x.shape)


def e4m3_decode(code: int) -> float:
    return _L().or_e4m3_decode(code)


def e4m3_encode(v: float) -> int:
    return _L().or_e4m3_encode(v)


def e2m1_decode(code: int) -> float:
    return _L().or_e2m1_decode(code)


def e2m1_encode(v: float) -> int:
    return _L().or_e2m1_encode(v)


def e8m0_decode(code: int) -> float:
    return _L().or_e8m0_decode(code)


def mxfp8_block_exp(amax: float) -> int:
    return _L().or_mxfp8_block_exp(amax)


# ----------------------------------------------------------------- MXFP8
def mxfp8_quantize_rowwise(x_bits):
    """Rowwise MXFP8 (1x32 blocks along rows) -> (q [R,C] u8, s [R,C/32] u8)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    _L().or_mxfp8_quantize_rowwise(_ptr(x), R, C, C, _ptr(q), _ptr(s))
    return q, s


def mxfp8_quantize_colwise(x_bits):
    """Columnwise MXFP8 (32x1 blocks down columns of the bf16 source), stored
    transposed -> (qT [C,R] u8, sT [C,R/32] u8)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert R % 32 == 0
    q = np.empty((C, R), np.uint8)
    s = np.empty((C, R // 32), np.uint8)
    _L().or_mxfp8_quantize_colwise(_ptr(x), R, C, C, _ptr(q), _ptr(s))
    return q, s


def dequant_mxfp8(q, s):
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    R, C = q.shape
    out = np.empty((R, C), np.float32)
    _L().or_dequant_mxfp8(_ptr(q), _ptr(s), R, C, _ptr(out))
    return out


# ----------------------------------------------------------------- MXFP4
def mxfp4_block_exp(amax: float) -> int:
    return _L().or_mxfp4_block_exp(amax)


def mxfp4_quantize_rowwise(x_bits):
    """Rowwise MXFP4 (1x32 blocks along rows) -> (q [R,C/2] packed E2M1,
    s [R,C/32] E8M0)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % 32 == 0
    q = np.zeros((R, C // 2), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    _L().or_mxfp4_quantize_rowwise(_ptr(x), R, C, C, _ptr(q), _ptr(s))
    return q, s


def mxfp4_quantize_colwise(x_bits):
    """Columnwise MXFP4 (32x1 blocks down columns), stored transposed ->
    (qT [C,R/2] packed, sT [C,R/32])."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert R % 32 == 0
    q = np.zeros((C, R // 2), np.uint8)
    s = np.empty((C, R // 32), np.uint8)
    _L().or_mxfp4_quantize_colwise(_ptr(x), R, C, C, _ptr(q), _ptr(s))
    return q, s


def dequant_mxfp4(q, s):
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    R, C = q.shape[0], q.shape[1] * 2
    out = np.empty((R, C), np.float32)
    _L().or_dequant_mxfp4(_ptr(q), _ptr(s), R, C, _ptr(out))
    return out


# ----------------------------------------------------------------- NVFP4
SCOPE_TOKEN, SCOPE_GROUP, SCOPE_TENSOR = 0, 1, 2


def nvfp4_quantize(x_bits, scope=SCOPE_TOKEN, offs=None):
    """Two-level NVFP4 -> (q [R,C/2] u8, s [R,C/16] u8 E4M3, s32 f32 decode
    scales: [R] per token, [G] per group, [1] per tensor)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % 16 == 0
    q = np.empty((R, C // 2), np.uint8)
    s = np.empty((R, C // 16), np.uint8)
    if scope == SCOPE_TOKEN:
        s32 = np.empty(R, np.float32)
        o, G = None, 0
    elif scope == SCOPE_GROUP:
        o = _c(offs, np.int64)
        G = len(o) - 1
        s32 = np.empty(G, np.float32)
    else:
        s32 = np.empty(1, np.float32)
        o, G = None, 0
    _L().or_nvfp4_quantize(_ptr(x), R, C, C, scope, _ptr(o), G, _ptr(q), _ptr(s), _ptr(s32))
    return q, s, s32


S32_NONE, S32_ROW, S32_TENSOR, S32_GROUP = 0, 1, 2, 3


def nvfp4_quantize_2d(x_bits):
    """NVFP4 weights with 16x16 block scales and one FP32 tensor scale ->
    (q_row [R,C/2], s_row [R,C/16], q_col [C,R/2], s_col [C,R/16], s32 [1]);
    the columnwise copy is the transpose of the rowwise one."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert R % 16 == 0 and C % 16 == 0
    q_row = np.zeros((R, C // 2), np.uint8)
    s_row = np.empty((R, C // 16), np.uint8)
    q_col = np.zeros((C, R // 2), np.uint8)
    s_col = np.empty((C, R // 16), np.uint8)
    s32 = np.empty(1, np.float32)
    _L().or_nvfp4_quantize_2d(_ptr(x), R, C, C, _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col), _ptr(s32))
    return q_row, s_row, q_col, s_col, s32


def rht16(x, sign_mask):
    """y = H16 diag(s) x / 4 in binary32 (fast Walsh-Hadamard order)."""
    xi = np.ascontiguousarray(np.asarray(x, np.float32).reshape(16))
    y = np.empty(16, np.float32)
    _L().or_rht16(_ptr(xi), int(sign_mask) & 0xFFFF, _ptr(y))
    return y


def nvfp4_quantize_rht_colwise(x_bits, sign_mask, stochastic=False, seed=0):
    """Transposed NVFP4 copy of a Wgrad input with the 16x16 random Hadamard
    transform along its rows -> (qT [C,R/2], sT [C,R/16], s32 [1]); the
    codes by stochastic rounding under `seed` when `stochastic`."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert R % 16 == 0
    qT = np.zeros((C, R // 2), np.uint8)
    sT = np.empty((C, R // 16), np.uint8)
    s32 = np.empty(1, np.float32)
    _L().or_nvfp4_quantize_rht_colwise(_ptr(x), R, C, C, int(sign_mask) & 0xFFFF, int(bool(stochastic)), int(seed),
                                       _ptr(qT), _ptr(sT), _ptr(s32))
    return qT, sT, s32


def philox4x32_10(counter, key):
    """Philox4x32-10 block: 4 x uint32 counter, 2 x uint32 key -> 4 x uint32."""
    c = np.ascontiguousarray(np.asarray(counter, np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, np.uint32).reshape(2))
    out = np.empty(4, np.uint32)
    _L().or_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits(seed, e):
    return int(_L().or_sr_bits(int(seed), int(e)))


def e2m1_sr(v, bits):
    return int(_L().or_e2m1_sr(float(v), int(bits) & 0xFFFFFFFF))


def nvfp4_quantize_sr(x_bits, seed):
    """Per-token NVFP4 with stochastically rounded codes -> (q, s, s32)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % 16 == 0
    q = np.zeros((R, C // 2), np.uint8)
    s = np.empty((R, C // 16), np.uint8)
    s32 = np.empty(R, np.float32)
    _L().or_nvfp4_quantize_sr(_ptr(x), R, C, C, int(seed), _ptr(q), _ptr(s), _ptr(s32))
    return q, s, s32


def dequant_nvfp4(q, s, s32=None, s32_mode=S32_ROW, offs=None):
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    R = q.shape[0]
    C = q.shape[1] * 2
    out = np.empty((R, C), np.float32)
    s32a = None if s32 is None else _c(s32, np.float32)
    o = None if offs is None else _c(offs, np.int64)
    G = 0 if o is None else len(o) - 1
    mode = S32_NONE if s32a is None else s32_mode
    _L().or_dequant_nvfp4(_ptr(q), _ptr(s), _ptr(s32a), mode, _ptr(o), G, R, C, _ptr(out))
    return out


# ------------------------------------------------------- tensor-core layout
def swizzled_bytes(rows, scols, offs=None):
    o = None if offs is None else _c(offs, np.int64)
    G = 0 if o is None else len(o) - 1
    return int(_L().or_swizzled_bytes(rows, scols, _ptr(o), G))


def swizzle_scales(canon, offs=None):
    """Canonical [rows, scols] scales -> flat tensor-core tile layout (u8)."""
    c = _c(canon, np.uint8)
    rows, scols = c.shape
    o = None if offs is None else _c(offs, np.int64)
    G = 0 if o is None else len(o) - 1
    out = np.empty(swizzled_bytes(rows, scols, o), np.uint8)
    _L().or_swizzle_scales(_ptr(c), rows, scols, _ptr(o), G, _ptr(out))
    return out


# ----------------------------------------------------------------- GEMM
FMT_MXFP8, FMT_NVFP4 = 0, 1
MODE_NONE, MODE_ROW, MODE_TENSOR = 0, 1, 2


def _mode_of(v, n):
    if v is None:
        return MODE_NONE
    return MODE_TENSOR if v.size == 1 and n != 1 else MODE_ROW


def gemm_ref(fmt, A, SA, B, SB, K, a32=None, b32=None, pairs=None):
    """FP64 reference of Y = A^ . B^T over exactly decoded operands.

    fmt: 0 MXFP8, 1 NVFP4, 2 MXFP4.
    A: [M, K] (MXFP8 bytes) or [M, K/2] (packed NVFP4 / MXFP4); SA canonical.
    Returns (ref, absref): [M, N] arrays, or [npairs] for sampled pairs.
    """
    A = _c(A, np.uint8); B = _c(B, np.uint8)
    SA = _c(SA, np.uint8); SB = _c(SB, np.uint8)
    M, N = A.shape[0], B.shape[0]
    a = None if a32 is None else _c(a32, np.float32)
    b = None if b32 is None else _c(b32, np.float32)
    pr = None if pairs is None else _c(pairs, np.int64).reshape(-1, 2)
    n = M * N if pr is None else pr.shape[0]
    ref = np.empty(n, np.float64)
    absref = np.empty(n, np.float64)
    scratch = np.empty(2 * K, np.float64)
    _L().or_gemm_ref(fmt, M, N, K, _ptr(A), _ptr(SA), _ptr(a), _mode_of(a, M),
                     _ptr(B), _ptr(SB), _ptr(b), _mode_of(b, N),
                     _ptr(pr), 0 if pr is None else pr.shape[0],
                     _ptr(ref), _ptr(absref), _ptr(scratch))
    if pr is None:
        return ref.reshape(M, N), absref.reshape(M, N)
    return ref, absref


def grouped_gemm_ref(fmt, offs, A, SA, B, SB, K, a32=None, b32=None, pairs=None):
    """FP64 reference of the MoE grouped GEMM: row m of group g times B[g]^T.

    B: [G, N, K] (or [G, N, K/2] packed); SB canonical [G*N, K/bs];
    pairs: [P, 2] (row, n) indices.  Returns (ref, absref) of length P.
    """
    o = _c(offs, np.int64)
    G = len(o) - 1
    A = _c(A, np.uint8); B = _c(B, np.uint8)
    SA = _c(SA, np.uint8); SB = _c(SB, np.uint8)
    N = B.shape[1]
    a = None if a32 is None else _c(a32, np.float32)
    b = None if b32 is None else _c(b32, np.float32)
    pr = _c(pairs, np.int64).reshape(-1, 2)
    ref = np.empty(pr.shape[0], np.float64)
    absref = np.empty(pr.shape[0], np.float64)
    scratch = np.empty(2 * K, np.float64)
    _L().or_grouped_gemm_ref(fmt, G, _ptr(o), N, K, _ptr(A), _ptr(SA), _ptr(a),
                             _ptr(B), _ptr(SB), _ptr(b), _ptr(pr), pr.shape[0],
                             _ptr(ref), _ptr(absref), _ptr(scratch))
    return ref, absref


def bf16_gemm_ref(A_bits, B_bits, pairs=None):
    """FP64 reference of Y = A . B^T over bf16 operands (bit patterns,
    A [M, K], B [N, K]): the dequantized-backward BF16 GEMM.
    Returns (ref, absref): [M, N] arrays, or [npairs] for sampled pairs."""
    A = _c(A_bits, np.uint16); B = _c(B_bits, np.uint16)
    (M, K), N = A.shape, B.shape[0]
    assert B.shape[1] == K
    pr = None if pairs is None else _c(pairs, np.int64).reshape(-1, 2)
    n = M * N if pr is None else pr.shape[0]
    ref = np.empty(n, np.float64)
    absref = np.empty(n, np.float64)
    _L().or_bf16_gemm_ref(M, N, K, _ptr(A), K, _ptr(B), K, _ptr(pr), 0 if pr is None else pr.shape[0],
                          _ptr(ref), _ptr(absref))
    if pr is None:
        return ref.reshape(M, N), absref.reshape(M, N)
    return ref, absref


def moe_combine(y_bits, rows, w):
    """out [T, H] f32 = sum_j w[t, j] * y[rows[t, j]] in binary32, j in order."""
    y = _c(y_bits, np.uint16)
    r = _c(rows, np.int64)
    ww = _c(w, np.float32)
    T, k = r.shape
    out = np.empty((T, y.shape[1]), np.float32)
    _L().or_moe_combine(_ptr(y), y.shape[0], y.shape[1], _ptr(r), _ptr(ww), T, k, _ptr(out))
    return out


# ----------------------------------------------------------------- SwiGLU
def swiglu(gu_bits):
    """h = RN_bf16(silu(g) * u) for a bf16 [R, 2F] gate|up matrix (bit patterns)."""
    gu = _c(gu_bits, np.uint16)
    R, F2 = gu.shape
    h = np.empty((R, F2 // 2), np.uint16)
    _L().or_swiglu(_ptr(gu), R, F2 // 2, _ptr(h))
    return h
