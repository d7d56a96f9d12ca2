"""Shared helpers of the test suite: building the CUDA library and the oracle,
moving numpy arrays to the device and back."""
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ensure_built():
    import oracle
    from moe_mx8_quantize_gb300 import build as libbuild
    oracle.build()
    libbuild.build()


def dev(a, dtype=None):
    """numpy -> cuda tensor (bytes preserved)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.to(dtype)


def host(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def gemm_tolerance_ok(y, ref, absref, bf16=False, K=0):
    """|y - ref| <= 1e-5 * sum_k |a^||b^| + K * 2^-126.  The second term is
    the FP32 accumulator's underflow: a product below the smallest normal
    FP32 value may contribute zero."""
    y = np.asarray(y, np.float64)
    tol = 1e-5 * absref + K * 2.0 ** -126
    if bf16:
        tol = tol + 2.0 ** -8 * np.abs(ref)
    bad = np.abs(y - ref) > tol
    return (~bad).all(), np.nonzero(bad.ravel())[0]


def scale_offsets(rows_idx, scols, padded_row_of=None):
    """Byte offsets, in a tensor-core scale buffer with scols logical scale
    columns, of the scales of the given rows (rows x scols array).
    padded_row_of maps a data row to its row in the (grouped) padded layout."""
    rows_idx = np.asarray(rows_idx, np.int64)
    pr = rows_idx if padded_row_of is None else padded_row_of(rows_idx)
    kt = -(-scols // 4)
    k = np.arange(scols, dtype=np.int64)
    r = pr[:, None]
    return ((r // 128) * kt + k[None, :] // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + k[None, :] % 4


def grouped_padded_row(offs):
    """Data row -> row of the per-group padded scale layout."""
    offs = np.asarray(offs, np.int64)
    n = np.diff(offs)
    pref = np.concatenate([[0], np.cumsum(-(-n // 128) * 128)])

    def f(rows):
        g = np.searchsorted(offs, rows, side="right") - 1
        return pref[g] + (rows - offs[g])
    return f


def swiglu_tolerance(g, ag, u, au, K):
    """Allowed |h - silu(g) u| for the GPU's h = RN_bf16(silu(g~) u~), where
    g, u are the FP64 references of the gate and up outputs (ag, au their
    sums of |a||b|) and g~, u~ the GPU's outputs: each within the GEMM
    tolerance 1e-5 sum|a||b| + K 2^-126 of its reference, then rounded to
    bf16 (at most half a unit, 2^-8 relative).  silu has slope in [-0.1,
    1.1]; silu(g~) u~ in binary32 with expf is within 2^-20 relative of the
    exact product; the final bf16 rounding adds at most half a unit (2^-8
    relative) and 2^-134 absolute (half the smallest bf16 subnormal).
    Returns (the FP64 reference of h, the tolerance)."""
    eg = 1e-5 * ag + K * 2.0 ** -126
    eu = 1e-5 * au + K * 2.0 ** -126
    dg = eg + 2.0 ** -8 * (np.abs(g) + eg)
    du = eu + 2.0 ** -8 * (np.abs(u) + eu)
    sil = g / (1.0 + np.exp(-g))
    h = sil * u
    prop = 1.1 * (np.abs(u) + du) * dg + np.abs(sil) * du
    tol = prop + 2.0 ** -8 * (np.abs(h) + prop) + 2.0 ** -20 * np.abs(h) + 2.0 ** -134
    return h, tol
