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
