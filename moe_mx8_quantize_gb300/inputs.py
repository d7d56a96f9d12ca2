"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle
checks.

This module holds no quantization arithmetic: it only draws bf16 tensors and
routings with the shapes and value mixes of the workloads the pages discuss
(a 2048x2048 -> 8192 linear layer, Qwen3-30B-A3B-shaped and DeepSeek-V3-shaped
MoE expert layers, a quantizer bandwidth sweep).  Every generator takes a seed
and a device; the same recipe runs on CPU or CUDA (the random streams differ
between devices, so a check that needs the values on the host copies them).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

BF16_MAX_BITS = 0x7F7F


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std, g, device, outlier_frac=0.0, outlier_mult=1.0):
    """N(0, std^2) in fp32, a fraction of entries multiplied by outlier_mult,
    rounded to bf16."""
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    if outlier_frac > 0:
        mask = torch.rand(shape, generator=g, device=device) < outlier_frac
        x = torch.where(mask, x * outlier_mult, x)
    return x.to(torch.bfloat16)


# ------------------------------------------------------------------ PR1
def pr1(seed: int = 0, device="cpu"):
    """X[128x512] activation and W[256x512] weight, N(0,1) with 1% of the
    entries scaled by 50 (outliers)."""
    g = _gen(seed, device)
    X = normal_bf16((128, 512), 1.0, g, device, 0.01, 50.0)
    W = normal_bf16((256, 512), 1.0, g, device, 0.01, 50.0)
    return {"X": X, "W": W}


# ------------------------------------------------------------------ linear
LINEAR_SHAPE = dict(tokens=2048, in_features=2048, out_features=8192)


def linear(seed: int = 1, device="cpu", tokens=2048, in_features=2048, out_features=8192):
    """Linear layer in_features -> out_features: input X ~ N(0,1),
    weight W ~ N(0, 0.02^2), output gradient dY ~ N(0, 1e-3^2)."""
    g = _gen(seed, device)
    X = normal_bf16((tokens, in_features), 1.0, g, device)
    W = normal_bf16((out_features, in_features), 0.02, g, device)
    dY = normal_bf16((tokens, out_features), 1e-3, g, device)
    return {"X": X, "W": W, "dY": dY}


# ------------------------------------------------------------------ routing
def route_uniform(tokens: int, experts: int, topk: int, g, device):
    """Top-k uniform routing: each token picks k distinct experts, all
    subsets equally likely (argsort of uniform noise)."""
    noise = torch.rand((tokens, experts), generator=g, device=device)
    return torch.argsort(noise, dim=1)[:, :topk].contiguous()


def route_zipf(tokens: int, experts: int, topk: int, s: float, g, device):
    """Top-k Zipf(s)-skewed routing: a seeded random permutation ranks the
    experts, P(rank r) ~ r^-s, k distinct experts drawn per token without
    replacement."""
    perm = torch.randperm(experts, generator=g, device=device)
    ranks = torch.arange(1, experts + 1, device=device, dtype=torch.float64)
    p_rank = ranks.pow(-s)
    probs = torch.empty(experts, device=device, dtype=torch.float64)
    probs[perm] = p_rank
    probs = (probs / probs.sum()).to(torch.float32)
    ids = torch.multinomial(probs.expand(tokens, experts), topk, replacement=False, generator=g)
    return ids.contiguous()


@dataclass
class Dispatch:
    """Rows of the grouped GEMM: row i holds token `token_of_row[i]` routed to
    expert e, rows sorted by expert; rows of expert e are
    [offsets[e], offsets[e+1])."""
    token_of_row: torch.Tensor   # int64 [T*k]
    expert_of_row: torch.Tensor  # int64 [T*k]
    offsets: torch.Tensor        # int64 [E+1]
    row_of_slot: torch.Tensor    # int64 [T, k]: the row holding token t's j-th expert choice


def dispatch(topk_ids: torch.Tensor, experts: int) -> Dispatch:
    T, k = topk_ids.shape
    flat = topk_ids.reshape(-1).to(torch.int64)
    order = torch.argsort(flat, stable=True)
    token = (order // k).to(torch.int64)
    expert = flat[order]
    counts = torch.bincount(flat, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int64, device=topk_ids.device)
    offsets[1:] = torch.cumsum(counts, 0)
    row_of_slot = torch.empty_like(order)
    row_of_slot[order] = torch.arange(order.numel(), device=order.device, dtype=torch.int64)
    return Dispatch(token, expert, offsets, row_of_slot.reshape(T, k))


def route_weights(tokens: int, topk: int, seed: int, device) -> torch.Tensor:
    """Router weights of the top-k choices: a softmax over k N(0,1) logits per
    token, float32 [tokens, topk] (own generator, so other inputs keep their
    streams)."""
    g = _gen(seed + 1000, device)
    logits = torch.randn((tokens, topk), generator=g, device=device, dtype=torch.float32)
    return torch.softmax(logits, dim=1).contiguous()


# ------------------------------------------------------------------ MoE
QWEN_SHAPE = dict(tokens=4096, hidden=2048, experts=128, ffn=768, topk=8)
DSV3_SHAPE = dict(tokens=16384, hidden=7168, experts=256, ffn=2048, topk=8)


def moe(seed: int, device, tokens, hidden, experts, ffn, topk, routing="uniform",
        zipf_s=1.1, outlier_frac=0.0, outlier_mult=1.0, with_weights=True):
    """MoE expert layer: activations X [tokens, hidden] ~ N(0,1) (optional
    outliers), per expert a joint gate|up weight W_gu [E, 2*ffn, hidden] and
    a down weight W_d [E, hidden, ffn], both ~ N(0, 0.02^2)."""
    g = _gen(seed, device)
    X = normal_bf16((tokens, hidden), 1.0, g, device, outlier_frac, outlier_mult)
    if routing == "uniform":
        ids = route_uniform(tokens, experts, topk, g, device)
    else:
        ids = route_zipf(tokens, experts, topk, zipf_s, g, device)
    out = {"X": X, "topk_ids": ids}
    if with_weights:
        out["W_gu"] = normal_bf16((experts, 2 * ffn, hidden), 0.02, g, device)
        out["W_d"] = normal_bf16((experts, hidden, ffn), 0.02, g, device)
    return out


def qwen_moe(seed: int = 2, device="cpu", **over):
    """Qwen3-30B-A3B-shaped expert layer: 4096 tokens, hidden 2048,
    128 experts, FFN 768, top-8 uniform routing."""
    kw = dict(QWEN_SHAPE)
    kw.update(over)
    return moe(seed, device, routing="uniform", **kw)


def dsv3_moe(seed: int = 3, device="cpu", **over):
    """DeepSeek-V3-shaped expert layer: 16384 tokens, hidden 7168, 256 routed
    experts, FFN 2048, top-8 Zipf(1.1) routing, 0.5% of activations x100."""
    kw = dict(DSV3_SHAPE)
    kw.update(over)
    return moe(seed, device, routing="zipf", zipf_s=1.1, outlier_frac=0.005,
               outlier_mult=100.0, **kw)


# ------------------------------------------------------------------ sweep
def sweep(rows: int, cols: int, seed: int = 4, device="cpu"):
    """Bandwidth-sweep tensor [rows, cols] (cols % 32 == 0) built from 1x32
    blocks of five kinds:
      70% N(0,1); 5% all zero; 5% N(0,1) with one +-bf16-max entry;
      10% bf16 subnormals only; 10% "tie" blocks: one entry +-448*2^e and the
      rest at odd multiples of 2^(p-4) * 2^e (values exactly halfway between
      neighbouring 4-bit-significand numbers), e drawn in [-20, 20];
    then 1% of all entries set to exactly zero.
    """
    assert cols % 32 == 0
    g = _gen(seed, device)
    nb = cols // 32
    base = torch.randn((rows, nb, 32), generator=g, device=device, dtype=torch.float32)
    kind = torch.rand((rows, nb, 1), generator=g, device=device)
    sign = torch.where(torch.rand((rows, nb, 32), generator=g, device=device) < 0.5, -1.0, 1.0)

    # subnormal-only blocks: bf16 bit patterns with exponent field 0
    mant = torch.randint(1, 128, (rows, nb, 32), generator=g, device=device, dtype=torch.int32)
    sub = (mant << 16).view(torch.float32) * sign

    # tie blocks
    e = torch.randint(-20, 21, (rows, nb, 1), generator=g, device=device).to(torch.float32)
    p = torch.randint(-6, 8, (rows, nb, 32), generator=g, device=device).to(torch.float32)
    odd = torch.randint(0, 8, (rows, nb, 32), generator=g, device=device).to(torch.float32) * 2 + 17
    tie = odd / 16.0 * torch.exp2(p) * torch.exp2(e) * sign
    lead = torch.randint(0, 32, (rows, nb, 1), generator=g, device=device)
    tie.scatter_(2, lead, (448.0 * torch.exp2(e)) * sign.gather(2, lead))

    # one +-bf16 max per block
    bf16max = torch.tensor([BF16_MAX_BITS << 16], dtype=torch.int32, device=device).view(torch.float32)
    maxblk = base.clone()
    pos = torch.randint(0, 32, (rows, nb, 1), generator=g, device=device)
    maxblk.scatter_(2, pos, bf16max.expand(rows, nb, 1) * sign.gather(2, pos))

    x = torch.where(kind < 0.70, base, torch.zeros_like(base))
    x = torch.where((kind >= 0.75) & (kind < 0.80), maxblk, x)
    x = torch.where((kind >= 0.80) & (kind < 0.90), sub, x)
    x = torch.where(kind >= 0.90, tie, x)
    zero = torch.rand((rows, nb, 32), generator=g, device=device) < 0.01
    x = torch.where(zero, torch.zeros_like(x), x)
    return x.reshape(rows, cols).to(torch.bfloat16)


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns on the host."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
