#!/usr/bin/env python
"""Benchmark of the microscaling hot path on one GB300 (or N replicas).

One step = every operation of the hot path, on seeded synthetic inputs:

  MXFP8 linear layer, input [2048, 2048] -> 8192 (forward + backward):
    rowwise+columnwise MXFP8 quantization of X, W and dY (one read of each,
    the three tensors in one launch),
    Fprop Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X (block-scaled
    tcgen05 GEMMs), and the dequantized-backward operands (X^, W^ in bf16);
  NVFP4 linear Fprop on the same layer: per-token X, per-tensor W;
  Qwen3-30B-A3B-shaped MoE expert layer with per-token NVFP4: 4096 tokens
    routed top-8 over 128 experts (32768 rows), hidden 2048, FFN 768:
    per-token activation quantization of the 4096 tokens (each token encoded
    once, before dispatch, and written to its 8 dispatched rows), per-expert
    weight quantization (gate|up joint), the gate|up grouped GEMM with SwiGLU
    and the per-token NVFP4 quantization of h in its epilogue, the down
    grouped GEMM, and the combine of each token's 8 expert outputs weighted
    by its router weights.

value = block-scaled GEMM FLOPs of the step / step time (quantizers,
dequantization and SwiGLU included in the time).  Per-kernel times come from
CUDA events on the launching stream inside the timed region.  The same linear
layer in MXFP4 (E2M1 x 32 blocks, E8M0 scales), its dequantized-backward mode
(dequantize + dense BF16 Dgrad / Wgrad) and its NVFP4 pretraining-recipe
variant (2-D weight blocks, random Hadamard transform on the Wgrad inputs,
stochastic rounding of gradients) are timed beside the step, per kernel,
under "extra", and so are the DeepSeek-V3-shaped MoE layer (its own step, with
its MXFP8 shared expert) and the quantizer bandwidth sweep (2^20 .. 2^30
elements).

`--impl reference` times the CPU oracle (test infrastructure) on all host
cores on a bounded sample of the same step and extrapolates to the full step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LINEAR = dict(tokens=2048, in_features=2048, out_features=8192)
QWEN = dict(tokens=4096, hidden=2048, experts=128, ffn=768, topk=8)
METRIC = "quantize HBM GB/s; MXFP8/NVFP4 block-scaled GEMM TFLOPS vs dense peak"
WORKLOAD = ("MXFP8 linear 2048x2048->8192 fwd+bwd (rowwise+colwise quant, Fprop/Dgrad/Wgrad, "
            "dequantized-backward operands) + NVFP4 linear Fprop + Qwen3-30B-A3B-shaped NVFP4 MoE "
            "expert layer (4096 tok, top-8 of 128 experts, hidden 2048, FFN 768; dispatch, SwiGLU, combine)")


# ----------------------------------------------------------------- peaks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# nominal dense-rate ratios to bf16 on GB300 (2.25 / 4.5 / 13.5 PFLOP/s)
RATIO = {"bf16": 1.0, "fp8": 2.0, "fp4": 6.0}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.5)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- the step
class MoeLayer:
    """One routed-expert layer with per-token NVFP4, resident in HBM: the
    tokens encoded once before dispatch and written to their top-k
    dispatched rows, per-expert weight quantization (gate|up joint), the
    gate|up grouped GEMM with SwiGLU in its epilogue, per-token quantization
    of h, the down grouped GEMM, and the router-weighted combine back to token
    order.  Routing (top-k ids -> expert offsets and row maps) is set-up."""

    # fused: h is quantized in the gate|up GEMM's epilogue (one thread-block
    # cluster per 128-row band, F <= 1024); unfused: in a separate launch
    LABELS_FUSED = ("nvfp4_quant_token moe_act", "nvfp4_quant_expert W_gu", "nvfp4_quant_expert W_d",
                    "nvfp4_moe_gemm gate_up+swiglu+quant_h", "nvfp4_grouped_gemm down", "moe_combine")
    LABELS_UNFUSED = ("nvfp4_quant_token moe_act", "nvfp4_quant_expert W_gu", "nvfp4_quant_expert W_d",
                      "nvfp4_moe_gemm gate_up+swiglu", "nvfp4_quant_token moe_h", "nvfp4_grouped_gemm down",
                      "moe_combine")

    def __init__(self, mx, torch, device, d, E, F, topk, route_w, ws):
        from moe_mx8_quantize_gb300 import inputs
        self.mx, self.ws = mx, ws
        H = d["X"].shape[1]
        TM = d["X"].shape[0]
        disp = inputs.dispatch(d["topk_ids"], E)
        self.offs = disp.offsets
        self.rows = R = int(disp.offsets[-1].item())
        self.X = d["X"].contiguous()                                         # token-major activations
        self.a_rows = disp.token_of_row.to(torch.int64).contiguous()       # token of each dispatched row
        self.dest_rows = torch.argsort(self.a_rows, stable=True).to(torch.int64).contiguous()
        self.rows_of_slot = disp.row_of_slot.contiguous()                  # (token, choice) -> row
        self.route_w = route_w
        self.W_gu = d["W_gu"].reshape(E * 2 * F, H).contiguous()
        self.W_d = d["W_d"].reshape(E * H, F).contiguous()
        self.e_offs_gu = torch.arange(E + 1, device=device, dtype=torch.int64) * (2 * F)
        self.e_offs_d = torch.arange(E + 1, device=device, dtype=torch.int64) * H
        u8 = lambda n: torch.empty(max(n, 16), dtype=torch.uint8, device=device)
        f32 = lambda n: torch.empty(max(n, 1), dtype=torch.float32, device=device)
        sb4 = lambda r, c: u8(mx.scale_bytes(mx.FMT_NVFP4, r, c))
        sb4g = lambda r, g, c: u8(mx.scale_bytes_grouped(mx.FMT_NVFP4, r, g, c))
        bf = lambda r, c: torch.empty((r, c), dtype=torch.bfloat16, device=device)
        self.A4, self.SA4, self.A432 = u8(R * H // 2)[: R * H // 2].view(R, H // 2), sb4g(R, E, H), f32(R)
        self.Wgu4 = u8(E * 2 * F * H // 2)[: E * 2 * F * H // 2].view(E, 2 * F, H // 2)
        self.SWgu4, self.Wgu432 = sb4(E * 2 * F, H), f32(E)
        self.Wd4 = u8(E * H * F // 2)[: E * H * F // 2].view(E, H, F // 2)
        self.SWd4, self.Wd432 = sb4(E * H, F), f32(E)
        self.Hs = bf(R, F)
        self.H4, self.SH4, self.H432 = u8(R * F // 2)[: R * F // 2].view(R, F // 2), sb4g(R, E, F), f32(R)
        self.OUT = bf(R, H)
        self.Y = bf(TM, H)                                                   # combined, token order
        self.E, self.F, self.H, self.TM, self.topk = E, F, H, TM, topk
        # the step quantizes h in a separate launch: measured faster than the
        # cluster-fused epilogue (timed beside the step as "moe_gate_up_quant_h")
        self.fused = False
        self.LABELS = self.LABELS_FUSED if self.fused else self.LABELS_UNFUSED

    def plan(self):
        R, E, F, H, TM, k = self.rows, self.E, self.F, self.H, self.TM, self.topk
        nvq = lambda r, c: 2.5625 * r * c + 4 * r
        # before dispatch: bf16 read once per token; codes, block scales and S_dec
        # written to each of the token's k dispatched rows
        nvqd = lambda t, c: 2 * t * c + k * (0.5625 * t * c + 4 * t)
        rows = [
            ("nvfp4_quant_token moe_act", "hbm", nvqd(TM, H)),
            ("nvfp4_quant_expert W_gu", "hbm", nvq(E * 2 * F, H)),
            ("nvfp4_quant_expert W_d", "hbm", nvq(E * H, F)),
            ("nvfp4_moe_gemm gate_up+swiglu+quant_h", "fp4", 2.0 * R * 2 * F * H),
            ("nvfp4_moe_gemm gate_up+swiglu", "fp4", 2.0 * R * 2 * F * H),
            ("nvfp4_quant_token moe_h", "hbm", nvq(R, F)),
            ("nvfp4_grouped_gemm down", "fp4", 2.0 * R * H * F),
            ("moe_combine", "hbm", 2.0 * R * H + 2.0 * TM * H + 12.0 * R),
        ]
        return [r for r in rows if r[0] in self.LABELS]

    def bytes_moved(self):
        """Algorithmic HBM bytes of the layer's kernels: the quantizers' and
        the combine's, plus the GEMMs' operands and outputs (NVFP4 codes and
        scales read; h written as bf16, or as NVFP4 when it is quantized in
        the gate|up epilogue; the bf16 down output written)."""
        R, E, F, H = self.rows, self.E, self.F, self.H
        q = sum(w for _, kind, w in self.plan() if kind == "hbm")
        h_out = (0.5625 * R * F + 4 * R) if self.fused else 2 * R * F
        gemm = (0.5625 * R * H + 0.5625 * E * 2 * F * H + h_out          # gate|up: A, W_gu in; h out
                + 0.5625 * R * F + 0.5625 * E * H * F + 2 * R * H)        # down: h4, W_d in; out
        return q + gemm

    def launches(self):
        mx, ws = self.mx, self.ws
        launches = [
            ("nvfp4_quant_token moe_act", lambda: mx.nvfp4_quantize_dispatch_into(
                self.X, self.dest_rows, self.topk, self.offs, self.A4, self.SA4, self.A432, mx.DISPATCH_ROWS, ws)),
            ("nvfp4_quant_expert W_gu", lambda: mx.nvfp4_quantize_into(self.W_gu, self.Wgu4.view(-1, self.H // 2),
                                                                       self.SWgu4, self.Wgu432, mx.SCOPE_GROUP,
                                                                       self.e_offs_gu, ws)),
            ("nvfp4_quant_expert W_d", lambda: mx.nvfp4_quantize_into(self.W_d, self.Wd4.view(-1, self.F // 2),
                                                                      self.SWd4, self.Wd432, mx.SCOPE_GROUP,
                                                                      self.e_offs_d, ws)),
            ("nvfp4_moe_gemm gate_up+swiglu+quant_h", lambda: mx.bs_grouped_gemm_swiglu_nvfp4_into(
                self.offs, self.rows, self.A4, self.SA4, self.Wgu4, self.SWgu4, self.H, self.H4, self.SH4,
                self.H432, self.A432, self.Wgu432, None, ws)),
            ("nvfp4_moe_gemm gate_up+swiglu", lambda: mx.bs_grouped_gemm_fused_into(
                mx.FMT_NVFP4, self.offs, self.rows, self.A4, self.SA4, self.Wgu4, self.SWgu4, self.H, self.Hs,
                self.A432, self.Wgu432, None, mx.EPI_SWIGLU, ws)),
            ("nvfp4_quant_token moe_h", lambda: mx.nvfp4_quantize_into(self.Hs, self.H4, self.SH4, self.H432,
                                                                       mx.SCOPE_TOKEN, self.offs, ws)),
            ("nvfp4_grouped_gemm down", lambda: mx.bs_grouped_gemm_into(mx.FMT_NVFP4, self.offs, self.H4, self.SH4,
                                                                         self.Wd4, self.SWd4, self.F, self.OUT,
                                                                         self.H432, self.Wd432, ws)),
            ("moe_combine", lambda: mx.moe_combine_into(self.OUT, self.rows_of_slot, self.route_w, self.Y)),
        ]
        return [l for l in launches if l[0] in self.LABELS]

    def gemm_flops(self):
        return sum(w for _, kind, w in self.plan() if kind in ("fp8", "fp4"))


class Step:
    """All buffers of one hot-path step, resident in HBM, and the launches."""

    def __init__(self, device, seed_base=0):
        import torch
        import moe_mx8_quantize_gb300 as mx
        from moe_mx8_quantize_gb300 import inputs

        self.mx, self.torch = mx, torch
        self.dev = device
        T, H, O = LINEAR["tokens"], LINEAR["in_features"], LINEAR["out_features"]
        lin = inputs.linear(seed=1 + seed_base, device=device)
        self.X, self.W, self.dY = lin["X"], lin["W"], lin["dY"]
        q = QWEN
        # one workspace per concurrent branch of the step (error word + scratch)
        self.ws = mx.new_workspace(max(q["experts"], 1), device)
        self.ws_b = mx.new_workspace(max(q["experts"], 1), device)
        self.ws_c = mx.new_workspace(max(q["experts"], 1), device)
        moe = inputs.qwen_moe(seed=2 + seed_base, device=device)
        route_w = inputs.route_weights(q["tokens"], q["topk"], 2 + seed_base, device)
        self.moe = MoeLayer(mx, torch, device, moe, q["experts"], q["ffn"], q["topk"], route_w, self.ws_c)
        u8 = lambda n: torch.empty(max(n, 16), dtype=torch.uint8, device=device)
        f32 = lambda n: torch.empty(max(n, 1), dtype=torch.float32, device=device)
        sb8 = lambda r, c: u8(mx.scale_bytes(mx.FMT_MXFP8, r, c))
        sb4 = lambda r, c: u8(mx.scale_bytes(mx.FMT_NVFP4, r, c))
        bf = lambda r, c: torch.empty((r, c), dtype=torch.bfloat16, device=device)
        # MXFP8 copies
        self.Xr, self.SXr, self.Xc, self.SXc = u8(T * H).view(-1)[: T * H].view(T, H), sb8(T, H), \
            u8(T * H)[: T * H].view(H, T), sb8(H, T)
        self.Wr, self.SWr, self.Wc, self.SWc = u8(O * H)[: O * H].view(O, H), sb8(O, H), \
            u8(O * H)[: O * H].view(H, O), sb8(H, O)
        self.dYr, self.SdYr, self.dYc, self.SdYc = u8(T * O)[: T * O].view(T, O), sb8(T, O), \
            u8(T * O)[: T * O].view(O, T), sb8(O, T)
        self.Y, self.dX = bf(T, O), bf(T, H)
        self.dW = torch.empty((O, H), dtype=torch.float32, device=device)
        self.Xhat, self.What = bf(T, H), bf(O, H)
        # NVFP4 linear
        self.X4, self.SX4, self.X432 = u8(T * H // 2)[: T * H // 2].view(T, H // 2), sb4(T, H), f32(T)
        self.W4, self.SW4, self.W432 = u8(O * H // 2)[: O * H // 2].view(O, H // 2), sb4(O, H), f32(1)
        self.Y4 = bf(T, O)
        self.H_, self.T, self.O = H, T, O

    # -- algorithmic work per launch (bytes or FLOPs) and roofline class
    def plan(self):
        T, H, O = self.T, self.H_, self.O
        mxq = lambda r, c: 4.0625 * r * c
        nvq = lambda r, c: 2.5625 * r * c + 4 * r
        return [
            ("mxfp8_quant_rc X+W+dY", "hbm", mxq(T, H) + mxq(O, H) + mxq(T, O)),
            ("mxfp8_gemm Fprop", "fp8", 2.0 * T * O * H),
            ("mxfp8_gemm Dgrad", "fp8", 2.0 * T * H * O),
            ("mxfp8_gemm Wgrad", "fp8", 2.0 * O * H * T),
            ("dequant_mxfp8 X", "hbm", (1 + 1 / 32 + 2) * T * H),
            ("dequant_mxfp8 W", "hbm", (1 + 1 / 32 + 2) * O * H),
            ("nvfp4_quant_token X", "hbm", nvq(T, H)),
            ("nvfp4_quant_tensor W", "hbm", nvq(O, H)),
            ("nvfp4_gemm Fprop", "fp4", 2.0 * T * O * H),
        ] + self.moe.plan()

    def launches(self):
        """The step as a list of (label, callable); each callable launches
        library kernels on the current stream."""
        mx = self.mx
        RC = mx.ROWWISE | mx.COLWISE
        ws, ws_b = self.ws, self.ws_b
        return [
            # the layer's three tensors, rowwise + columnwise, in one launch
            ("mxfp8_quant_rc X+W+dY", lambda: mx.mx8_quantize_batch_into(mx.FMT_MXFP8, (
                (self.X, self.Xr, self.SXr, self.Xc, self.SXc), (self.W, self.Wr, self.SWr, self.Wc, self.SWc),
                (self.dY, self.dYr, self.SdYr, self.dYc, self.SdYc)), RC, ws)),
            ("mxfp8_gemm Fprop", lambda: mx.bs_gemm_into(mx.FMT_MXFP8, self.Xr, self.SXr, self.Wr, self.SWr, self.H_, self.Y, ws=ws)),
            ("mxfp8_gemm Dgrad", lambda: mx.bs_gemm_into(mx.FMT_MXFP8, self.dYr, self.SdYr, self.Wc, self.SWc, self.O, self.dX, ws=ws)),
            ("mxfp8_gemm Wgrad", lambda: mx.bs_gemm_into(mx.FMT_MXFP8, self.dYc, self.SdYc, self.Xc, self.SXc, self.T, self.dW, ws=ws)),
            ("dequant_mxfp8 X", lambda: mx.dequantize_into(mx.FMT_MXFP8, self.Xr, self.SXr, self.Xhat)),
            ("dequant_mxfp8 W", lambda: mx.dequantize_into(mx.FMT_MXFP8, self.Wr, self.SWr, self.What)),
            ("nvfp4_quant_token X", lambda: mx.nvfp4_quantize_into(self.X, self.X4, self.SX4, self.X432, mx.SCOPE_TOKEN, None, ws_b)),
            ("nvfp4_quant_tensor W", lambda: mx.nvfp4_quantize_into(self.W, self.W4, self.SW4, self.W432, mx.SCOPE_TENSOR, None, ws_b)),
            ("nvfp4_gemm Fprop", lambda: mx.bs_gemm_into(mx.FMT_NVFP4, self.X4, self.SX4, self.W4, self.SW4, self.H_, self.Y4,
                                                         self.X432, self.W432, ws=ws_b, a32_mode=mx.S32_ROW, b32_mode=mx.S32_TENSOR)),
        ] + self.moe.launches()

    # The step's three independent chains: the MXFP8 linear layer, the NVFP4
    # linear Fprop and the NVFP4 MoE layer.  The end-to-end measurement runs
    # each on its own stream (its own workspace), so one chain's host copies
    # overlap another's kernels; within a chain the order is the data order
    # above.
    BRANCHES = (
        ("mxfp8_quant_rc X+W+dY", "mxfp8_gemm Fprop", "mxfp8_gemm Dgrad", "mxfp8_gemm Wgrad", "dequant_mxfp8 X",
         "dequant_mxfp8 W"),
        ("nvfp4_quant_token X", "nvfp4_quant_tensor W", "nvfp4_gemm Fprop"),
        MoeLayer.LABELS_UNFUSED,          # the Qwen-shaped layer (FFN 768)
    )

    def workspaces(self):
        return (self.ws, self.ws_b, self.ws_c)

    def run_concurrent(self, streams, io=False):
        """Launches the step as its three branches on `streams` (the first is
        the caller's current stream), forked from and joined back into it.  With
        io, each branch first copies its inputs from pinned host memory and last
        copies its results back (the e2e measurement)."""
        torch = self.torch
        fns = dict(self.launches())
        s0 = streams[0]
        fork = torch.cuda.Event()
        fork.record(s0)
        done = []
        for b, labels in enumerate(self.BRANCHES):
            st = streams[b]
            with torch.cuda.stream(st):
                if b > 0:
                    st.wait_event(fork)
                if io:
                    for d, h in self.io_in[b]:
                        d.copy_(h, non_blocking=True)
                    if b == 0:               # X is also an input of branch 1
                        self.x_ready.record(st)
                if io and b == 1:
                    st.wait_event(self.x_ready)
                for lab in labels:
                    fns[lab]()
                if io:
                    for d, h in self.io_out[b]:
                        h.copy_(d, non_blocking=True)
                if b > 0:
                    e = torch.cuda.Event()
                    e.record(st)
                    done.append(e)
        for e in done:
            s0.wait_event(e)

    def setup_io(self):
        """Pinned host copies of each branch's per-step inputs and results."""
        torch = self.torch
        pin = lambda t: t.detach().cpu().pin_memory()
        self.io_in = ([(self.X, pin(self.X)), (self.dY, pin(self.dY))], [], [(self.moe.X, pin(self.moe.X))])
        empty = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        self.io_out = ([(self.Y, empty(self.Y)), (self.dX, empty(self.dX))], [(self.Y4, empty(self.Y4))],
                       [(self.moe.Y, empty(self.moe.Y))])
        self.x_ready = torch.cuda.Event()

    # kernel launches per label (the rest launch one; group scope adds a memset)
    KERNELS_PER_LABEL = {"nvfp4_quant_tensor W": 2}   # tensor abs-max, then the encode

    def gemm_flops(self):
        return sum(w for _, kind, w in self.plan() if kind in ("fp8", "fp4"))


class FusedQuantH:
    """The Qwen-shaped layer's gate|up GEMM with SwiGLU and the per-token NVFP4
    quantization of h fused into its epilogue (clusters of F / 128 CTAs),
    timed beside the step against the two launches the step uses; it reads
    the step's operands and writes the same codes, scales and S_dec."""

    def __init__(self, step):
        self.lay = step.moe

    def plan(self):
        L = self.lay
        return [("nvfp4_moe_gemm gate_up+swiglu+quant_h", "fp4", 2.0 * L.rows * 2 * L.F * L.H)]

    def launches(self):
        L = self.lay
        mx = L.mx
        return [("nvfp4_moe_gemm gate_up+swiglu+quant_h", lambda: mx.bs_grouped_gemm_swiglu_nvfp4_into(
            L.offs, L.rows, L.A4, L.SA4, L.Wgu4, L.SWgu4, L.H, L.H4, L.SH4, L.H432, L.A432, L.Wgu432, None, L.ws))]


class Dsv3Moe:
    """The DeepSeek-V3-shaped routed-expert layer (16384 tokens, hidden 7168,
    256 experts, FFN 2048, top-8 Zipf(1.1), 0.5% of activations x100), the
    same launches as the step's MoE layer, timed as its own step beside it."""

    def __init__(self, step, seed=3):
        torch, mx = step.torch, step.mx
        from moe_mx8_quantize_gb300 import inputs
        q = inputs.DSV3_SHAPE
        self.ws = mx.new_workspace(q["experts"], step.dev)
        d = inputs.dsv3_moe(seed=seed, device=step.dev)
        route_w = inputs.route_weights(q["tokens"], q["topk"], seed, step.dev)
        self.layer = MoeLayer(mx, torch, step.dev, d, q["experts"], q["ffn"], q["topk"], route_w, self.ws)
        self.shape = q

    def plan(self):
        return self.layer.plan()

    def launches(self):
        return self.layer.launches()


class Dsv3SharedExpert:
    """The DeepSeek-V3 shared expert, kept at higher precision than the
    routed experts: MXFP8 rowwise quantization of the 16384 x 7168 tokens and
    of its weights, gate|up Fprop (7168 -> 2 x 2048), SwiGLU, MXFP8 of h, down
    Fprop (2048 -> 7168).  Timed beside the routed layer."""

    def __init__(self, dsv3, seed=31):
        lay = dsv3.layer
        mx = lay.mx
        import torch
        from moe_mx8_quantize_gb300 import inputs
        dev = lay.X.device
        T, H, F = lay.TM, lay.H, lay.F
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.X = lay.X
        self.Wgu = inputs.normal_bf16((2 * F, H), 0.02, g, dev)
        self.Wd = inputs.normal_bf16((H, F), 0.02, g, dev)
        u8 = lambda r, c: torch.empty((r, c), dtype=torch.uint8, device=dev)
        sb = lambda r, c: torch.empty(max(mx.scale_bytes(mx.FMT_MXFP8, r, c), 16), dtype=torch.uint8, device=dev)
        bf = lambda r, c: torch.empty((r, c), dtype=torch.bfloat16, device=dev)
        self.Xq, self.SX = u8(T, H), sb(T, H)
        self.Wguq, self.SWgu = u8(2 * F, H), sb(2 * F, H)
        self.Wdq, self.SWd = u8(H, F), sb(H, F)
        self.GU, self.h = bf(T, 2 * F), bf(T, F)
        self.hq, self.Sh = u8(T, F), sb(T, F)
        self.Y = bf(T, H)
        self.mx, self.ws, self.T, self.H, self.F = mx, dsv3.ws, T, H, F

    def plan(self):
        T, H, F = self.T, self.H, self.F
        q = lambda r, c: (2 + 1 + 1 / 32) * r * c
        return [
            ("mxfp8_quant_row shared X", "hbm", q(T, H)),
            ("mxfp8_quant_row shared W_gu", "hbm", q(2 * F, H)),
            ("mxfp8_quant_row shared W_d", "hbm", q(H, F)),
            ("mxfp8_gemm shared gate_up", "fp8", 2.0 * T * 2 * F * H),
            ("swiglu shared", "hbm", 6.0 * T * F),
            ("mxfp8_quant_row shared h", "hbm", q(T, F)),
            ("mxfp8_gemm shared down", "fp8", 2.0 * T * H * F),
        ]

    def launches(self):
        mx, ws = self.mx, self.ws
        R = mx.ROWWISE
        return [
            ("mxfp8_quant_row shared X", lambda: mx.mx8_quantize_into(self.X, self.Xq, self.SX, None, None, R, ws)),
            ("mxfp8_quant_row shared W_gu", lambda: mx.mx8_quantize_into(self.Wgu, self.Wguq, self.SWgu, None, None, R, ws)),
            ("mxfp8_quant_row shared W_d", lambda: mx.mx8_quantize_into(self.Wd, self.Wdq, self.SWd, None, None, R, ws)),
            ("mxfp8_gemm shared gate_up", lambda: mx.bs_gemm_into(mx.FMT_MXFP8, self.Xq, self.SX, self.Wguq, self.SWgu,
                                                                  self.H, self.GU, ws=ws)),
            ("swiglu shared", lambda: mx.swiglu_into(self.GU, self.h)),
            ("mxfp8_quant_row shared h", lambda: mx.mx8_quantize_into(self.h, self.hq, self.Sh, None, None, R, ws)),
            ("mxfp8_gemm shared down", lambda: mx.bs_gemm_into(mx.FMT_MXFP8, self.hq, self.Sh, self.Wdq, self.SWd,
                                                               self.F, self.Y, ws=ws)),
        ]


class Mxfp4Linear:
    """The step's linear layer in MXFP4 (32-element E2M1 blocks under one E8M0
    scale): rowwise + columnwise quantization of X, W and dY, Fprop, Dgrad and
    Wgrad, and the dequantized W^.  Measured beside the step (its own timed
    region), not part of `value`."""

    def __init__(self, step):
        torch, mx = step.torch, step.mx
        self.step, self.mx = step, mx
        T, H, O = step.T, step.H_, step.O
        dev = step.dev
        u8 = lambda r, c: torch.empty((r, c), dtype=torch.uint8, device=dev)
        sb = lambda r, c: torch.empty(max(mx.scale_bytes(mx.FMT_MXFP4, r, c), 16), dtype=torch.uint8, device=dev)
        self.Xr, self.SXr, self.Xc, self.SXc = u8(T, H // 2), sb(T, H), u8(H, T // 2), sb(H, T)
        self.Wr, self.SWr, self.Wc, self.SWc = u8(O, H // 2), sb(O, H), u8(H, O // 2), sb(H, O)
        self.dYr, self.SdYr, self.dYc, self.SdYc = u8(T, O // 2), sb(T, O), u8(O, T // 2), sb(O, T)
        self.Y = torch.empty((T, O), dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty((O, H), dtype=torch.float32, device=dev)
        self.What = torch.empty((O, H), dtype=torch.bfloat16, device=dev)

    def plan(self):
        st = self.step
        T, H, O = st.T, st.H_, st.O
        q = lambda r, c: (2 + 2 * (0.5 + 1 / 32)) * r * c     # bf16 in, two packed copies + scales out
        return [
            ("mxfp4_quant_rc X+W+dY", "hbm", q(T, H) + q(O, H) + q(T, O)),
            ("mxfp4_gemm Fprop", "fp4", 2.0 * T * O * H),
            ("mxfp4_gemm Dgrad", "fp4", 2.0 * T * H * O),
            ("mxfp4_gemm Wgrad", "fp4", 2.0 * O * H * T),
            ("dequant_mxfp4 W", "hbm", (0.5 + 1 / 32 + 2) * O * H),
        ]

    def launches(self):
        mx, st = self.mx, self.step
        RC = mx.ROWWISE | mx.COLWISE
        ws = st.ws
        return [
            ("mxfp4_quant_rc X+W+dY", lambda: mx.mx8_quantize_batch_into(mx.FMT_MXFP4, (
                (st.X, self.Xr, self.SXr, self.Xc, self.SXc), (st.W, self.Wr, self.SWr, self.Wc, self.SWc),
                (st.dY, self.dYr, self.SdYr, self.dYc, self.SdYc)), RC, ws)),
            ("mxfp4_gemm Fprop", lambda: mx.bs_gemm_into(mx.FMT_MXFP4, self.Xr, self.SXr, self.Wr, self.SWr, st.H_, self.Y, ws=ws)),
            ("mxfp4_gemm Dgrad", lambda: mx.bs_gemm_into(mx.FMT_MXFP4, self.dYr, self.SdYr, self.Wc, self.SWc, st.O, self.dX, ws=ws)),
            ("mxfp4_gemm Wgrad", lambda: mx.bs_gemm_into(mx.FMT_MXFP4, self.dYc, self.SdYc, self.Xc, self.SXc, st.T, self.dW, ws=ws)),
            ("dequant_mxfp4 W", lambda: mx.dequantize_into(mx.FMT_MXFP4, self.Wr, self.SWr, self.What)),
        ]


class DequantBackward:
    """The dequantized-backward mode of the step's linear layer: the MXFP8
    copies the block-scaled backward uses, rebuilt in bf16 by dequantize(),
    then Dgrad = deq(dY_row) deq(W_col)^T and Wgrad = deq(dY_col) deq(X_col)^T
    as dense BF16 tensor-core GEMMs.  Measured beside the step (it reads the
    step's quantized copies), not part of `value`."""

    def __init__(self, step):
        torch = step.torch
        self.step, self.mx = step, step.mx
        T, H, O = step.T, step.H_, step.O
        bf = lambda r, c: torch.empty((r, c), dtype=torch.bfloat16, device=step.dev)
        self.dYr_h, self.Wc_h, self.dYc_h, self.Xc_h = bf(T, O), bf(H, O), bf(O, T), bf(H, T)
        self.dX = bf(T, H)
        self.dW = torch.empty((O, H), dtype=torch.float32, device=step.dev)

    def plan(self):
        st = self.step
        T, H, O = st.T, st.H_, st.O
        dq = lambda r, c: (1 + 1 / 32 + 2) * r * c
        return [
            ("dequant_mxfp8 dY_row", "hbm", dq(T, O)),
            ("dequant_mxfp8 W_col", "hbm", dq(H, O)),
            ("dequant_mxfp8 dY_col", "hbm", dq(O, T)),
            ("dequant_mxfp8 X_col", "hbm", dq(H, T)),
            ("bf16_gemm Dgrad", "bf16", 2.0 * T * H * O),
            ("bf16_gemm Wgrad", "bf16", 2.0 * O * H * T),
        ]

    def launches(self):
        mx, st = self.mx, self.step
        f = mx.FMT_MXFP8
        return [
            ("dequant_mxfp8 dY_row", lambda: mx.dequantize_into(f, st.dYr, st.SdYr, self.dYr_h)),
            ("dequant_mxfp8 W_col", lambda: mx.dequantize_into(f, st.Wc, st.SWc, self.Wc_h)),
            ("dequant_mxfp8 dY_col", lambda: mx.dequantize_into(f, st.dYc, st.SdYc, self.dYc_h)),
            ("dequant_mxfp8 X_col", lambda: mx.dequantize_into(f, st.Xc, st.SXc, self.Xc_h)),
            ("bf16_gemm Dgrad", lambda: mx.bf16_gemm_into(self.dYr_h, self.Wc_h, self.dX, ws=st.ws)),
            ("bf16_gemm Wgrad", lambda: mx.bf16_gemm_into(self.dYc_h, self.Xc_h, self.dW, ws=st.ws)),
        ]


class Nvfp4RecipeLinear:
    """The step's linear layer under the NVFP4 pretraining recipe's variants:
    W with 2-D 16x16 block scales (one copy for the forward and its transpose
    for Dgrad), X per token, the gradient dY per token with stochastically
    rounded codes, and the Wgrad inputs dY and X quantized columnwise after
    the 16x16 random Hadamard transform (stochastic codes for dY); then
    Fprop, Dgrad and Wgrad.  Measured beside the step, not part of `value`."""

    SIGNS = 0xB2D5          # the shared random sign vector of the transform
    KERNELS = {"nvfp4_2d W": 2, "nvfp4_rht_colwise_sr dY": 2, "nvfp4_rht_colwise X": 2}

    def __init__(self, step):
        torch, mx = step.torch, step.mx
        self.step, self.mx = step, mx
        T, H, O = step.T, step.H_, step.O
        dev = step.dev
        u8 = lambda r, c: torch.empty((r, c), dtype=torch.uint8, device=dev)
        sb = lambda r, c: torch.empty(max(mx.scale_bytes(mx.FMT_NVFP4, r, c), 16), dtype=torch.uint8, device=dev)
        f32 = lambda n: torch.empty(n, dtype=torch.float32, device=dev)
        self.Wr, self.SWr, self.Wc, self.SWc, self.W32 = u8(O, H // 2), sb(O, H), u8(H, O // 2), sb(H, O), f32(1)
        self.Xr, self.SXr, self.X32 = u8(T, H // 2), sb(T, H), f32(T)
        self.dYr, self.SdYr, self.dY32 = u8(T, O // 2), sb(T, O), f32(T)
        self.dYc, self.SdYc, self.dYc32 = u8(O, T // 2), sb(O, T), f32(1)
        self.Xc, self.SXc, self.Xc32 = u8(H, T // 2), sb(H, T), f32(1)
        self.Y = torch.empty((T, O), dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty((O, H), dtype=torch.float32, device=dev)

    def plan(self):
        st = self.step
        T, H, O = st.T, st.H_, st.O
        nvq = lambda r, c: 2.5625 * r * c + 4 * r
        return [
            ("nvfp4_2d W", "hbm", (2 + 2 * 0.5625) * O * H),
            ("nvfp4_quant_token X", "hbm", nvq(T, H)),
            ("nvfp4_quant_token_sr dY", "hbm", nvq(T, O)),
            ("nvfp4_rht_colwise_sr dY", "hbm", 2.5625 * T * O),
            ("nvfp4_rht_colwise X", "hbm", 2.5625 * T * H),
            ("nvfp4_gemm Fprop", "fp4", 2.0 * T * O * H),
            ("nvfp4_gemm Dgrad", "fp4", 2.0 * T * H * O),
            ("nvfp4_gemm Wgrad", "fp4", 2.0 * O * H * T),
        ]

    def launches(self):
        mx, st = self.mx, self.step
        ws = st.ws_b
        RC = mx.ROWWISE | mx.COLWISE
        return [
            ("nvfp4_2d W", lambda: mx.nvfp4_quantize_2d_into(st.W, self.Wr, self.SWr, self.Wc, self.SWc, self.W32, RC, ws)),
            ("nvfp4_quant_token X", lambda: mx.nvfp4_quantize_into(st.X, self.Xr, self.SXr, self.X32, mx.SCOPE_TOKEN, None, ws)),
            ("nvfp4_quant_token_sr dY", lambda: mx.nvfp4_quantize_per_token_sr_into(st.dY, 77, self.dYr, self.SdYr, self.dY32)),
            ("nvfp4_rht_colwise_sr dY", lambda: mx.nvfp4_quantize_rht_colwise_into(st.dY, self.SIGNS, self.dYc, self.SdYc,
                                                                                    self.dYc32, True, 78, ws)),
            ("nvfp4_rht_colwise X", lambda: mx.nvfp4_quantize_rht_colwise_into(st.X, self.SIGNS, self.Xc, self.SXc,
                                                                                self.Xc32, False, 0, ws)),
            ("nvfp4_gemm Fprop", lambda: mx.bs_gemm_into(mx.FMT_NVFP4, self.Xr, self.SXr, self.Wr, self.SWr, st.H_, self.Y,
                                                         self.X32, self.W32, ws=ws, a32_mode=mx.S32_ROW, b32_mode=mx.S32_TENSOR)),
            ("nvfp4_gemm Dgrad", lambda: mx.bs_gemm_into(mx.FMT_NVFP4, self.dYr, self.SdYr, self.Wc, self.SWc, st.O, self.dX,
                                                         self.dY32, self.W32, ws=ws, a32_mode=mx.S32_ROW, b32_mode=mx.S32_TENSOR)),
            ("nvfp4_gemm Wgrad", lambda: mx.bs_gemm_into(mx.FMT_NVFP4, self.dYc, self.SdYc, self.Xc, self.SXc, st.T, self.dW,
                                                         self.dYc32, self.Xc32, ws=ws, a32_mode=mx.S32_TENSOR,
                                                         b32_mode=mx.S32_TENSOR)),
        ]


CSRC = os.path.join(ROOT, "moe_mx8_quantize_gb300", "csrc")
# Translation units holding the kernels of each bench label (first matching
# prefix wins).  A kernel's code is its translation unit plus the launch
# setup in api.cu and the shared headers.
KERNEL_TUS = (
    ("mxfp8_quant_rc", ("quant_mxfp8.cu",)), ("mxfp4_quant_rc", ("quant_mxfp8.cu",)),
    ("dequant_", ("dequant.cu",)), ("moe_combine", ("dequant.cu",)),
    ("nvfp4_quant_tensor", ("quant_nvfp4.cu", "quant_nvfp4_2d.cu")),
    ("nvfp4_quant_token_sr", ("quant_wgrad.cu",)), ("nvfp4_rht", ("quant_wgrad.cu",)),
    ("nvfp4_2d", ("quant_nvfp4_2d.cu",)), ("nvfp4_quant", ("quant_nvfp4.cu",)),
    ("mxfp8_gemm", ("bs_gemm.cu",)), ("mxfp4_gemm", ("bs_gemm.cu",)), ("nvfp4_gemm", ("bs_gemm.cu",)),
    ("nvfp4_moe_gemm", ("bs_gemm.cu",)), ("nvfp4_grouped_gemm", ("bs_gemm.cu",)), ("bf16_gemm", ("bs_gemm.cu",)),
)


def kernel_source_hash(label=None, names=None, read=None):
    """sha256 (first 16 hex) of the kernel sources: of every file in csrc/, or,
    for a bench label, of its translation units + api.cu + the headers.
    `names` / `read` give another source state (file list, name -> bytes)."""
    names = sorted(names if names is not None else os.listdir(CSRC))
    if read is None:
        def read(name):
            with open(os.path.join(CSRC, name), "rb") as f:
                return f.read()
    if label is not None:
        tus = next((t for prefix, t in KERNEL_TUS if label.startswith(prefix)), None)
        if tus is not None:
            names = [n for n in names if n in tus or n == "api.cu" or n.endswith((".cuh", ".h"))]
    h = hashlib.sha256()
    for name in names:
        h.update(read(name))
    return h.hexdigest()[:16]


def read_traffic(label):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current sources of this label's kernels."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash(label)
    with open(p) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.rstrip("\n").split("\t")
            if len(parts) >= 3 and parts[0] == label and parts[1] == cur:
                return float(parts[2])
    return None


# ----------------------------------------------------------------- ranks
class Ranks:
    """Rank layout of a run under torchrun (RANK / WORLD_SIZE / LOCAL_RANK)
    and the host-side collectives of a replicas-only job: every rank runs its
    own copy of the step; ranks meet only at the barriers around a timed
    region and in the max over ranks of its duration.  `backend` "nccl" on
    GPUs, "gloo" for CPU tests; a single rank needs no process group."""

    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1 and backend is not None:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x, device="cpu"):
        """Max over ranks of a float (a timed region's duration)."""
        if self.dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def emit(self, out, file=None):
        """Rank 0 prints the job's one JSON line."""
        if self.rank == 0:
            print(json.dumps(out), file=file or sys.stdout, flush=True)

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def job_tflops(world, flops_per_replica, ms_step):
    """Whole-job throughput of `world` replicas, each doing flops_per_replica
    per step, when a step takes ms_step (the max over ranks): TFLOP/s."""
    return world * flops_per_replica / (ms_step / 1e3) / 1e12


# ----------------------------------------------------------------- GPU arm
def time_each(launches, K2, stream):
    """Per-launch device time (ms, mean of K2 runs) of a list of (label,
    callable).  Preferred: a graph of the launches with an event pair
    captured around every launch, replayed K2 times (no host launch gaps
    inside the pairs); where this PyTorch cannot capture events, eager runs
    with an event pair around every launch on the launching stream."""
    import torch
    try:
        pairs = [(lab, torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True)) for lab, _ in launches]
        fns = dict(launches)
        tgraph = torch.cuda.CUDAGraph()
        tside = torch.cuda.Stream()
        tside.wait_stream(stream)
        with torch.cuda.stream(tside):
            with torch.cuda.graph(tgraph, stream=tside, capture_error_mode="relaxed"):
                for lab, a, b in pairs:
                    a.record()
                    fns[lab]()
                    b.record()
        stream.wait_stream(tside)
        tgraph.replay()
        torch.cuda.synchronize()
        acc = {lab: 0.0 for lab, _ in launches}
        for _ in range(K2):
            tgraph.replay()
            torch.cuda.synchronize()
            for lab, a, b in pairs:
                acc[lab] += a.elapsed_time(b)
        return ({lab: v / K2 for lab, v in acc.items()},
                f"{K2} replays of a graph of the launches with captured CUDA events around each launch")
    except (TypeError, RuntimeError):
        pass
    ev = {lab: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K2)] for lab, _ in launches}
    torch.cuda.synchronize()
    for i in range(K2):
        for lab, fn in launches:
            a, b = ev[lab][i]
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return ({lab: statistics.mean(a.elapsed_time(b) for a, b in prs) for lab, prs in ev.items()},
            f"{K2} eager runs, CUDA events around each launch")


# Nominal dense tensor rates per GPU (TFLOP/s) quoted as context: 4.5 PF FP8 and
# 9 PF FP4 (the dense FP8 / FP4 peaks the GEMM fractions are also given
# against), 2.25 PF BF16.
NOMINAL_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0, "fp4": 9000.0}


def rate_row(lab, kind, work, ms, peaks):
    """One breakdown entry: achieved rate against the measured peak.  The
    kernels are timed alone, each inside a sub-second region, so a
    contraction's peak is the burst bf16 figure times the nominal dtype
    ratio; its fraction of the nominal dense rate is given beside it."""
    s = ms / 1e3
    if kind == "hbm":
        ach, peak, unit = work / s / 1e9, peaks["hbm"], "GB/s"
    else:
        ach, peak, unit = work / s / 1e12, peaks["bf16"] * RATIO[kind], "TFLOP/s"
    row = {"kernel": lab, "us": round(ms * 1e3, 2), "achieved": round(ach, 1), "unit": unit,
           "peak": round(peak, 1), "frac": round(ach / peak, 4)}
    if kind != "hbm":
        row["frac_nominal"] = round(ach / NOMINAL_TFLOPS[kind], 4)
    return row


def graph_ms(launches, reps, stream):
    """Mean device time (ms) of one pass over `launches`, from `reps` replays
    of a CUDA graph of them between two events on the launching stream."""
    import torch
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side, capture_error_mode="relaxed"):
            for _, fn in launches:
                fn()
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def time_part(part, K2, stream, peaks, check_errors, key):
    """Warm-up, per-launch timing (time_each) and the breakdown rows of one
    part measured beside the step; returns (rows, launches per pass, from)."""
    import torch
    fl = part.launches()
    for _ in range(3):
        for _, fn in fl:
            fn()
    torch.cuda.synchronize()
    check_errors(f"in the {key} warm-up")
    fper, ffrom = time_each(fl, K2, stream)
    check_errors(f"in the {key} timing")
    fplan = {lab: (kind, w) for lab, kind, w in part.plan()}
    rows = [rate_row(lab, *fplan[lab], ms, peaks) for lab, ms in fper.items()]
    return rows, sum(getattr(part, "KERNELS", {}).get(lab, 1) for lab, _ in fl), ffrom


def run_dsv3(step, K2, stream, peaks, check_errors):
    """The DeepSeek-V3-shaped MoE layer as its own step: routed-expert
    TFLOP/s over the whole layer's time (graph replays), the per-kernel
    breakdown, and the fraction of its roofline bound max(FLOPs / FP4 peak,
    bytes / HBM peak); the MXFP8 shared expert beside it."""
    d = Dsv3Moe(step)
    lay = d.layer
    rows, nlaunch, ffrom = time_part(d, K2, stream, peaks, check_errors, "dsv3 layer")
    reps = max(3, min(K2, 30))
    ms = graph_ms(d.launches(), reps, stream)
    check_errors("in the dsv3 step timing")
    flops = lay.gemm_flops()
    bytes_ = lay.bytes_moved()
    t_c = flops / (peaks["bf16"] * RATIO["fp4"] * 1e12)
    t_b = bytes_ / (peaks["hbm"] * 1e9)
    bound = max(t_c, t_b)
    shared = Dsv3SharedExpert(d)
    srows, snl, _ = time_part(shared, K2, stream, peaks, check_errors, "dsv3 shared expert")
    sms = graph_ms(shared.launches(), reps, stream)
    sfl = sum(w for _, kind, w in shared.plan() if kind == "fp8")
    out = {
        "workload": "DeepSeek-V3-shaped routed-expert layer, per-token NVFP4: 16384 tokens, hidden 7168, "
                    "256 experts, FFN 2048, top-8 Zipf(1.1), 0.5% of activations x100 (131072 dispatched rows)",
        "ms_per_step": round(ms, 4), "steps": reps, "value": round(flops / (ms / 1e3) / 1e12, 2),
        "unit": "TFLOP/s", "gemm_flops_per_step": flops, "algorithmic_bytes_per_step": bytes_,
        "roofline": {"bound_ms": round(bound * 1e3, 4), "by": "hbm" if t_b > t_c else "fp4",
                     "compute_ms": round(t_c * 1e3, 4), "bytes_ms": round(t_b * 1e3, 4),
                     "frac": round(bound / (ms / 1e3), 4)},
        "breakdown": rows, "breakdown_from": ffrom,
        "shared_expert_mxfp8": {"ms_per_step": round(sms, 4), "value": round(sfl / (sms / 1e3) / 1e12, 2),
                                "unit": "TFLOP/s", "gemm_flops_per_step": sfl, "breakdown": srows},
    }
    launches = nlaunch * (K2 + 3 + reps + 1) + snl * (K2 + 3 + reps + 1)
    del d, shared
    return out, launches


SWEEP = ((1 << 20, 2048), (1 << 24, 4096), (1 << 27, 7168), (1 << 30, 2048))


def run_sweep(step, reps, stream, peaks, check_errors):
    """Quantizer bandwidth sweep, 2^20 .. 2^30 bf16 elements of the sweep's
    value mix: MXFP8 rowwise + columnwise (4.0625 B per element) and NVFP4
    per token (2.5625 B per element + 4 B per row).  Each launch is timed
    alone between CUDA events, after a 512 MB write that evicts L2, so
    every size streams from HBM."""
    import torch
    mx = step.mx
    from moe_mx8_quantize_gb300 import inputs
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=step.dev)
    out, launches = [], 0
    for numel, cols in SWEEP:
        rows = max(128, (numel // cols) // 128 * 128)
        x = inputs.sweep(rows, cols, seed=4 + numel.bit_length(), device=step.dev)
        n = rows * cols
        u8 = lambda k: torch.empty(max(k, 16), dtype=torch.uint8, device=step.dev)
        qr, qc = u8(n).view(-1)[:n].view(rows, cols), u8(n)[:n].view(cols, rows)
        sr, sc = u8(mx.scale_bytes(mx.FMT_MXFP8, rows, cols)), u8(mx.scale_bytes(mx.FMT_MXFP8, cols, rows))
        q4, s4 = u8(n // 2)[: n // 2].view(rows, cols // 2), u8(mx.scale_bytes(mx.FMT_NVFP4, rows, cols))
        s32 = torch.empty(rows, dtype=torch.float32, device=step.dev)
        kinds = (("mxfp8_quant_rc", 4.0625 * n,
                  lambda: mx.mx8_quantize_into(x, qr, sr, qc, sc, mx.ROWWISE | mx.COLWISE, step.ws)),
                 ("nvfp4_quant_token", 2.5625 * n + 4 * rows,
                  lambda: mx.nvfp4_quantize_into(x, q4, s4, s32, mx.SCOPE_TOKEN, None, step.ws)))
        for name, work, fn in kinds:
            for _ in range(2):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for a, b in ev:
                flush.fill_(1)
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            check_errors(f"in the sweep ({name}, {numel})")
            ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
            row = rate_row(name, "hbm", work, ms, peaks)
            row.update({"elements": n, "rows": rows, "cols": cols})
            out.append(row)
            launches += reps + 2
        del x, qr, qc, sr, sc, q4, s4, s32
    del flush
    return {"rows": out, "from": f"{reps} launches per point, each alone between CUDA events after a "
                                  f"512 MB write that evicts L2"}, launches


def run_gpu(args):
    import torch
    import __graft_entry__
    import moe_mx8_quantize_gb300 as mx

    ranks = Ranks("nccl")
    world, rank, local = ranks.world, ranks.rank, ranks.local
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build() if rank == 0 or world == 1 else None
    if world > 1:
        ranks.barrier()
        mx.load()
    step = Step(dev, seed_base=0)
    launches = step.launches()
    plan = {lab: (kind, w) for lab, kind, w in step.plan()}
    stream = torch.cuda.current_stream()

    barrier = ranks.barrier

    # warm-up (eager), then capture one step as a CUDA graph
    def eager_step():
        for _, fn in launches:
            fn()

    def check_errors(when):
        for ws in step.workspaces():
            st = mx.check_device_error(ws)
            if st != mx.OK:
                raise RuntimeError(f"device error {when}: {mx.status_string(st)}")

    assert sorted(l for b in step.BRANCHES for l in b) == sorted(l for l, _ in launches)
    for _ in range(args.warmup):
        eager_step()
    torch.cuda.synchronize()
    check_errors("after warm-up")
    # the step as a CUDA graph, its launches in order on one stream.  (Capturing
    # the three independent branches on three streams measured slower: the
    # persistent kernels already fill the GPU, and the group-scope quantizer's
    # second read loses its L2 residency to the concurrent branches.)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side, capture_error_mode="relaxed"):
            eager_step()
    stream.wait_stream(side)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()

    # timed region 1: K graph replays (the step time and `value`)
    K = args.steps
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    check_errors("in timed region")
    total_ms = ranks.max(total_ms, dev)
    ms_step = total_ms / K

    # timed region 2: the per-kernel durations of the breakdown and the
    # roofline (see time_each)
    K2 = max(3, min(K, 100))
    per, breakdown_from = time_each(launches, K2, stream)
    check_errors("in the per-kernel timing")
    peaks = load_peaks()
    breakdown = [rate_row(lab, *plan[lab], ms, peaks) for lab, ms in per.items()]
    dom = max(breakdown, key=lambda b: b["us"])
    dkind, dwork = plan[dom["kernel"]]
    traffic = read_traffic(dom["kernel"])
    roofline = {"kernel": dom["kernel"], "bound": "hbm" if dkind == "hbm" else "tensor",
                "achieved": dom["achieved"], "peak": dom["peak"], "unit": dom["unit"],
                "frac": dom["frac"], "traffic": traffic,
                "algorithmic": dwork, "peak_source": f"{peaks['source']} "
                + ("hbm copy" if dkind == "hbm" else f"bf16 burst x {RATIO[dkind]:g} ({dkind} nominal ratio)")}

    flops = step.gemm_flops()
    value = job_tflops(world, flops, ms_step)
    launches_per_step = sum(Step.KERNELS_PER_LABEL.get(lab, 1) for lab, _ in launches)
    gpu_launches = launches_per_step * (K + K2)

    # timed region 3: the MXFP4 linear layer, the dequantized-backward BF16
    # GEMMs and the NVFP4 recipe variants, beside the step (each in its own
    # graph with event pairs); then the DeepSeek-V3-shaped MoE layer and the
    # quantizer bandwidth sweep, each its own timed region
    extra = None
    if not args.no_extra:
        extra = {}
        for key, part in (("mxfp4_linear", Mxfp4Linear(step)), ("dequantized_backward", DequantBackward(step)),
                          ("nvfp4_recipe_linear", Nvfp4RecipeLinear(step)), ("moe_gate_up_quant_h", FusedQuantH(step))):
            extra[key], nl, extra["from"] = time_part(part, K2, stream, peaks, check_errors, key)
            gpu_launches += nl * (K2 + 3)
        extra["dsv3_moe_layer"], nl = run_dsv3(step, K2, stream, peaks, check_errors)
        gpu_launches += nl
        extra["quantizer_sweep"], nl = run_sweep(step, 10, stream, peaks, check_errors)
        gpu_launches += nl

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, args, ranks, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(args.cpu_seconds)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/e2m1 block-scaled, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemm_flops_per_step": flops,
                   "l2": "inputs larger than L2 (step working set ~2.7 GB of HBM; no flush)",
                   "value_definition": "block-scaled GEMM FLOPs / step time incl. quantizers",
                   "parallelism": f"replicas x{world} (no data-path collective)"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": gpu_launches, "breakdown": breakdown, "extra": extra,
        "timing": {"value_from": f"{K} CUDA-graph replays of the step",
                   "breakdown_from": breakdown_from,
                   "kernels_sum_ms_per_step": round(sum(b["us"] for b in breakdown) / 1e3, 4)},
    }
    ranks.emit(out)
    ranks.close()


def run_e2e(step, args, ranks, dev):
    """Same step through the public API with host buffers: every step copies
    its inputs (X, dY, the MoE layer's token activations) from pinned host memory
    and reads its results (Y, dX, NVFP4 Y, the combined MoE output) back; weights stay
    resident.  The three branches run on their own streams, each copying its
    own inputs in and results out, so one branch's copies overlap another's
    kernels."""
    import torch
    step.setup_io()
    streams = [torch.cuda.current_stream()] + [torch.cuda.Stream() for _ in step.BRANCHES[1:]]
    stream = streams[0]
    K = max(3, min(args.steps, 50))
    for _ in range(2):
        step.run_concurrent(streams, io=True)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    ranks.barrier()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(K):
        step.run_concurrent(streams, io=True)
    b.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    ms = ranks.max(a.elapsed_time(b), dev) / K
    bi = sum(h.numel() * h.element_size() for br in step.io_in for _, h in br)
    bo = sum(h.numel() * h.element_size() for br in step.io_out for _, h in br)
    return {"value": round(job_tflops(ranks.world, step.gemm_flops(), ms), 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": K, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}


# ----------------------------------------------------------------- CPU oracle
def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


STEP_FLOPS = (2.0 * 2048 * 8192 * 2048 * 4 + 2.0 * 32768 * 1536 * 2048 + 2.0 * 32768 * 2048 * 768)


def oracle_step_seconds(budget_s, threads=1):
    """Times the oracle on a bounded sample of every operation of the step and
    extrapolates (per element / per output) to the full step.  With threads >
    1 each thread runs the single-thread sample on its own slab (the C
    oracle releases the interpreter lock), so the sample grows with the
    threads.  Returns (seconds for one full step, description of the sample,
    wall seconds of the sample)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import torch
    import oracle
    from moe_mx8_quantize_gb300 import inputs

    oracle.build()
    T, H, O = LINEAR["tokens"], LINEAR["in_features"], LINEAR["out_features"]
    E, F, R = QWEN["experts"], QWEN["ffn"], QWEN["tokens"] * QWEN["topk"]
    g = torch.Generator().manual_seed(7)
    # the 64-row / 0.02%-of-outputs sample takes about 3.5 s on one core;
    # scale it to the requested budget
    factor = max(budget_s / 3.5, 0.02)
    rows = max(32, int(round(64 * factor / 32)) * 32)   # colwise blocks need 32-row slabs
    frac_gemm = 0.0002 * factor
    pool = ThreadPoolExecutor(threads) if threads > 1 else None

    def par(fn, items):
        if pool is None:
            for it in items:
                fn(it)
        else:
            list(pool.map(fn, items))

    def slab(r, c, std=1.0):
        return inputs.bits(inputs.normal_bf16((r, c), std, g, "cpu"))

    def slabs(r, c):
        return [slab(r, c) for _ in range(threads)]

    total = 0.0
    t_wall = time.perf_counter()

    def timed(fn):
        t = time.perf_counter()
        fn()
        return time.perf_counter() - t

    # MXFP8 rowwise + colwise quantization: `rows`-row slabs, scaled per element
    for name, (r, c) in {"X": (T, H), "W": (O, H), "dY": (T, O)}.items():
        xs = slabs(rows, c)
        s = timed(lambda: par(lambda x: (oracle.mxfp8_quantize_rowwise(x), oracle.mxfp8_quantize_colwise(x)), xs))
        total += s * (r * c) / (threads * rows * c)
    # dequantize X^, W^
    qs = [oracle.mxfp8_quantize_rowwise(x) for x in slabs(rows, H)]
    s = timed(lambda: par(lambda qq: oracle.dequant_mxfp8(*qq), qs))
    total += s * (T * H + O * H) / (threads * rows * H)
    # NVFP4 quantizers (token scope cost per element also bounds group/tensor)
    for r, c in ((T, H), (O, H), (QWEN["tokens"], H), (E * 2 * F, H), (E * H, F), (R, F)):
        xs = slabs(rows, c)
        s = timed(lambda: par(oracle.nvfp4_quantize, xs))
        total += s * (r * c) / (threads * rows * c)
    # SwiGLU
    gus = slabs(rows, 2 * F)
    s = timed(lambda: par(oracle.swiglu, gus))
    total += s * R / (threads * rows)
    # combine: `rows` tokens of 8 choices each
    yys = slabs(rows * 8, H)
    rws = np.arange(rows * 8, dtype=np.int64).reshape(rows, 8)
    ww = np.full((rows, 8), 0.125, np.float32)
    s = timed(lambda: par(lambda yy: oracle.moe_combine(yy, rws, ww), yys))
    total += s * QWEN["tokens"] / (threads * rows)
    # GEMMs: sampled outputs, scaled per output
    rng = np.random.default_rng(0)
    for fmt, (M, N, K) in ((0, (T, O, H)), (0, (T, H, O)), (0, (O, H, T)), (1, (T, O, H)),
                           (1, (R, 2 * F, H)), (1, (R, H, F))):
        n_out = max(32, int(M * N * frac_gemm))
        a = slab(32, K)
        b = slab(64, K)
        if fmt == 0:
            A, SA = oracle.mxfp8_quantize_rowwise(a)
            B, SB = oracle.mxfp8_quantize_rowwise(b)
            a32 = b32 = None
        else:
            A, SA, a32 = oracle.nvfp4_quantize(a)
            B, SB, b32 = oracle.nvfp4_quantize(b)
        work = []
        for _ in range(threads):
            pairs = np.stack([rng.integers(0, 32, n_out), rng.integers(0, 64, n_out)], 1)
            work.append(pairs[np.argsort(pairs[:, 0], kind="stable")])
        s = timed(lambda: par(lambda pr: oracle.gemm_ref(fmt, A, SA, B, SB, K, a32, b32, pairs=pr), work))
        total += s * (M * N) / (threads * n_out)
    wall = time.perf_counter() - t_wall
    if pool is not None:
        pool.shutdown()
    desc = (f"{threads} thread(s), each: quantizers/dequant/SwiGLU on {rows}-row slabs of every tensor, GEMMs on "
            f"sampled outputs ({frac_gemm * 100:.4f}% of each); extrapolated per element/output to the full step")
    return total, desc, wall


def oracle_baseline(budget_s):
    """The oracle timed on the host cores, single-threaded and on all cores."""
    import __graft_entry__  # noqa: F401  (sys.path)
    cores = os.cpu_count() or 1
    secs1, sample1, wall1 = oracle_step_seconds(budget_s, 1)
    secsn, samplen, walln = oracle_step_seconds(budget_s, cores) if cores > 1 else (secs1, sample1, wall1)
    return {"value": round(STEP_FLOPS / secsn / 1e12, 8), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": samplen, "sample_wall_s": round(walln, 2), "est_full_step_s": round(secsn, 2),
            "single_thread": {"value": round(STEP_FLOPS / secs1 / 1e12, 8), "cores": 1, "sample": sample1,
                              "sample_wall_s": round(wall1, 2), "est_full_step_s": round(secs1, 2)},
            "cores_available": os.cpu_count(), "cpu": cpu_model()}


def run_reference(args):
    # the oracle on the host cores: rank 0 alone runs and prints; under
    # torchrun the other ranks exit at once without work
    ranks = Ranks()
    world = ranks.world
    if ranks.rank != 0:
        return
    K = args.steps
    cores = os.cpu_count() or 1
    # each step times a bounded sample of the step's work on all host cores,
    # sized so the whole run stays near two minutes
    per_step = min(args.cpu_seconds / 4, 120.0 / max(1, K + args.warmup))
    for _ in range(args.warmup):
        oracle_step_seconds(per_step, cores)
    t0 = time.perf_counter()
    est, walls = [], []
    desc = ""
    for _ in range(K):
        secs, desc, wall = oracle_step_seconds(per_step, cores)
        est.append(secs)
        walls.append(wall)
    total_wall = time.perf_counter() - t0
    secs = statistics.mean(est)
    value = STEP_FLOPS / secs / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "TFLOP/s",
           "n_gpus": world, "steps": K, "warmup": args.warmup,
           "ms_per_step": round(statistics.mean(walls) * 1e3, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64 oracle (decoded e4m3/e2m1 operands)", "data": "synthetic",
           "config": {"workload": WORKLOAD, "sampled": True},
           "timing": {"ms_per_step": "measured wall time of one sampled step (a bounded sample of every "
                                     "operation of the step), not of the full step",
                      "value": "throughput of the sample, extrapolated per element / output: full-step "
                               "FLOPs over the estimated full-step time",
                      "est_full_step_ms": round(secs * 1e3, 1), "wall_s": round(total_wall, 2)},
           "cpu_baseline": {"kind": "oracle", "cores": cores, "value": round(value, 8), "sample": desc,
                            "cpu": cpu_model()},
           "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    ranks.emit(out)


def run_profile(args):
    """For ncu: every launch of the step and of the parts timed beside it
    (not the DeepSeek-V3 layer or the sweep, whose kernels are the step's at
    other shapes), once as warm-up and once more to be captured
    (`ncu --launch-skip` = the launches of the first pass).  Prints the labels
    in launch order with their kernel counts."""
    import torch
    import __graft_entry__
    import moe_mx8_quantize_gb300 as mx
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    step = Step(dev)
    parts = [("step", step, step.launches(), Step.KERNELS_PER_LABEL),
             ("mxfp4_linear", None, None, {}), ("dequantized_backward", None, None, {}),
             ("nvfp4_recipe_linear", None, None, Nvfp4RecipeLinear.KERNELS), ("moe_gate_up_quant_h", None, None, {})]
    objs = {"mxfp4_linear": Mxfp4Linear, "dequantized_backward": DequantBackward,
            "nvfp4_recipe_linear": Nvfp4RecipeLinear, "moe_gate_up_quant_h": FusedQuantH}
    seq = []
    for name, obj, fl, kern in parts:
        if obj is None:
            obj = objs[name](step)
            fl = obj.launches()
        seq += [(f"{name}: {lab}", fn, kern.get(lab, 1)) for lab, fn in fl]
    for _ in range(2):
        for _, fn, _ in seq:
            fn()
        torch.cuda.synchronize()
    for ws in step.workspaces():
        if mx.check_device_error(ws) != mx.OK:
            raise RuntimeError("device error in the profile pass")
    print(json.dumps({"kernels_per_pass": sum(k for _, _, k in seq),
                      "launches": [[lab, k] for lab, _, k in seq]}))


def run_profile_case(args):
    """For ncu: one launch of the DeepSeek-V3-shaped kernels on synthetic
    operands, sized for a capture --
      dsv3_gemms: the gate|up (SwiGLU) and down grouped NVFP4 GEMMs at the
        full layer shape (131072 dispatched rows, Zipf(1.1) routing over 256
        experts, hidden 7168, FFN 2048), random E2M1 codes and E4M3 block
        scales of 1.0 (about 9 GB on the device);
      dsv3_wgu: group-scope NVFP4 quantization of 24 experts' gate|up weights
        ([4096, 7168] bf16 each, 1.4 GB)."""
    import torch
    import __graft_entry__
    import moe_mx8_quantize_gb300 as mx
    from moe_mx8_quantize_gb300 import inputs
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q = inputs.DSV3_SHAPE
    T, H, E, F, k = q["tokens"], q["hidden"], q["experts"], q["ffn"], q["topk"]
    if args.profile_case == "dsv3_gemms":
        ids = inputs.route_zipf(T, E, k, 1.1, torch.Generator(device="cpu").manual_seed(3), "cpu")
        offs = inputs.dispatch(ids, E).offsets.to(dev)
        R = T * k
        u8 = lambda n: torch.randint(0, 256, (n,), dtype=torch.uint8, device=dev)
        sc = lambda n: torch.full((n,), 0x38, dtype=torch.uint8, device=dev)
        A4, SA4 = u8(R * H // 2).view(R, H // 2), sc(mx.scale_bytes_grouped(mx.FMT_NVFP4, R, E, H))
        W4, SW4 = u8(E * 2 * F * H // 2).view(E, 2 * F, H // 2), sc(mx.scale_bytes(mx.FMT_NVFP4, E * 2 * F, H))
        H4, SH4 = u8(R * F // 2).view(R, F // 2), sc(mx.scale_bytes_grouped(mx.FMT_NVFP4, R, E, F))
        Wd4, SWd4 = u8(E * H * F // 2).view(E, H, F // 2), sc(mx.scale_bytes(mx.FMT_NVFP4, E * H, F))
        A32, W32 = torch.full((R,), 0.01, device=dev), torch.full((E,), 0.01, device=dev)
        hs = torch.empty((R, F), dtype=torch.bfloat16, device=dev)
        out = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        ws = mx.new_workspace(E, dev)
        mx.bs_grouped_gemm_fused_into(mx.FMT_NVFP4, offs, R, A4, SA4, W4, SW4, H, hs, A32, W32, None,
                                      mx.EPI_SWIGLU, ws)
        mx.bs_grouped_gemm_into(mx.FMT_NVFP4, offs, H4, SH4, Wd4, SWd4, F, out, A32, W32, ws)
    elif args.profile_case == "dsv3_wgu":
        n = 24
        W = inputs.normal_bf16((n * 2 * F, H), 0.02, torch.Generator(device="cuda").manual_seed(5), "cuda")
        offs = torch.arange(n + 1, device=dev, dtype=torch.int64) * (2 * F)
        qw = torch.empty((n * 2 * F, H // 2), dtype=torch.uint8, device=dev)
        sw = torch.empty(mx.scale_bytes(mx.FMT_NVFP4, n * 2 * F, H), dtype=torch.uint8, device=dev)
        s32 = torch.empty(n, dtype=torch.float32, device=dev)
        ws = mx.new_workspace(n, dev)
        mx.nvfp4_quantize_into(W, qw, sw, s32, mx.SCOPE_GROUP, offs, ws)
    else:
        raise SystemExit(f"unknown profile case {args.profile_case}")
    torch.cuda.synchronize()
    if mx.check_device_error(ws) != mx.OK:
        raise RuntimeError("device error in the profile case")
    print(json.dumps({"case": args.profile_case, "device_gb": round(torch.cuda.memory_allocated() / 1e9, 2)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mx8q", choices=["mx8q", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the measurements beside the step")
    ap.add_argument("--profile", action="store_true", help="run every launch twice for ncu and exit")
    ap.add_argument("--profile-case", choices=["dsv3_gemms", "dsv3_wgu"],
                    help="run one DeepSeek-V3-shaped kernel case once for ncu and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
    elif args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
