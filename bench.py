#!/usr/bin/env python
"""Benchmark of the 4-bit MoE expert-layer step on B300.

One step = one pass of the whole hot path over one batch of the Inkling-shaped layer (16384
tokens, d_model 4096, SwiGLU width 2048, 384 experts, top-8 of N(0,1) logits plus a per-expert
N(0,1) bias, Student-t(3) activations, N(0, 0.02) expert weights held as FP32 masters):

  forward   top-k routing and dispatch plan; NVFP4 (Four Over Six) quantisation of X, of every
            expert's gate/up and down weights (per-expert scales; the weight path pipelined over
            expert chunks on two streams) and of H; NVFP4 row gather; grouped NVFP4 GEMMs (gate/up
            with the SwiGLU and the amax of H in its last stage, then down); Hadamard(128) NVFP4
            return-path encode (its amax from the down GEMM), then decode and weighted combine in
            one pass;
  backward  combine gradient; MXFP8 quantisation of dY and dGU (row-wise and transposed);
            dequantise -> transpose -> MXFP8 requantisation with Philox stochastic rounding of
            W_down, H, W_gate/up and X; grouped MXFP8 dgrad (row-grouped) and wgrad
            (contraction-grouped) GEMMs for both projections; SwiGLU backward; SGD on the FP32
            master weights, fused into the weight-gradient GEMMs (the next step quantises the
            masters, rounded to bf16 as they are read); the dispatch's gradient (each token's k
            rows of dX summed back into token order).

`value` is expert-GEMM TFLOP/s of the whole step: the algorithmic FLOPs of the six expert GEMMs
(routed rows only) divided by the device time of the step.  The JSON line also carries per-kernel
times, the requantisation GB/s, the roofline of the dominant kernel, clocks, the end-to-end
number through the C ABI with host buffers, and the CPU oracle's rate on a bounded sample.

`--impl reference` times the oracle (the plain CPU definition of the method) on a bounded sample
of the same workload: one expert with one 128-row tile of routed tokens, through every step.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

# The oracle legs (the reference arm and the CPU baseline) run on one host thread: their float64
# matmuls are held to one BLAS thread, which has to be fixed before numpy loads its BLAS.
if "--impl=reference" in sys.argv or "--cpu-leg" in sys.argv or (
        "--impl" in sys.argv and sys.argv[sys.argv.index("--impl") + 1:][:1] == ["reference"]):
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

T_TOK, D_MODEL, D_FF, N_EXP, TOP_K = 16384, 4096, 2048, 384, 8
WORKLOAD = "inkling-moe-layer-step: T=16384 d=4096 f=2048 E=384 top8, NVFP4 fwd + MXFP8 bwd + SGD"
SMALL = dict(T=4096, d=2048, f=1024, E=8, k=2)
METRIC = "expert NVFP4 GEMM TFLOPS + requant GB/s, as % of B300 roofline"
LR = 1e-3
WEIGHT_CHUNKS = 4  # expert chunks per projection in the weight path's pipeline
# DRAM bytes per step of the kernel groups, read + written, from a one-pass ncu capture of this
# layer step at full size (dram__bytes_read.sum + dram__bytes_write.sum of the group's launches,
# averaged over the two timed steps): profiles/layer_step_dram_bytes.md.  A kernel changed since
# its capture has no entry.
DRAM_PER_STEP = {"gemm_mxfp8_wgrad_sgd": 72.182e9}
MULTI_KERNEL_GROUPS = {"quant_w", "route", "quant_x", "hadamard", "mxfp8_quant"}
GROUP_LAUNCHES = {"gemm_mxfp8_wgrad_sgd": 2, "requant": 2, "gemm_nvfp4": 2, "gemm_mxfp8_dgrad": 2,
                  "quant_w": 4 * WEIGHT_CHUNKS}  # two launches per chunk, WEIGHT_CHUNKS chunks per projection


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"], src="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


# ---------------------------------------------------------------------------------------------
# the device step
# ---------------------------------------------------------------------------------------------
def weight_chunk_bounds(E):
    """Expert bounds of the weight path's chunks, gate/up then down: WEIGHT_CHUNKS equal chunks."""
    even = [E * i // WEIGHT_CHUNKS for i in range(WEIGHT_CHUNKS + 1)]
    return even, even


class LayerStep:
    """All device buffers of one layer step and the sequence of library calls."""

    def __init__(self, T, d, f, E, k, device, seed_workload=5):
        import torch
        from precision_moe_numerics_03_b300 import inputs, moe4
        self.torch, self.m = torch, moe4
        self.T, self.d, self.f, self.E, self.k = T, d, f, E, k
        self.dev = device
        dev = device
        u8 = dict(dtype=torch.uint8, device=dev)
        self.rows_cap = (T * k + 127 * E + 127) // 128 * 128
        R = self.rows_cap
        g = lambda s: inputs.device_generator(seed_workload, s, dev)
        # inputs of a step
        self.X = inputs.device_student_t((T, d), g(0), dev).view(torch.int16)
        lg = torch.randn((T, E), generator=g(1), device=dev)
        bias = torch.randn((E,), generator=g(2), device=dev)
        self.logits = (lg + bias).contiguous()
        self.dy = inputs.device_normal((T, d), 1.0, g(3), dev).view(torch.int16)
        # FP32 master weights and their bf16 copies
        self.W32_gu = torch.randn((E, 2 * f, d), generator=g(4), device=dev).mul_(0.02)
        self.W32_d = torch.randn((E, d, f), generator=g(5), device=dev).mul_(0.02)
        self.Wb_gu = self.W32_gu.to(torch.bfloat16).view(torch.int16)
        self.Wb_d = self.W32_d.to(torch.bfloat16).view(torch.int16)
        # per-expert amax of the bf16 copies: written by the fused wgrad + SGD epilogue of each step
        # and read by the next step's weight quantisation (here seeded for the first step)
        self.amax_h = torch.zeros(1, dtype=torch.float32, device=dev)
        self.amax_y = torch.zeros(1, dtype=torch.float32, device=dev)
        self.amax_gu = self.Wb_gu.view(torch.bfloat16).view(E, -1).abs().amax(dim=1).float().contiguous()
        self.amax_d = self.Wb_d.view(torch.bfloat16).view(E, -1).abs().amax(dim=1).float().contiguous()
        # routing
        self.idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.row_of = torch.empty((T, k), dtype=torch.int32, device=dev)
        # the weight path's side stream (higher priority: its quantiser's CTAs are placed first)
        self.side = torch.cuda.Stream(device=dev, priority=-1)
        self.ev_fork = torch.cuda.Event()
        self.n_wchunks = sum(len(b) - 1 for b in weight_chunk_bounds(E))
        self.ev_q = [torch.cuda.Event() for _ in range(self.n_wchunks)]
        self.src_of = torch.empty(R, dtype=torch.int32, device=dev)
        self.plan_ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_PERMUTE_PLAN, T, k, E), dev)
        self.qws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, E), dev)
        self.hws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT), dev)
        # forward tensors
        self.Xq_c, self.Xq_s = torch.empty((T, d // 2), **u8), torch.empty((T, d // 16), **u8)
        self.Xq_g = torch.empty(1, dtype=torch.float32, device=dev)
        self.Xp_c, self.Xp_s = torch.empty((R, d // 2), **u8), torch.empty((R, d // 16), **u8)
        self.Wgu_c, self.Wgu_s = torch.empty((E, 2 * f, d // 2), **u8), torch.empty((E, 2 * f, d // 16), **u8)
        self.Wgu_g = torch.empty(E, dtype=torch.float32, device=dev)
        self.Wd_c, self.Wd_s = torch.empty((E, d, f // 2), **u8), torch.empty((E, d, f // 16), **u8)
        self.Wd_g = torch.empty(E, dtype=torch.float32, device=dev)
        self.GU = torch.empty((R, 2 * f), dtype=torch.float32, device=dev)
        self.H = torch.empty((R, f), dtype=torch.int16, device=dev)
        self.Hq_c, self.Hq_s = torch.empty((R, f // 2), **u8), torch.empty((R, f // 16), **u8)
        self.Hq_g = torch.empty(1, dtype=torch.float32, device=dev)
        self.Y = torch.empty((R, d), dtype=torch.int16, device=dev)
        self.Yc_c, self.Yc_s = torch.empty((R, d // 2), **u8), torch.empty((R, d // 16), **u8)
        self.Yc_g = torch.empty(1, dtype=torch.float32, device=dev)
        self.Yhat = torch.empty((R, d), dtype=torch.int16, device=dev)
        self.y = torch.empty((T, d), dtype=torch.int16, device=dev)
        # backward tensors
        self.dYr_q, self.dYr_e = torch.empty((R, d), **u8), torch.empty((R, d // 32), **u8)
        self.dYc_q, self.dYc_e = torch.empty(d * R, **u8), torch.empty(d * R // 32, **u8)
        self.WdT_q, self.WdT_e = torch.empty((E, f, d), **u8), torch.empty((E, f, d // 32), **u8)
        self.HqT_q, self.HqT_e = torch.empty(f * R, **u8), torch.empty(f * R // 32, **u8)
        self.dH = torch.empty((R, f), dtype=torch.float32, device=dev)
        self.dGU = torch.empty((R, 2 * f), dtype=torch.int16, device=dev)
        self.dGUr_q, self.dGUr_e = torch.empty((R, 2 * f), **u8), torch.empty((R, 2 * f // 32), **u8)
        self.dGUc_q, self.dGUc_e = torch.empty(2 * f * R, **u8), torch.empty(2 * f * R // 32, **u8)
        self.WguT_q, self.WguT_e = torch.empty((E, d, 2 * f), **u8), torch.empty((E, d, 2 * f // 32), **u8)
        self.XpT_q, self.XpT_e = torch.empty(d * R, **u8), torch.empty(d * R // 32, **u8)
        self.dXp = torch.empty((R, d), dtype=torch.int16, device=dev)
        self.dX = torch.empty((T, d), dtype=torch.int16, device=dev)
        # scratch for the GEMMs' scale-layout change (largest call)
        wsz = max(moe4.moe4_workspace_size_gemm(1, R, E, f, d), moe4.moe4_workspace_size_gemm(1, R, E, d, 2 * f),
                  moe4.moe4_workspace_size_gemm(1, d, 1, f, R), moe4.moe4_workspace_size_gemm(1, 2 * f, 1, d, R))
        self.gws = moe4.workspace(wsz, dev)
        self.Rp = None
        self.launches = 0
        self.step_index = 0

    # algorithmic FLOPs of the six expert GEMMs (routed rows only)
    def gemm_flops(self):
        rows = self.T * self.k
        fwd = 2 * rows * (2 * self.f) * self.d + 2 * rows * self.d * self.f
        return fwd, 2 * fwd

    def run(self, timer=None, io=None, ev=None):
        """One layer step; io = (X, logits, dy, y) device tensors to use instead of the step's own.
        ev (end to end): events the step's stream waits on right before the first use of each
        input ("logits", "X", "dy", all recorded after their host-to-device copies), and one it
        records as soon as y is complete ("y"), so that the copies overlap the step's own work."""
        m, torch = self.m, self.torch
        T, d, f, E, k = self.T, self.d, self.f, self.E, self.k
        FOS, MMA, OMMA = m.FOUR_OVER_SIX, m.SF_MMA_LAYOUT, m.SF_OUT_MMA
        tm = timer if timer is not None else _NullTimer()
        X, logits, dy, y = io if io is not None else (self.X, self.logits, self.dy, self.y)
        cur = torch.cuda.current_stream()
        wait = (lambda name: cur.wait_event(ev[name])) if ev is not None else (lambda name: None)
        n = 0
        seed = 1000 + self.step_index
        self.step_index += 1
        # ---------------- forward
        wait("logits")
        with tm("route"):
            m.moe4_route_topk(logits, T, E, k, self.idx, self.w)
            m.moe4_permute_plan(self.idx, T, k, E, self.offs, self.row_of, self.src_of, self.rows_cap, self.plan_ws)
        n += 4
        Rp = int(self.offs[E].item())          # host needs the padded row count (one 4-byte read)
        self.Rp = Rp
        with tm("quant_w"):
            # the FP32 master weights, rounded to bf16 as they are read (no stored bf16 copy), to
            # NVFP4 for the forward, then requantised to the MXFP8 transposes the backward's dgrad
            # reads; experts that received no rows are skipped.  Software-pipelined over expert
            # chunks: chunk i+1's quantiser (HBM-bound) runs on a side stream on part of each SM
            # while chunk i's requantiser (issue-bound) takes the rest.
            self.weight_path(seed, cur)
        n += 2 * self.n_wchunks  # each chunk: the quantiser, then the requantiser
        wait("X")  # the weight path needs none of the step's inputs: X's copy can run beside it
        with tm("quant_x"):
            m.nvfp4_quantize(X, 1, T, d, d, self.Xq_c, self.Xq_s, self.Xq_g, None, FOS, self.qws)
            m.moe4_permute_nvfp4(self.Xq_c, self.Xq_s, T, d, self.src_of, Rp, self.Xp_c, self.Xp_s, MMA)
        n += 3
        with tm("gemm_nvfp4"):
            # the gate/up projection; its last stage also forms H = SwiGLU(GU) and the amax of H
            m.grouped_expert_gemm_nvfp4_swiglu(self.Xp_c, self.Xp_s, self.Xq_g, self.Wgu_c, self.Wgu_s, self.Wgu_g,
                                               self.offs, E, Rp, f, d, self.GU, self.H, self.amax_h, MMA)
        n += 1
        with tm("quant_h"):  # H to NVFP4 in one pass, its amax from the GEMM
            m.nvfp4_quantize(self.H[:Rp], 1, Rp, f, f, self.Hq_c, self.Hq_s, self.Hq_g, self.amax_h,
                             FOS | MMA | m.AMAX_GIVEN)
        n += 1
        with tm("gemm_nvfp4"):
            # the down projection; its last stage also returns the amax of the Hadamard-rotated rows
            m.grouped_expert_gemm_nvfp4_hadamard_amax(self.Hq_c, self.Hq_s, self.Hq_g, self.Wd_c, self.Wd_s,
                                                      self.Wd_g, self.offs, E, Rp, d, f, self.Y, self.amax_y, MMA)
        n += 1
        with tm("hadamard"):  # the NVFP4 return-path encoder, its per-tensor amax given by the GEMM
            m.hadamard_quant(self.Y[:Rp], Rp, d, self.Yc_c, self.Yc_s, self.Yc_g, FOS | m.AMAX_GIVEN, self.amax_y)
        n += 1
        with tm("combine"):  # decode of the returned rows (rotation back, bf16) and the weighted combine
            m.moe4_combine_hadamard(self.Yc_c, self.Yc_s, self.Yc_g, self.row_of, self.w, T, k, d, y)
        n += 1
        if ev is not None:
            ev["y"].record(cur)
        wait("dy")
        # ---------------- backward
        with tm("mxfp8_quant"):  # combine gradient straight into both MXFP8 layouts of dY
            m.moe4_combine_backward_mxfp8(dy, self.row_of, self.w, self.src_of, T, k, d, Rp, self.dYr_q, self.dYr_e,
                                          self.dYc_q, self.dYc_e, OMMA)
        n += 1
        with tm("requant"):
            m.mxfp8_requant_transpose_sr(self.Hq_c, self.Hq_s, self.Hq_g, 1, Rp, f, self.HqT_q, self.HqT_e, seed, 2,
                                         m.SR | MMA | OMMA)
        n += 1
        with tm("gemm_mxfp8_dgrad"):
            m.grouped_gemm_mxfp8(self.dYr_q, self.dYr_e, self.WdT_q, self.WdT_e, self.offs, E, Rp, f, d, self.dH,
                                 m.OUT_F32 | m.GROUP_M | MMA, self.gws)
        n += 1
        with tm("gemm_mxfp8_wgrad_sgd"):
            m.grouped_gemm_mxfp8_wgrad_sgd(self.dYc_q, self.dYc_e, self.HqT_q, self.HqT_e, self.offs, E, d, f, Rp,
                                           self.W32_d, None, LR, self.amax_d, MMA, self.gws)
        n += 2  # the expert ranking for the tile schedule, the GEMM
        with tm("swiglu_bwd"):
            m.moe4_swiglu_backward(self.GU[:Rp], self.dH[:Rp], Rp, f, self.dGU[:Rp])
        n += 1
        with tm("mxfp8_quant"):
            m.mxfp8_quantize_rowcol(self.dGU[:Rp], Rp, 2 * f, self.dGUr_q, self.dGUr_e, self.dGUc_q, self.dGUc_e, OMMA)
        n += 1
        with tm("requant"):
            m.mxfp8_requant_transpose_sr(self.Xp_c, self.Xp_s, self.Xq_g, 1, Rp, d, self.XpT_q, self.XpT_e, seed, 4,
                                         m.SR | MMA | OMMA)
        n += 1
        with tm("gemm_mxfp8_dgrad"):
            m.grouped_gemm_mxfp8(self.dGUr_q, self.dGUr_e, self.WguT_q, self.WguT_e, self.offs, E, Rp, d, 2 * f,
                                 self.dXp, m.OUT_BF16 | m.GROUP_M | MMA, self.gws)
        n += 1
        with tm("gemm_mxfp8_wgrad_sgd"):
            m.grouped_gemm_mxfp8_wgrad_sgd(self.dGUc_q, self.dGUc_e, self.XpT_q, self.XpT_e, self.offs, E, 2 * f, d,
                                           Rp, self.W32_gu, None, LR, self.amax_gu, MMA, self.gws)
        n += 2
        with tm("dispatch_bwd"):  # each token's k dispatched rows of dX summed back into token order
            m.moe4_dispatch_backward(self.dXp, self.row_of, T, k, d, self.dX)
        n += 1
        self.launches += n
        return n

    def weight_path(self, seed, cur):
        """Both projections' weight paths, WEIGHT_CHUNKS expert chunks each: the first chunk's
        quantiser on the whole GPU, then every chunk's requantiser on the step's stream beside the
        next chunk's quantiser (MOE4_SHARE_SMS) on the side stream."""
        m, E, d, f = self.m, self.E, self.d, self.f
        WF = m.FOUR_OVER_SIX | m.SR | m.SF_MMA_LAYOUT | m.SF_OUT_MMA
        chunks = []
        for (W, am, c, sf, g, qt, et, rows, cols, sid), bounds in zip((
                (self.W32_gu, self.amax_gu, self.Wgu_c, self.Wgu_s, self.Wgu_g, self.WguT_q, self.WguT_e, 2 * f, d, 3),
                (self.W32_d, self.amax_d, self.Wd_c, self.Wd_s, self.Wd_g, self.WdT_q, self.WdT_e, d, f, 1)),
                weight_chunk_bounds(E)):
            for e0, e1 in zip(bounds[:-1], bounds[1:]):
                # mat_base = the chunk's first expert: its random numbers are those of one call over
                # the projection's whole stack
                chunks.append(((W[e0:e1], e1 - e0, rows, cols, am[e0:e1], c[e0:e1], sf[e0:e1], g[e0:e1], qt[e0:e1],
                                et[e0:e1], seed, sid, self.offs[e0:e1 + 1]), e0))
        m.nvfp4_quantize_f32_requant(*chunks[0][0], WF | m.PASS_QUANT, mat_base=chunks[0][1])
        self.ev_fork.record(cur)
        self.side.wait_event(self.ev_fork)
        for i, (args, e0) in enumerate(chunks):
            if i + 1 < len(chunks):
                m.nvfp4_quantize_f32_requant(*chunks[i + 1][0], WF | m.PASS_QUANT | m.SHARE_SMS, self.side,
                                             mat_base=chunks[i + 1][1])
                self.ev_q[i + 1].record(self.side)
            if i > 0:
                cur.wait_event(self.ev_q[i])
            m.nvfp4_quantize_f32_requant(*args, WF | m.PASS_REQUANT, mat_base=e0)

    # algorithmic HBM bytes of the kernel groups (per step), for the roofline
    def group_bytes(self):
        T, d, f, E, k = self.T, self.d, self.f, self.E, self.k
        rows = T * k
        offs = self.offs.cpu().numpy()
        live = int(np.count_nonzero(np.diff(offs)))
        nv = 0.5625       # NVFP4 bytes per value (codes + E4M3 scale per 16)
        mx = 1.03125      # MXFP8 bytes per value (E4M3 + E8M0 per 32)
        w_gu, w_d = E * 2 * f * d, E * d * f
        b = {}
        # the weights of experts with rows: FP32 read, NVFP4 and the MXFP8 transpose written (amax from
        # the SGD epilogue)
        b["quant_w"] = (w_gu + w_d) * live / E * (4 + nv + mx)
        b["quant_x"] = T * d * (2 + 2 + nv) + rows * d * nv * 2          # + gather read/write
        b["gemm_nvfp4"] = (rows * d * nv + live * 2 * f * d * nv + rows * 2 * f * 4 + rows * f * 2 +  # + H
                           rows * f * nv + live * d * f * nv + rows * d * 2)
        b["requant"] = rows * (f + d) * (nv + mx)                        # H and the gathered X
        # combine gradient formed from dy (read once) straight into both MXFP8 layouts of dY, and one
        # read of dGU for its two layouts
        b["mxfp8_quant"] = rows * d * 2 * mx + T * d * 2 + rows * 2 * f * (2 + 2 * mx)
        b["gemm_mxfp8_dgrad"] = (rows * d * mx + live * f * d * mx + rows * f * 4 +          # down
                                 rows * 2 * f * mx + live * d * 2 * f * mx + rows * d * 2)   # gate/up
        # wgrad operands + the SGD epilogue: read W32, write W32 (the bf16 copy is not stored)
        b["gemm_mxfp8_wgrad_sgd"] = (rows * d * mx + rows * f * mx + rows * 2 * f * mx + rows * d * mx +
                                     (w_gu + w_d) * live / E * (4 + 4))   # experts without rows are skipped
        b["quant_h"] = rows * f * (2 + nv)             # SwiGLU and its amax in the gate/up GEMM
        b["swiglu_bwd"] = rows * (2 * f * 4 + f * 4 + 2 * f * 2)
        b["hadamard"] = rows * d * (2 + nv)            # amax from the down GEMM's last stage
        b["combine"] = rows * d * nv + T * d * 2       # decoded from the NVFP4 rows as it combines
        b["dispatch_bwd"] = rows * d * 2 + T * d * 2
        b["route"] = T * E * 4 + rows * 4 * 4
        return b


def measure_next_rows(step, reps=3):
    """Rows beyond the layer step, timed after it on the same routed batch (not part of `value`):
    the MXFP8 forward kept for the final layers (bf16 -> MXFP8 nearest-even quantisation of X, of
    both expert weights and of H, the MXFP8 row gather, the rows-grouped MXFP8 GEMMs for gate/up and
    down with SwiGLU between them), and the 8.25-bit Hadamard + MXFP8 return-path codec."""
    torch, m = step.torch, step.m
    T, d, f, E, k, Rp, dev = step.T, step.d, step.f, step.E, step.k, step.Rp, step.dev
    # the final layers' forward reads bf16 weights: refresh the copies from the updated FP32 masters
    m.moe4_convert(2, step.W32_gu, step.W32_gu.numel(), step.Wb_gu)
    m.moe4_convert(2, step.W32_d, step.W32_d.numel(), step.Wb_d)
    u8 = dict(dtype=torch.uint8, device=dev)
    Xq, Xe = torch.empty((T, d), **u8), torch.empty((T, d // 32), **u8)
    Xpq, Xpe = torch.empty((Rp, d), **u8), torch.empty((Rp, d // 32), **u8)
    Gq, Ge = torch.empty((E, 2 * f, d), **u8), torch.empty((E, 2 * f, d // 32), **u8)
    Dq, De = torch.empty((E, d, f), **u8), torch.empty((E, d, f // 32), **u8)
    Hq, He = torch.empty((Rp, f), **u8), torch.empty((Rp, f // 32), **u8)
    Cq, Ce = torch.empty((Rp, d), **u8), torch.empty((Rp, d // 32), **u8)
    ws = m.workspace(max(m.moe4_workspace_size_gemm(1, Rp, E, 2 * f, d), m.moe4_workspace_size_gemm(1, Rp, E, d, f)),
                     dev)
    R, GM = m.ROWWISE, m.GROUP_M

    def fwd(tm):
        with tm("mx_quant"):
            m.mxfp8_quantize(step.X, T, d, Xq, Xe, 0, 0, R)
            m.moe4_permute_nvfp4(Xq, Xe, T, d, step.src_of, Rp, Xpq, Xpe, m.MXFP8)
            m.mxfp8_quantize(step.Wb_gu, E * 2 * f, d, Gq, Ge, 0, 0, R)
            m.mxfp8_quantize(step.Wb_d, E * d, f, Dq, De, 0, 0, R)
        with tm("gemm_mxfp8_fwd"):
            m.grouped_gemm_mxfp8(Xpq, Xpe, Gq, Ge, step.offs, E, Rp, 2 * f, d, step.GU, m.OUT_F32 | GM, ws)
        with tm("mx_quant"):
            m.moe4_swiglu(step.GU[:Rp], Rp, f, step.H[:Rp])
            m.mxfp8_quantize(step.H[:Rp], Rp, f, Hq, He, 0, 0, R)
        with tm("gemm_mxfp8_fwd"):
            m.grouped_gemm_mxfp8(Hq, He, Dq, De, step.offs, E, Rp, d, f, step.Y, m.OUT_BF16 | GM, ws)
        with tm("codec_mx"):
            m.hadamard_quant(step.Y[:Rp], Rp, d, Cq, Ce, None, m.MXFP8)
            m.hadamard_dequant(Cq, Ce, None, Rp, d, step.Yhat[:Rp], m.MXFP8)

    MMA = m.SF_MMA_LAYOUT

    def down_codec(tm):
        # the down projection with the return-path codec fused into its final stage, beside the
        # unfused pair (bf16 product to memory, then the codec); NVFP4 operands of the step
        with tm("down_unfused"):
            m.grouped_expert_gemm_nvfp4(step.Hq_c, step.Hq_s, step.Hq_g, step.Wd_c, step.Wd_s, step.Wd_g, step.offs,
                                        E, Rp, d, f, step.Y, m.OUT_BF16 | MMA)
            m.hadamard_quant(step.Y[:Rp], Rp, d, Cq, Ce, None, m.MXFP8)
        with tm("down_fused"):
            m.grouped_expert_gemm_nvfp4_hadamard_mx(step.Hq_c, step.Hq_s, step.Hq_g, step.Wd_c, step.Wd_s,
                                                    step.Wd_g, step.offs, E, Rp, d, f, Cq, Ce, MMA)

    for _ in range(2):
        fwd(_NullTimer())
        down_codec(_NullTimer())
    torch.cuda.synchronize()
    timer = EventTimer(torch)
    for _ in range(reps):
        fwd(timer)
        down_codec(timer)
    torch.cuda.synchronize()
    if m.moe4_get_status() != m.OK:
        raise RuntimeError("a device wait timed out in the MXFP8 forward")
    per = {n: t / reps for n, t in timer.totals().items()}
    fwd_flops = step.gemm_flops()[0]
    rows = T * k
    codec_bytes = rows * d * (2 + 1.03125 + 1.03125 + 2)
    return {
        "mxfp8_forward": {
            "gemm_ms": round(per["gemm_mxfp8_fwd"], 4),
            "gemm_TFLOP/s": round(fwd_flops / (per["gemm_mxfp8_fwd"] / 1e3) / 1e12, 1),
            "quant_swiglu_ms": round(per["mx_quant"], 4),
            "note": "bf16 -> MXFP8 (nearest-even) of X, W_gu, W_d and H + gather + SwiGLU; same routed batch",
        },
        "fused_down_gemm_codec": {
            "fused_ms": round(per["down_fused"], 4),
            "unfused_ms": round(per["down_unfused"], 4),
            "note": "down GEMM with the 8.25-bit Hadamard + MXFP8 codec in its epilogue vs bf16 GEMM then codec",
        },
        "hadamard_mxfp8_codec": {
            "ms": round(per["codec_mx"], 4),
            "GB/s": round(codec_bytes / (per["codec_mx"] / 1e3) / 1e9, 1),
            "bits_per_value": 8.25,
        },
    }


def compute_probe(kind, reps=5, dev="cuda:0"):
    """The grouped GEMM on a compute-bound shape (not the layer's): 8 groups of 8192 rows, N = K =
    8192, bf16 out (about 5.3k FLOP per byte).  kind 0: NVFP4 (Four Over Six operands, tensor-core
    scale layout); kind 1: MXFP8 (nearest-even operands, rows grouped).  Returns (ms, TFLOP/s)."""
    import torch
    from precision_moe_numerics_03_b300 import inputs, moe4 as m
    E, rows_e, N, K = 8, 8192, 8192, 8192
    R = E * rows_e
    g = lambda s: inputs.device_generator(11, s, dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    x = inputs.device_normal((R, K), 1.0, g(0), dev).view(torch.int16)
    w = inputs.device_normal((E * N, K), 0.02, g(1), dev).view(torch.int16)
    offs = torch.arange(0, R + 1, rows_e, dtype=torch.int32, device=dev)
    out = torch.empty((R, N), dtype=torch.int16, device=dev)
    if kind == 0:
        MMA = m.SF_MMA_LAYOUT
        ac, asf = torch.empty((R, K // 2), **u8), torch.empty((R, K // 16), **u8)
        bc, bsf = torch.empty((E * N, K // 2), **u8), torch.empty((E * N, K // 16), **u8)
        ag, bg = torch.empty(1, dtype=torch.float32, device=dev), torch.empty(E, dtype=torch.float32, device=dev)
        qws = m.workspace(m.moe4_workspace_size(m.OP_NVFP4_QUANTIZE, E), dev)
        m.nvfp4_quantize(x, 1, R, K, K, ac, asf, ag, None, m.FOUR_OVER_SIX | MMA, qws)
        m.nvfp4_quantize(w, E, N, K, K, bc, bsf, bg, None, m.FOUR_OVER_SIX | MMA, qws)
        del x, w
        call = lambda: m.grouped_expert_gemm_nvfp4(ac, asf, ag, bc, bsf, bg, offs, E, R, N, K, out, m.OUT_BF16 | MMA)
    else:
        aq, ae = torch.empty((R, K), **u8), torch.empty((R, K // 32), **u8)
        bq, be = torch.empty((E * N, K), **u8), torch.empty((E * N, K // 32), **u8)
        m.mxfp8_quantize(x, R, K, aq, ae, 0, 0, m.ROWWISE)
        m.mxfp8_quantize(w, E * N, K, bq, be, 0, 0, m.ROWWISE)
        del x, w
        ws = m.workspace(m.moe4_workspace_size_gemm(1, R, E, N, K), dev)
        call = lambda: m.grouped_gemm_mxfp8(aq, ae, bq, be, offs, E, R, N, K, out, m.OUT_BF16 | m.GROUP_M, ws)
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(reps):
        call()
    e0.record()
    torch.cuda.synchronize()
    if m.moe4_get_status() != m.OK:
        raise RuntimeError("a device wait timed out in the compute probe")
    ms = s0.elapsed_time(e0) / reps
    return ms, 2.0 * R * N * K / (ms / 1e3) / 1e12


def measure_tensor_peaks(dev="cuda:0", iters=20000, sustain_s=3.0):
    """The tensor pipe's dense NVFP4 and MXFP8 rates on this GPU, in TFLOP/s, from the library's
    throughput probe (one CTA per SM, operands resident in shared memory, the GEMMs' own MMA
    instructions).  burst: five launches after two untimed ones; sustained: launches back to back
    for `sustain_s` seconds, the rate over the last third (under the power cap, as a kernel inside a
    long step runs)."""
    import torch
    from precision_moe_numerics_03_b300 import moe4 as m
    n = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(n, dtype=torch.int32, device=dev)
    out = {"ctas": n, "iters": iters}
    for kind, name, flop in ((0, "nvfp4", 2.0 ** 24), (1, "mxfp8", 2.0 ** 23)):
        launch = lambda: m.moe4_tensor_peak_probe(kind, iters, n, sink)
        work = n * iters * flop
        for _ in range(2):
            launch()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(5):
            launch()
        e0.record()
        torch.cuda.synchronize()
        burst = 5 * work / (s0.elapsed_time(e0) / 1e3) / 1e12
        chunks = []
        t_end = time.perf_counter() + sustain_s
        while time.perf_counter() < t_end:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(10):
                launch()
            b.record()
            b.synchronize()
            chunks.append(a.elapsed_time(b))
        tail = chunks[len(chunks) * 2 // 3:]
        sustained = 10 * len(tail) * work / (sum(tail) / 1e3) / 1e12
        out[name] = {"burst_TFLOPs": round(burst, 1), "sustained_TFLOPs": round(sustained, 1)}
    if m.moe4_get_status() != m.OK:
        raise RuntimeError("a device wait timed out in the tensor peak probe")
    return out


class _NullTimer:
    def __call__(self, name):
        return self

    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


class EventTimer:
    """CUDA events on the launching stream around each named group of calls."""

    def __init__(self, torch):
        self.torch = torch
        self.records = []

    def __call__(self, name):
        self._name = name
        return self

    def __enter__(self):
        s = self.torch.cuda.Event(enable_timing=True)
        s.record()
        self._start = s
        return self

    def __exit__(self, *a):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record()
        self.records.append((self._name, self._start, e))
        return False

    def totals(self):
        out = {}
        for name, s, e in self.records:
            out[name] = out.get(name, 0.0) + s.elapsed_time(e)
        return out


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and reference arm)
# ---------------------------------------------------------------------------------------------
def oracle_sample_step(d=D_MODEL, f=D_FF, rows=128, seed=0):
    """One expert, one 128-row tile of routed tokens, every step of the method on the oracle.  Run
    it in a process started with one BLAS thread (the reference arm, or `--cpu-leg`): the oracle's C
    is single-threaded too.  Returns (expert-GEMM FLOPs, seconds)."""
    return _oracle_sample_step(d, f, rows, seed)


def cpu_leg_in_child():
    """The CPU baseline in a fresh process with one BLAS thread: the step sample and the requant
    sample of the oracle.  Returns their JSON record."""
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg"], capture_output=True, text=True,
                         timeout=600)
    if out.returncode != 0:
        raise RuntimeError("CPU baseline leg failed: " + out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def oracle_requant_sample(rows=1024, d=D_MODEL, seed=0):
    """The oracle's dequantise -> transpose -> MXFP8 stochastic-rounding requantisation of a slice
    of the backward-requant workload's activations (Student-t(3), d_model 4096), on one thread.
    Returns (algorithmic bytes at 0.5625 B read + 1.03125 B written per value, seconds)."""
    import oracle
    from precision_moe_numerics_03_b300 import inputs
    rng = inputs.host_rng(4, 200 + seed)
    x = oracle.bf16_to_f32(inputs.to_bf16_bits(inputs.host_student_t(rng, (rows, d))))
    q = oracle.nvfp4_quantize(x)
    t0 = time.perf_counter()
    oracle.mxfp8_requant_transpose(*q, sr=True, seed=seed, stream_id=4)
    secs = time.perf_counter() - t0
    return rows * d * (0.5625 + 1.03125), secs


def _oracle_sample_step(d, f, rows, seed):
    import oracle
    from precision_moe_numerics_03_b300 import inputs
    rng = inputs.host_rng(5, 100 + seed)
    x = inputs.to_bf16_bits(inputs.host_student_t(rng, (rows, d)))
    w_gu = rng.standard_normal((2 * f, d), dtype=np.float32) * np.float32(0.02)
    w_d = rng.standard_normal((d, f), dtype=np.float32) * np.float32(0.02)
    dy = inputs.to_bf16_bits(inputs.host_normal(rng, (rows, d)))
    t0 = time.perf_counter()
    o = oracle
    wb_gu, wb_d = o.bf16_to_f32(o.f32_to_bf16(w_gu)), o.bf16_to_f32(o.f32_to_bf16(w_d))
    xq = o.nvfp4_quantize(o.bf16_to_f32(x))
    gq = o.nvfp4_quantize(wb_gu)
    dq = o.nvfp4_quantize(wb_d)
    offs = np.array([0, rows])
    xh, gh, dh_ = o.nvfp4_dequantize(*xq), o.nvfp4_dequantize(*gq), o.nvfp4_dequantize(*dq)
    gu, _ = o.grouped_gemm_m(xh, gh[None], offs)
    h = o.swiglu(gu)
    hq = o.nvfp4_quantize(o.bf16_to_f32(o.f32_to_bf16(h)))
    y, _ = o.grouped_gemm_m(o.nvfp4_dequantize(*hq), dh_[None], offs)
    yc = o.hadamard_quant(o.bf16_to_f32(o.f32_to_bf16(y.astype(np.float32))))
    o.hadamard_dequant(*yc)
    dyf = o.bf16_to_f32(dy)
    dyr = o.mxfp8_dequantize(*o.mxfp8_quantize(dyf, colwise=False))
    dyc = o.mxfp8_dequantize(*o.mxfp8_quantize(dyf, colwise=True))
    wdT = o.mxfp8_dequantize(*o.mxfp8_requant_transpose(*dq, sr=True, seed=seed, stream_id=1))
    hT = o.mxfp8_dequantize(*o.mxfp8_requant_transpose(*hq, sr=True, seed=seed, stream_id=2))
    dH, _ = o.grouped_gemm_m(dyr, wdT[None], offs)
    dWd, _ = o.grouped_gemm_k(dyc, hT, offs)
    dgu = o.bf16_to_f32(o.f32_to_bf16(o.swiglu_backward(gu.astype(np.float32), dH.astype(np.float32))))
    dgur = o.mxfp8_dequantize(*o.mxfp8_quantize(dgu, colwise=False))
    dguc = o.mxfp8_dequantize(*o.mxfp8_quantize(dgu, colwise=True))
    wguT = o.mxfp8_dequantize(*o.mxfp8_requant_transpose(*gq, sr=True, seed=seed, stream_id=3))
    xT = o.mxfp8_dequantize(*o.mxfp8_requant_transpose(*xq, sr=True, seed=seed, stream_id=4))
    o.grouped_gemm_m(dgur, wguT[None], offs)
    dWgu, _ = o.grouped_gemm_k(dguc, xT, offs)
    o.sgd_update(w_gu, dWgu[0].astype(np.float32), LR)
    o.sgd_update(w_d, dWd[0].astype(np.float32), LR)
    secs = time.perf_counter() - t0
    fwd = 2 * rows * 2 * f * d + 2 * rows * d * f
    return 3 * fwd, secs


def cpu_cores_used():
    """The oracle legs run on one host thread (single-threaded C, one BLAS thread)."""
    return 1


# ---------------------------------------------------------------------------------------------
def max_over_ranks(x, dist):
    """The largest of a float over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    dims = dict(d=SMALL["d"], f=SMALL["f"]) if args.small else {}
    flops, secs = 0, 0.0
    for i in range(args.warmup):
        oracle_sample_step(seed=i, **dims)
    for i in range(args.steps):
        fl, s = oracle_sample_step(seed=100 + i, **dims)
        flops += fl
        secs += s
    value = flops / secs / 1e12
    sample = "one expert (gate/up 4096x4096, down 4096x2048 weights) and one 128-row tile of routed tokens per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 GEMM / f32 quantisers",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def profile_case(name):
    """One kernel on a case larger than L2 but a few GB at most: 2 untimed + 3 launches."""
    import torch
    from precision_moe_numerics_03_b300 import inputs, moe4
    moe4.load()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    g = lambda s: inputs.device_generator(7, s, dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    E, d, f = 16, 4096, 2048            # 16 experts of the Inkling shape: 268 M gate/up weights
    calls = []
    if name in ("requant", "quant_w", "sgd"):
        w = inputs.device_normal((E * 2 * f, d), 0.02, g(0), dev).view(torch.int16)
        c, s_ = torch.empty((E, 2 * f, d // 2), **u8), torch.empty((E, 2 * f, d // 16), **u8)
        gd = torch.empty(E, dtype=torch.float32, device=dev)
        ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, E), dev)
        quant = lambda: moe4.nvfp4_quantize(w, E, 2 * f, d, d, c, s_, gd, None,
                                            moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT, ws)
        quant()
        if name == "quant_w":  # as in the layer step: the FP32 master weights, with their MXFP8 transposes
            w32 = inputs.device_normal((E * 2 * f, d), 0.02, g(8), dev, dtype=torch.float32)
            am = w32.to(torch.bfloat16).abs().view(E, -1).amax(dim=1).float().contiguous()
            q, e8 = torch.empty((E, d, 2 * f), **u8), torch.empty((E, d, 2 * f // 32), **u8)
            fl = moe4.FOUR_OVER_SIX | moe4.SR | moe4.SF_MMA_LAYOUT | moe4.SF_OUT_MMA
            calls.append(lambda: moe4.nvfp4_quantize_f32_requant(w32, E, 2 * f, d, am, c, s_, gd, q, e8, 1, 3, None,
                                                                 fl))
        elif name == "requant":
            q, e8 = torch.empty((E, d, 2 * f), **u8), torch.empty((E, d, 2 * f // 32), **u8)
            calls.append(lambda: moe4.mxfp8_requant_transpose_sr(c, s_, gd, E, 2 * f, d, q, e8, 1, 3,
                                                                 moe4.SR | moe4.SF_MMA_LAYOUT))
        else:
            w32 = torch.randn((E * 2 * f * d,), generator=g(1), device=dev)
            dw = torch.randn((E * 2 * f * d,), generator=g(2), device=dev)
            calls.append(lambda: moe4.moe4_sgd_update(w32, dw, w32.numel(), LR, w.view(-1)))
    elif name in ("mxfp8_rowcol", "hadamard"):
        rows = 32768                     # a quarter of the routed rows at d_model 4096: 268 MB of bf16
        x = inputs.device_student_t((rows, d), g(3), dev).view(torch.int16)
        if name == "mxfp8_rowcol":
            qr, er = torch.empty((rows, d), **u8), torch.empty((rows, d // 32), **u8)
            qc, ec = torch.empty((d, rows), **u8), torch.empty((d, rows // 32), **u8)
            calls.append(lambda: moe4.mxfp8_quantize_rowcol(x, rows, d, qr, er, qc, ec))
        else:
            c, s_ = torch.empty((rows, d // 2), **u8), torch.empty((rows, d // 16), **u8)
            gd = torch.empty(1, dtype=torch.float32, device=dev)
            ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT), dev)
            out = torch.empty((rows, d), dtype=torch.int16, device=dev)
            calls.append(lambda: moe4.hadamard_quant(x, rows, d, c, s_, gd, moe4.FOUR_OVER_SIX, ws))
            calls.append(lambda: moe4.hadamard_dequant(c, s_, gd, rows, d, out))
    elif name == "hadamard_given":       # as in the layer step: the rotated amax comes from the down GEMM
        rows = 32768
        x = inputs.device_student_t((rows, d), g(3), dev)
        h = torch.ones((1, 1), device=dev)
        while h.shape[0] < 128:          # Sylvester's construction, normalised below
            h = torch.cat([torch.cat([h, h], 1), torch.cat([h, -h], 1)], 0)
        am = ((x.float().view(-1, 128) @ h) / 128 ** 0.5).abs().max().reshape(1).contiguous()
        x = x.view(torch.int16)
        c, s_ = torch.empty((rows, d // 2), **u8), torch.empty((rows, d // 16), **u8)
        gd = torch.empty(1, dtype=torch.float32, device=dev)
        calls.append(lambda: moe4.hadamard_quant(x, rows, d, c, s_, gd, moe4.FOUR_OVER_SIX | moe4.AMAX_GIVEN, am))
    elif name == "combine_hadamard":     # 8192 tokens x top-8 returned rows of d_model 4096, decoded as combined
        T, k = 8192, 8
        x = inputs.device_student_t((T * k, d), g(3), dev).view(torch.int16)
        c, s_ = torch.empty((T * k, d // 2), **u8), torch.empty((T * k, d // 16), **u8)
        gd = torch.empty(1, dtype=torch.float32, device=dev)
        ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_HADAMARD_QUANT), dev)
        moe4.hadamard_quant(x, T * k, d, c, s_, gd, moe4.FOUR_OVER_SIX, ws)
        row_of = torch.randperm(T * k, generator=g(4), device=dev).to(torch.int32).view(T, k)
        w = torch.softmax(torch.randn((T, k), generator=g(5), device=dev), dim=1).contiguous()
        y = torch.empty((T, d), dtype=torch.int16, device=dev)
        calls.append(lambda: moe4.moe4_combine_hadamard(c, s_, gd, row_of, w, T, k, d, y))
    elif name in ("swiglu_bwd", "swiglu_bwd_mxfp8"):
        rows = 32768                     # a fifth of the layer's padded rows, SwiGLU width 2048
        gu = torch.randn((rows, 2 * f), generator=g(11), device=dev)
        dh = torch.randn((rows, f), generator=g(12), device=dev)
        if name == "swiglu_bwd":
            dgu = torch.empty((rows, 2 * f), dtype=torch.int16, device=dev)
            calls.append(lambda: moe4.moe4_swiglu_backward(gu, dh, rows, f, dgu))
        else:
            qr, er = torch.empty((rows, 2 * f), **u8), torch.empty((rows, 2 * f // 32), **u8)
            qc, ec = torch.empty((2 * f, rows), **u8), torch.empty((2 * f, rows // 32), **u8)
            calls.append(lambda: moe4.moe4_swiglu_backward_mxfp8(gu, dh, rows, f, qr, er, qc, ec, moe4.SF_OUT_MMA))
    elif name == "tensor_peaks":  # the four kinds of the tensor-pipe probe, as TFLOP/s
        n = torch.cuda.get_device_properties(dev).multi_processor_count
        sink = torch.zeros(n, dtype=torch.int32, device=dev)
        res = {}
        for kind, flop in ((0, 2.0 ** 24), (1, 2.0 ** 23), (2, 2.0 ** 24), (3, 2.0 ** 23)):
            for iters in (5000, 20000):
                for _ in range(2):
                    moe4.moe4_tensor_peak_probe(kind, iters, n, sink)
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(5):
                    moe4.moe4_tensor_peak_probe(kind, iters, n, sink)
                b.record()
                torch.cuda.synchronize()
                res["kind%d_iters%d" % (kind, iters)] = round(n * iters * flop / (a.elapsed_time(b) / 5 / 1e3) / 1e12, 1)
        if moe4.moe4_get_status() != moe4.OK:
            raise RuntimeError("a device wait timed out")
        print(json.dumps(res))
        return 0
    elif name in ("gemm_nvfp4_probe", "gemm_mxfp8_probe"):
        compute_probe(0 if name == "gemm_nvfp4_probe" else 1, reps=3, dev=dev)
        print("profile case %s done" % name)
        return 0
    elif name in ("gemm_nvfp4", "gemm_nvfp4_swiglu", "gemm_nvfp4_down_amax"):
        rows = 128 * 64
        x = inputs.device_student_t((rows, d), g(3), dev).view(torch.int16)
        w = inputs.device_normal((E * 2 * f, d), 0.02, g(0), dev).view(torch.int16)
        ac, as_ = torch.empty((rows, d // 2), **u8), torch.empty((rows, d // 16), **u8)
        ag = torch.empty(1, dtype=torch.float32, device=dev)
        bc, bs = torch.empty((E, 2 * f, d // 2), **u8), torch.empty((E, 2 * f, d // 16), **u8)
        bg = torch.empty(E, dtype=torch.float32, device=dev)
        ws = moe4.workspace(moe4.moe4_workspace_size(moe4.OP_NVFP4_QUANTIZE, E), dev)
        flags = moe4.FOUR_OVER_SIX | moe4.SF_MMA_LAYOUT
        moe4.nvfp4_quantize(x, 1, rows, d, d, ac, as_, ag, None, flags, ws)
        moe4.nvfp4_quantize(w, E, 2 * f, d, d, bc, bs, bg, None, flags, ws)
        offs = torch.arange(0, rows + 1, rows // E, dtype=torch.int32, device=dev)
        if name == "gemm_nvfp4":  # the gate/up projection: binary32 out
            out = torch.empty((rows, 2 * f), dtype=torch.float32, device=dev)
            calls.append(lambda: moe4.grouped_expert_gemm_nvfp4(ac, as_, ag, bc, bs, bg, offs, E, rows, 2 * f, d, out,
                                                                moe4.OUT_F32 | moe4.SF_MMA_LAYOUT))
        elif name == "gemm_nvfp4_swiglu":  # the gate/up projection as the step runs it: GU, h and its amax
            out = torch.empty((rows, 2 * f), dtype=torch.float32, device=dev)
            hout = torch.empty((rows, f), dtype=torch.int16, device=dev)
            am = torch.empty(1, dtype=torch.float32, device=dev)
            calls.append(lambda: moe4.grouped_expert_gemm_nvfp4_swiglu(ac, as_, ag, bc, bs, bg, offs, E, rows, f, d, out,
                                                                       hout, am, moe4.SF_MMA_LAYOUT))
        else:  # the down projection as the step runs it: bf16 out and the rotated amax for the codec
            hc, hs = torch.empty((rows, f // 2), **u8), torch.empty((rows, f // 16), **u8)
            h = inputs.device_student_t((rows, f), g(9), dev).view(torch.int16)
            moe4.nvfp4_quantize(h, 1, rows, f, f, hc, hs, ag, None, flags, ws)
            wd = inputs.device_normal((E * d, f), 0.02, g(10), dev).view(torch.int16)
            dc, ds_ = torch.empty((E, d, f // 2), **u8), torch.empty((E, d, f // 16), **u8)
            moe4.nvfp4_quantize(wd, E, d, f, f, dc, ds_, bg, None, flags, ws)
            y = torch.empty((rows, d), dtype=torch.int16, device=dev)
            am = torch.empty(1, dtype=torch.float32, device=dev)
            calls.append(lambda: moe4.grouped_expert_gemm_nvfp4_hadamard_amax(hc, hs, ag, dc, ds_, bg, offs, E, rows, d,
                                                                              f, y, am, moe4.SF_MMA_LAYOUT))
    else:
        rows = 128 * 64
        offs = torch.arange(0, rows + 1, rows // E, dtype=torch.int32, device=dev)
        if name in ("gemm_mxfp8_wgrad", "gemm_mxfp8_wgrad_sgd"):
            M, N = 2 * f, d
            a = torch.randint(0, 120, (M, rows), generator=g(4), device=dev, dtype=torch.int32).to(torch.uint8)
            b = torch.randint(0, 120, (N, rows), generator=g(5), device=dev, dtype=torch.int32).to(torch.uint8)
            ae = torch.full((M, rows // 32), 120, **u8)
            be = torch.full((N, rows // 32), 120, **u8)
            out = torch.randn((E, M, N), generator=g(6), device=dev).mul_(0.02)
            ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, M, 1, N, rows), dev)
            if name == "gemm_mxfp8_wgrad":
                calls.append(lambda: moe4.grouped_gemm_mxfp8(a, ae, b, be, offs, E, M, N, rows, out,
                                                             moe4.OUT_F32 | moe4.GROUP_K, ws))
            else:  # as in the layer step: no stored bf16 copy
                amax = torch.empty(E, dtype=torch.float32, device=dev)
                calls.append(lambda: moe4.grouped_gemm_mxfp8_wgrad_sgd(a, ae, b, be, offs, E, M, N, rows, out, None,
                                                                       LR, amax, 0, ws))
        else:
            N, K = d, 2 * f
            a = torch.randint(0, 120, (rows, K), generator=g(4), device=dev, dtype=torch.int32).to(torch.uint8)
            b = torch.randint(0, 120, (E * N, K), generator=g(5), device=dev, dtype=torch.int32).to(torch.uint8)
            ae = torch.full((rows, K // 32), 120, **u8)
            be = torch.full((E * N, K // 32), 120, **u8)
            out = torch.empty((rows, N), dtype=torch.int16, device=dev)
            ws = moe4.workspace(moe4.moe4_workspace_size_gemm(1, rows, E, N, K), dev)
            calls.append(lambda: moe4.grouped_gemm_mxfp8(a, ae, b, be, offs, E, rows, N, K, out,
                                                         moe4.OUT_BF16 | moe4.GROUP_M, ws))
    for _ in range(5):
        for c_ in calls:
            c_()
    torch.cuda.synchronize()
    if moe4.moe4_get_status() != moe4.OK:
        raise RuntimeError("a device wait timed out")
    print("profile case %s done" % name)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # ten steps: the copy pipeline of the end-to-end measurement fills once and drains once per run
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--small", action="store_true", help="the small 8-expert shapes (a quick check, not a bench line)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--no-next", action="store_true", help="skip the supplementary MXFP8-forward and 8.25-bit codec timings")
    ap.add_argument("--profile-case", default=None,
                    choices=["requant", "quant_w", "gemm_nvfp4", "gemm_nvfp4_swiglu", "gemm_nvfp4_down_amax",
                             "gemm_mxfp8_wgrad",
                             "gemm_mxfp8_wgrad_sgd",
                             "gemm_mxfp8_dgrad", "sgd", "mxfp8_rowcol", "hadamard", "hadamard_given", "combine_hadamard",
                             "gemm_nvfp4_probe", "tensor_peaks",
                             "swiglu_bwd", "swiglu_bwd_mxfp8",
                             "gemm_mxfp8_probe"],
                    help="run one kernel a few times on a mid-size case (for ncu captures; prints no bench line)")
    args = ap.parse_args()
    if args.cpu_leg:  # the CPU baseline's oracle samples, in their own one-thread process
        fl, secs = oracle_sample_step(seed=0)
        rb, rsecs = oracle_requant_sample()
        print(json.dumps({"flops": fl, "seconds": secs, "requant_bytes": rb, "requant_seconds": rsecs}))
        return 0
    if args.profile_case:
        return profile_case(args.profile_case)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return rc

    import torch
    from precision_moe_numerics_03_b300 import moe4
    moe4.load()
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    if args.small:
        step = LayerStep(SMALL["T"], SMALL["d"], SMALL["f"], SMALL["E"], SMALL["k"], dev)
    else:
        step = LayerStep(T_TOK, D_MODEL, D_FF, N_EXP, TOP_K, dev)
    torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    if moe4.moe4_get_status() != moe4.OK:
        raise RuntimeError("a device wait timed out during warm-up")

    # ------------------------------------------------ timed region (device)
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    timer = EventTimer(torch)
    launches = 0
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(args.steps):
        launches += step.run(timer)
    t_end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    elapsed_ms = t_start.elapsed_time(t_end)
    if moe4.moe4_get_status() != moe4.OK:
        raise RuntimeError("a device wait timed out in the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, dist)
    ms = elapsed_ms / args.steps
    fwd_flops, bwd_flops = step.gemm_flops()
    step_flops = fwd_flops + bwd_flops
    value = world * step_flops * args.steps / (elapsed_ms / 1e3) / 1e12

    # per-kernel-group times (ms per step) and the roofline of the dominant group
    peaks = load_peaks()
    per = {k: v / args.steps for k, v in timer.totals().items()}
    gbytes = step.group_bytes()
    comps = {}
    for name, t in sorted(per.items(), key=lambda kv: -kv[1]):
        entry = {"ms": round(t, 4), "share": round(t / ms, 4)}
        if name in gbytes:
            entry["GB/s"] = round(gbytes[name] / (t / 1e3) / 1e9, 1)
        comps[name] = entry
    comps["gemm_nvfp4"]["TFLOP/s"] = round(fwd_flops / (per["gemm_nvfp4"] / 1e3) / 1e12, 1)
    comps["gemm_mxfp8_dgrad"]["TFLOP/s"] = round(fwd_flops / (per["gemm_mxfp8_dgrad"] / 1e3) / 1e12, 1)
    comps["gemm_mxfp8_wgrad_sgd"]["TFLOP/s"] = round(fwd_flops / (per["gemm_mxfp8_wgrad_sgd"] / 1e3) / 1e12, 1)
    # dense FP4 / FP8 peaks of this GPU, measured by the tensor-pipe probe (sustained: the GEMMs
    # are timed inside a long step), after the timed region
    tpk = measure_tensor_peaks(dev)
    fp4_peak = tpk["nvfp4"]["sustained_TFLOPs"]
    fp8_peak = tpk["mxfp8"]["sustained_TFLOPs"]
    # the dominant kernel: the group with the most time among those that run one kernel ("quant_w"
    # runs two, the FP32-master quantiser and the requantiser, each below the fused SGD GEMM)
    dom = max((k for k in per if k not in MULTI_KERNEL_GROUPS), key=per.get)
    t_dom = per[dom]
    flops_dom = {"gemm_nvfp4": (fwd_flops, fp4_peak), "gemm_mxfp8_dgrad": (fwd_flops, fp8_peak),
                 "gemm_mxfp8_wgrad_sgd": (fwd_flops, fp8_peak)}.get(dom)
    if flops_dom is not None and flops_dom[0] / flops_dom[1] / 1e12 > gbytes[dom] / peaks["hbm"] / 1e9:
        ach = flops_dom[0] / (t_dom / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": flops_dom[1], "unit": "TFLOP/s",
                "frac": ach / flops_dom[1], "traffic": None, "kernel": dom}
    else:
        ach = gbytes[dom] / (t_dom / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s", "frac": ach / peaks["hbm"],
                "traffic": None, "kernel": dom}
    # the metric against both denominators: measured HBM copy and the derived FP4 peak, and the
    # nominal 8 TB/s and the pages' 15 PF dense FP4; for the NVFP4 GEMMs also the fraction of the
    # time bound max(bytes / bandwidth, FLOPs / peak) of their own traffic and work
    t_g = per["gemm_nvfp4"] / 1e3
    bound_meas = max(gbytes["gemm_nvfp4"] / (peaks["hbm"] * 1e9), fwd_flops / (fp4_peak * 1e12))
    bound_nom = max(gbytes["gemm_nvfp4"] / 8000e9, fwd_flops / 15000e12)
    req_gbs = gbytes["requant"] / (per["requant"] / 1e3) / 1e9
    metric_detail = {
        "nvfp4_gemm": {"TFLOP/s": comps["gemm_nvfp4"]["TFLOP/s"],
                       "frac_fp4_peak_measured": round(comps["gemm_nvfp4"]["TFLOP/s"] / fp4_peak, 4),
                       "frac_fp4_peak_15PF": round(comps["gemm_nvfp4"]["TFLOP/s"] / 15000.0, 4),
                       "frac_time_bound_measured": round(bound_meas / t_g, 4),
                       "frac_time_bound_nominal": round(bound_nom / t_g, 4)},
        "requant": {"GB/s": round(req_gbs, 1), "frac_hbm_measured": round(req_gbs / peaks["hbm"], 4),
                    "frac_hbm_nominal_8TBs": round(req_gbs / 8000.0, 4),
                    "note": "issue-bound (Philox4x32-10): ncu issue-slot figures in profiles/"},
        "tensor_peaks": tpk,
        "peaks_note": "FP4/FP8 denominators: the sustained rate of moe4_tensor_peak_probe on this GPU; HBM: "
                      "MEASURED_PEAKS.json copy bandwidth",
    }
    nl = GROUP_LAUNCHES.get(dom, 1)
    roof["launches_per_step"] = nl
    if dom in DRAM_PER_STEP:
        roof["traffic"] = DRAM_PER_STEP[dom] / nl
        roof["traffic_note"] = ("DRAM bytes per launch (read + write), one-pass ncu capture of this step at full "
                                "size; algorithmic bytes per launch %.4g" % (gbytes[dom] / nl))
    roof["peak_source"] = peaks["src"]
    req_t = per.get("requant", 0.0)
    requant_gbs = gbytes["requant"] / (req_t / 1e3) / 1e9 if req_t else None

    # ------------------------------------------------ end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        # Each step's inputs (X, logits, dy) come from pinned host memory and its output y goes back
        # to pinned host memory, inside the timed region.  As in a training loop, step i+1's inputs
        # are copied on a side stream while step i computes (two device input sets, logits first,
        # each input with its own event, so that a step waits for an input only where it first
        # reads it: the weight path runs while X and dy arrive), and step i's y is copied back as
        # soon as the combine has written it, beside the backward (two device y buffers; step i+2
        # writes its y only once that copy is done).  The region ends when every copy is done.
        hX = torch.empty(step.X.shape, dtype=step.X.dtype, pin_memory=True)
        hX.copy_(step.X)
        hL = torch.empty(step.logits.shape, dtype=step.logits.dtype, pin_memory=True)
        hL.copy_(step.logits)
        hD = torch.empty(step.dy.shape, dtype=step.dy.dtype, pin_memory=True)
        hD.copy_(step.dy)
        hY = [torch.empty(step.y.shape, dtype=step.y.dtype, pin_memory=True) for _ in range(2)]
        io = [(step.X, step.logits, step.dy, step.y),
              (torch.empty_like(step.X), torch.empty_like(step.logits), torch.empty_like(step.dy),
               torch.empty_like(step.y))]
        cs = torch.cuda.Stream()
        ev = [{name: torch.cuda.Event() for name in ("logits", "X", "dy", "y")} for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def copy_in(b):
            with torch.cuda.stream(cs):
                for name, dst, src in (("logits", io[b][1], hL), ("X", io[b][0], hX), ("dy", io[b][2], hD)):
                    dst.copy_(src, non_blocking=True)
                    ev[b][name].record(cs)

        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        copy_in(0)
        for i in range(args.steps):
            b = i % 2
            if i + 1 < args.steps:
                if i >= 1:
                    cs.wait_event(ev_done[1 - b])  # step i-1 is done with that input set
                copy_in(1 - b)
            if i >= 2:
                torch.cuda.current_stream().wait_event(ev_out[b])  # step i-2's y has been read back
            step.run(io=io[b], ev=ev[b])
            ev_done[b].record()
            cs.wait_event(ev[b]["y"])
            with torch.cuda.stream(cs):
                hY[b].copy_(io[b][3], non_blocking=True)
                ev_out[b].record(cs)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(e2e_s, dist)
        h2d = hX.numel() * 2 + hL.numel() * 4 + hD.numel() * 2
        d2h = hY[0].numel() * 2 + 4
        e2e = {"value": world * step_flops * args.steps / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_s / args.steps * 1e3}

    nxt = None
    if not args.no_next:
        nxt = measure_next_rows(step)
        mf = nxt["mxfp8_forward"]
        mf["nvfp4_gemm_ms"] = round(per["gemm_nvfp4"], 4)
        mf["nvfp4_gemm_speedup"] = round(mf["gemm_ms"] / per["gemm_nvfp4"], 3)
        mf["nvfp4_quant_swiglu_ms"] = round(per["quant_x"] + per["quant_w"] + per["quant_h"], 4)
        nxt["hadamard_mxfp8_codec"]["nvfp4_encode_and_decode_combine_ms"] = round(per["hadamard"] + per["combine"], 4)
        probe = {"shape": "8 groups x 8192 rows, N = K = 8192, bf16 out (compute-bound; not the layer's shape)"}
        # timed alone: the burst rates of the tensor-pipe probe
        pk = {"nvfp4": tpk["nvfp4"]["burst_TFLOPs"], "mxfp8": tpk["mxfp8"]["burst_TFLOPs"]}
        for kind, name in ((0, "nvfp4"), (1, "mxfp8")):
            pm, pt = compute_probe(kind)
            probe[name] = {"ms": round(pm, 4), "TFLOP/s": round(pt, 1), "frac_of_measured_peak": round(pt / pk[name], 3)}
        probe["peaks_TFLOPs"] = {k: round(v, 1) for k, v in pk.items()}
        probe["peak_source"] = "moe4_tensor_peak_probe burst rate on this GPU"
        nxt["gemm_compute_probe"] = probe

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        leg = cpu_leg_in_child()
        fl, secs, rb, rsecs = leg["flops"], leg["seconds"], leg["requant_bytes"], leg["requant_seconds"]
        cpu = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
               "sample": "one expert (gate/up 4096x4096, down 4096x2048 weights) and one 128-row tile of routed "
                         "tokens through every step", "seconds": round(secs, 2),
               "requant_GBps": round(rb / rsecs / 1e9, 4),
               "requant_sample": "1024 x 4096 Student-t(3) activations: NVFP4 -> dequantise -> transpose -> MXFP8 "
                                 "stochastic rounding, %.2f s" % rsecs,
               "host_cores_available": os.cpu_count()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4/mxfp8 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": WORKLOAD if not args.small else "small-moe-step", "tokens": step.T,
                       "d_model": step.d, "d_ff": step.f, "experts": step.E, "top_k": step.k,
                       "rows_padded": step.Rp, "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "inputs larger than L2 (126 MB): no flush needed"},
            "requant_GBps": requant_gbs, "requant_frac_hbm": requant_gbs / peaks["hbm"] if requant_gbs else None,
            "nvfp4_gemm_TFLOPs": comps["gemm_nvfp4"]["TFLOP/s"],
            "nvfp4_gemm_frac_fp4_peak": comps["gemm_nvfp4"]["TFLOP/s"] / fp4_peak,
            "metric_detail": metric_detail,
            "components": comps,
            "roofline": roof,
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": launches,
            "cpu_baseline": cpu,
            "next_rows": nxt,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
