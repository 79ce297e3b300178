#!/usr/bin/env python
"""Benchmark: gated delta rule forward + VJP tokens/s on GB300 (one JSON line).

Default workload: the Qwen3.5-9B GatedDeltaNet layer shape of the mlx-lm
page's performance table (B=1, T=2048, Hk=16, Hv=64, Dk=192, Dv=128, bf16
inputs, fp32 state), forward + full backward per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--gates ab|lb|kc] [--fused-conv K]
                  [--compress-rank R [--compress-iters N]] [--eager]

One process per GPU (torchrun for N > 1); every rank runs its own replica
of the workload (weak scaling, no collective on the data path).  Timing:
W untimed warm-up steps, then one step's C-ABI calls captured into a CUDA
graph (eager launches with --eager, or where capture is refused), then K
replays each bracketed by CUDA events on the launching stream; L2 is flushed
(256 MiB write) between timed steps outside the events; barrier + synchronize around the timed region; the max over
ranks is reported.  ``value`` = tokens of all ranks / time.  The per-phase
kernel times behind the roofline come from a second pass over the same K
steps with the library's phase events (the timed steps carry none).

``--impl reference`` times the fp64 CPU oracle (the only reference
implementation this method has here) on the host cores, on a bounded sample
of the same workload, and prints the same JSON line with "impl": "reference".
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_delta_rule_06_gb300 import workloads as wl  # noqa: E402

C = 64
METRIC = "GDN fwd+bwd tokens/s (Qwen3.5-9B shape, T=2048) and % of TC/HBM roofline"
DECODE_METRIC = "GDN decode tokens/s (B=256 state step) and % of HBM roofline"
# the page's own figure for this workload: 149.8 ms fwd+bwd at T=2048 on an
# M-series Mac (mlx-lm PR performance table) -> 2048 / 0.1498 tokens/s
PAGE_TOKENS_PER_S = {"qwen35_9b_layer_T2048_bf16": 2048 / 0.1498}
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12  # SMs x FFMA lanes x 2 x max clock


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------------------
# algorithmic work (the method's own bytes and flops, per phase)
# ---------------------------------------------------------------------------

def method_model(w, gates="ab", nseg=1, nseg_bwd=1, conv_k=0, rank=0, iters=3):
    """The method's own bytes and flops, per phase and per step.

    Bytes count only the method's tensors: the primal inputs and outputs, the
    cotangents, and one fp32 state checkpoint per (b, h, chunk), which the
    forward writes once and the backward reads once.  A phase is charged for
    each of those tensors it reads or writes itself; intermediates the
    implementation keeps between its kernels (gate sums, WY images, state
    cotangent images, per-value-head q / k cotangents) count nothing.  Flops
    per token and value head (C the chunk, G the GQA group, Grams shared by a
    key head's G value heads): forward 2C(3Dk + 2Dv) + C^2/3 for the
    chunk-local products and 6 Dk Dv for the scan; backward
    18C Dk + 10C Dv + 14 Dk Dv + 4C^2, of which 6 Dk Dv + 2C Dv is the
    reverse scan; each less (1 - 1/G) 4C Dk for the shared Grams.  The step
    counts every method tensor once per pass plus the checkpoints written and
    read: 673 MB and 110.8 GFLOP at B1 T2048 Hk16 Hv64 Dk192 Dv128 bf16."""
    es = 2 if w.dtype == torch.bfloat16 else 4
    B, T, Hk, Hv, Dk, Dv = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv
    G = Hv // Hk
    NC = (T + C - 1) // C
    BH = B * Hv
    th = B * T * Hv  # (token, value head) pairs
    qk = 2 * B * T * Hk * Dk * es  # q and k
    vv = B * T * Hv * Dv * es  # v, o, dO, dv each
    ab = 2 * B * T * Hv * es  # a and b (or log_decay and beta); da and db
    st = BH * Dk * Dv * 4  # one fp32 state tensor
    ckpt = BH * NC * Dk * Dv * 4  # the fp32 chunk checkpoints
    shared = (1 - 1 / G) * 4 * C * Dk
    f_chunk = th * (2 * C * (3 * Dk + 2 * Dv) + C * C / 3 - shared)
    f_scan = th * 6 * Dk * Dv
    f_bwd = th * (18 * C * Dk + 10 * C * Dv + 14 * Dk * Dv + 4 * C * C - shared)
    f_bscan = th * (6 * Dk * Dv + 2 * C * Dv)
    m = {
        "prep": dict(flops=0.0, bytes=qk + ab),
        "fwd_chunk": dict(flops=f_chunk, bytes=qk + vv),
        "fwd_scan": dict(flops=f_scan, bytes=qk + st + vv + st + ckpt),
        "bwd_scan": dict(flops=f_bscan, bytes=qk + vv + st + st),
        "bwd_chunk": dict(flops=f_bwd - f_bscan, bytes=qk + 2 * vv + ckpt + vv),
        "bwd_scan_chunk": dict(flops=f_bwd, bytes=qk + 2 * vv + st + ckpt + vv + st),
        "bwd_reduce": dict(flops=0.0, bytes=qk + ab + qk + ab + 2 * Hv * 4),
        "decode": dict(flops=BH * (4 * Dk * Dv + 2 * Dk),
                       bytes=2 * st + B * Hk * 2 * Dk * es + B * Hv * 2 * Dv * es + B * Hv * 2 * es),
    }
    Wd = Dv + -(-Dk // 128) * 128
    if nseg > 1:
        # the associative form's own work: per-segment maps over Wd columns and
        # the chain of segment start states
        L = -(-NC // nseg)
        mu = B * Hv * (nseg - 1) * L * C
        m["fwd_seg_maps"] = dict(flops=mu * (6 * Dk * Wd + 2 * C * Wd), bytes=qk)
        m["fwd_seg_chain"] = dict(flops=BH * (nseg - 1) * 2 * Dk * Dk * Dv, bytes=st)
    if nseg_bwd > 1:
        Lb = -(-NC // nseg_bwd)
        mb = B * Hv * (nseg_bwd - 1) * Lb * C
        m["bwd_seg_maps"] = dict(flops=mb * (6 * Dk * Wd + 2 * C * Wd), bytes=qk + vv)
        m["bwd_seg_chain"] = dict(flops=BH * (nseg_bwd - 1) * 2 * Dk * Dk * Dv, bytes=st)
    if conv_k:
        # fused short convolution: the mixed projection, the carried windows in
        # and out and the taps replace the q / k / v reads
        Cm = 2 * Hk * Dk + Hv * Dv
        m["decode"]["flops"] += B * Cm * 2 * conv_k
        m["decode"]["bytes"] += (B * Cm * (1 + 2 * conv_k) + Cm * conv_k) * es \
            - (B * Hk * 2 * Dk + BH * Dv) * es
    io_fwd = qk + vv + ab + vv + 2 * st
    io_bwd = qk + 2 * vv + ab + st + qk + vv + ab + st
    m["_step"] = dict(bytes=io_fwd + io_bwd + 2 * ckpt, flops=f_chunk + f_scan + f_bwd)
    if rank:
        # compressed chunk states: the initial state and rank-r factors of the
        # NC - 1 boundaries (fp32) take the checkpoints' place; the truncation
        # at a boundary costs 2 Dk Dv r flops for S Omega, each of `iters`
        # iterations two such products, then R = Q^T S
        fac = BH * (Dk * Dv + (NC - 1) * (Dk + Dv) * rank) * 4
        m["compress"] = dict(flops=BH * (NC - 1) * (2 * iters + 2) * 2 * Dk * Dv * rank,
                             bytes=fac - st)
        m["expand"] = dict(flops=BH * (NC - 1) * 2 * Dk * Dv * rank, bytes=fac)
        m["fwd_scan"]["bytes"] -= ckpt
        m["bwd_scan_chunk"]["bytes"] -= ckpt
        m["bwd_chunk"]["bytes"] -= ckpt
        m["_step"] = dict(bytes=io_fwd + io_bwd + 2 * fac,
                          flops=m["_step"]["flops"] + m["compress"]["flops"] + m["expand"]["flops"])
    if gates == "kc":
        # per-key-channel gates.  Gate inputs log_decay [B, T, Hv, Dk] and beta;
        # checkpoints per 64-step chunk as for the scalar gates.  The chunked
        # form (bf16 at the tensor-core scans' shapes): the scalar form's flops
        # with no Gram shared between value heads (each has its own decays);
        # the gradient phase split into the tensor-core products (the three state
        # products, Pbar, Dbar V^T, T^T Dbar, Wbar K_r^T, T^T Wbar:
        # 6 Dk Dv + 6 C Dv + 3 C Dk), the 64 x 64 gate products (2 C^2) and the
        # decayed-Gram sums (the rest).
        # The recurrent form (other shapes): per step forward decay, prediction,
        # update and read-out (7 Dk Dv), backward the recompute and the reverse
        # step (20 Dk Dv).
        gin = B * T * Hv * (Dk + 1) * es
        fk_chunk = th * (2 * C * (3 * Dk + 2 * Dv) + C * C / 3)
        fk_bwd = th * (18 * C * Dk + 10 * C * Dv + 14 * Dk * Dv + 4 * C * C)
        fk_prod = th * (6 * Dk * Dv + 6 * C * Dv + 3 * C * Dk)
        m["prep"] = dict(flops=0.0, bytes=qk)
        m["kc_chunk"] = dict(flops=fk_chunk, bytes=qk + vv + gin)
        m["kc_scan"] = dict(flops=f_scan, bytes=st + vv + st + ckpt)
        m["kc_bwd_scan"] = dict(flops=f_bscan, bytes=vv + st + st)
        m["kc_bwd_prod"] = dict(flops=fk_prod, bytes=ckpt + 3 * vv)
        fk_gate = th * 2 * C * C
        m["kc_bwd_gate"] = dict(flops=fk_gate, bytes=2 * B * T * Hv * es)
        m["kc_bwd_chan"] = dict(flops=fk_bwd - f_bscan - fk_prod - fk_gate,
                                bytes=qk + gin + B * T * Hv * Dk * es)
        m["kc_fwd"] = dict(flops=7.0 * th * Dk * Dv, bytes=qk + vv + gin + vv + 2 * st + ckpt)
        m["kc_bwd"] = dict(flops=20.0 * th * Dk * Dv,
                           bytes=qk + 2 * vv + gin + st + ckpt + vv + gin + st)
        m["bwd_reduce"] = dict(flops=0.0, bytes=2 * qk)
        m["_step"] = dict(bytes=(qk + 2 * vv + gin + 2 * st) + (2 * qk + 3 * vv + 2 * gin + 2 * st)
                          + 2 * ckpt, flops=fk_chunk + f_scan + fk_bwd)
    return m


def design_model(w, conv_k=0, gates="ab", nseg=1, nseg_bwd=1):
    """Per-phase bytes this implementation has to move at the least, in the
    storage formats its kernels use (not the method's algorithmic bytes): bf16
    inputs keep the saved intermediates as bf16 operand images (checkpoints,
    T, W, P, Delta as hi + lo, state cotangents, -Dbar, the q / k rows of each
    chunk) and the per-value-head q / k cotangents in bf16, fp32 inputs all of
    them as fp32 arrays.  Reported beside the roofline as design_bytes."""
    es = 2 if w.dtype == torch.bfloat16 else 4
    img = 2 if w.dtype == torch.bfloat16 else 4  # checkpoint / T / cotangent images
    B, T, Hk, Hv, Dk, Dv = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv
    NC = (T + C - 1) // C
    Tp = NC * C
    BH, BHk = B * Hv, B * Hk
    units = BH * NC  # (b, h, chunk)
    qk = BHk * NC * 2 * C * Dk * es  # q and k tiles, read once per key head
    m = {}
    # a, b, q, k in; Gamma (fp64), beta, r_q, r_k out, and on the tensor-core
    # path the q / k chunk images
    m["prep"] = dict(flops=0.0, bytes=2 * B * T * Hv * es + 2 * B * T * Hk * Dk * es
                     + 2 * BH * Tp * 4 + BH * Tp * 8 + 2 * BHk * Tp * 4
                     + (qk if w.dtype == torch.bfloat16 else 0))
    # q, k, v tiles in; W, P, T images and U (fp32) out
    m["fwd_chunk"] = dict(
        flops=units * (6 * C * C * Dk + 2 * C * C * Dv + C ** 3 / 3),
        bytes=qk + units * (C * Dv * es + 2 * C * 4 + C * 8
                            + C * Dk * es + C * C * es + C * C * img + C * Dv * 4))
    # W, P, q, k, U in; checkpoint image, Delta (hi + lo) and o out
    m["fwd_scan"] = dict(
        flops=units * (6 * C * Dk * Dv + 2 * C * C * Dv),
        bytes=qk + units * (C * Dk * es + C * C * es + C * Dv * 4 + Dk * Dv * img
                            + C * Dv * 4 + C * Dv * es) + 2 * BH * Dk * Dv * 4)
    if nseg > 1:
        # segmented scan: the maps scan segments 0 .. nseg - 2 over Wd = Dv + Dk
        # (padded) columns (W, P, q, k images and U in, the maps out); the chain
        # reads each map once and writes each start state; the scan proper then
        # also reads the start states
        L = -(-NC // nseg)
        Wd = Dv + -(-Dk // 128) * 128
        mu = BH * (nseg - 1) * L
        m["fwd_seg_maps"] = dict(
            flops=mu * (6 * C * Dk * Wd + 2 * C * C * Wd),
            bytes=mu * (C * Dk * es + C * C * es + 2 * C * Dk * es + C * Dv * 4)
            + BH * (nseg - 1) * Dk * Wd * 4)
        m["fwd_seg_chain"] = dict(
            flops=BH * (nseg - 1) * 2 * Dk * Dk * Dv,
            bytes=BH * (nseg - 1) * Dk * (Wd + Dv) * 4)
        m["fwd_scan"]["bytes"] += BH * (nseg - 1) * Dk * Dv * 4
    if nseg_bwd > 1:
        # the reverse scan in segments: maps (dO, P, k, q, W in; maps out), the chain
        Lb = -(-NC // nseg_bwd)
        Wd = Dv + -(-Dk // 128) * 128
        mb = BH * (nseg_bwd - 1) * Lb
        m["bwd_seg_maps"] = dict(
            flops=mb * (6 * C * Dk * Wd + 2 * C * C * Wd),
            bytes=mb * (C * Dv * es + C * C * es + 3 * C * Dk * es)
            + BH * (nseg_bwd - 1) * Dk * Wd * 4)
        m["bwd_seg_chain"] = dict(
            flops=BH * (nseg_bwd - 1) * 2 * Dk * Dk * Dv,
            bytes=BH * (nseg_bwd - 1) * Dk * (Wd + Dv) * 4)
    # dO, P, k, q, W in; chunk-end cotangent and -Dbar images out
    m["bwd_scan"] = dict(
        flops=units * (6 * C * Dk * Dv + 2 * C * C * Dv),
        bytes=qk + units * (C * Dv * es + C * C * es + C * Dk * es + Dk * Dv * img + C * Dv * img)
        + BH * Dk * Dv * 4)
    # checkpoint and cotangent images, Delta, -Dbar, T, q, k, dO, v in;
    # dq, dk per value head, dv, log-decay and beta cotangents out
    m["bwd_chunk"] = dict(
        flops=units * (6 * C * C * Dv + 14 * C * C * Dk + 6 * C * Dk * Dv + 4 * C ** 3),
        bytes=qk + units * (2 * Dk * Dv * img + C * Dv * 4 + C * Dv * img + C * C * img
                            + 2 * C * Dv * es + 4 * C * 4
                            + 2 * C * Dk * img + C * Dv * es + 2 * C * 4))
    # the reverse scan and the per-chunk gradients as one launch (the images the
    # first writes and the second reads counted in both)
    m["bwd_scan_chunk"] = dict(flops=m["bwd_scan"]["flops"] + m["bwd_chunk"]["flops"],
                               bytes=m["bwd_scan"]["bytes"] + m["bwd_chunk"]["bytes"])
    m["bwd_reduce"] = dict(
        flops=0.0,
        bytes=2 * BH * T * Dk * img + 4 * BHk * T * Dk * es + 2 * BH * T * 4 + 4 * B * T * Hv * es)
    m["decode"] = dict(flops=BH * (4 * Dk * Dv + 2 * Dk),
                       bytes=BH * 2 * Dk * Dv * 4 + BHk * 2 * Dk * es + BH * 2 * Dv * es
                       + BH * 2 * es)
    if conv_k:
        # fused short convolution: the mixed projection, the carried windows in and
        # out and the taps replace the q / k / v reads
        Cm = 2 * Hk * Dk + Hv * Dv
        m["decode"]["flops"] += B * Cm * 2 * conv_k
        m["decode"]["bytes"] += (B * Cm * (1 + 2 * conv_k) + Cm * conv_k) * es \
            - (BHk * 2 * Dk + BH * Dv) * es
    # whole step: inputs and outputs once, plus the chunk checkpoints (in the
    # format stored) written once and read once
    io_fwd = (2 * B * T * Hk * Dk + B * T * Hv * Dv + 2 * B * T * Hv) * es \
        + B * T * Hv * Dv * es + 2 * BH * Dk * Dv * 4
    io_bwd = (2 * B * T * Hk * Dk + 2 * B * T * Hv * Dv + 2 * B * T * Hv) * es \
        + (2 * B * T * Hk * Dk + B * T * Hv * Dv + 2 * B * T * Hv) * es + 2 * BH * Dk * Dv * 4
    ckpt = 2 * units * Dk * Dv * img
    m["_step"] = dict(bytes=io_fwd + io_bwd + ckpt,
                      flops=sum(m[k]["flops"] for k in ("fwd_chunk", "fwd_scan", "bwd_scan",
                                                        "bwd_chunk")))
    if gates == "kc":
        gin = B * T * Hv * (Dk + 1) * es  # log_decay [.., Dk] and beta
        io_in = 2 * B * T * Hk * Dk * es + B * T * Hv * Dv * es + gin
        tok = B * T * Hv
        m["prep"] = dict(flops=0.0, bytes=2 * B * T * Hk * Dk * es + 2 * BHk * Tp * 4)
        # chunked form: per (b, h, chunk) the Q_r, K_d, K_r and W images, P and T
        # images, U (fp32), e_C and the decayed Gram (fp32) out of the chunk
        # kernel; the scans read them as the scalar scans do; the tensor-core
        # gradient pass writes Kbar_d, Qbar_r, Wbar (fp32 rows), Pbar and M1
        # (fp32), which the CUDA-core pass reads with q, k, the gates, T and G
        # and turns into fp32 per-value-head q / k cotangents
        m["kc_chunk"] = dict(
            flops=units * (6 * C * C * Dk + 2 * C * C * Dv + C ** 3 / 3),
            bytes=io_in + units * (4 * C * Dk * es + 2 * C * C * es + C * Dv * 4 + Dk * 4 + C * C * 4))
        m["kc_scan"] = dict(
            flops=units * (6 * C * Dk * Dv + 2 * C * C * Dv),
            bytes=units * (3 * C * Dk * es + C * C * es + C * Dv * 4 + Dk * 4 + Dk * Dv * img
                           + C * Dv * 4 + C * Dv * es) + 2 * BH * Dk * Dv * 4)
        m["kc_bwd_scan"] = dict(
            flops=units * (6 * C * Dk * Dv + 2 * C * C * Dv),
            bytes=units * (C * Dv * es + C * C * es + 3 * C * Dk * es + Dk * 4 + Dk * Dv * img
                           + C * Dv * img) + 2 * BH * Dk * Dv * 4)
        m["kc_bwd_prod"] = dict(
            flops=units * (6 * C * Dk * Dv + 6 * C * C * Dv + 3 * C * C * Dk),
            bytes=units * (2 * C * Dv * es + C * Dv * 4 + C * Dv * img + C * C * img + 2 * Dk * Dv * img
                           + C * Dk * es + 3 * C * C * 4 + C * Dv * es + 3 * C * Dk * 4 + Dk * 4))
        # the gate pass reads beta, T, M and G and writes Gbar over M and the
        # beta cotangent; the channel pass reads q, k, the gates, Pbar, Gbar,
        # Qbar_r, Kbar_d, Kbar_r, ebar and writes the fp32 per-value-head q / k
        # cotangents and the log-decay cotangent
        m["kc_bwd_gate"] = dict(
            flops=units * 4 * C ** 3 / 3,
            bytes=2 * B * T * Hv * es + units * (C * C * img + 3 * C * C * 4))
        m["kc_bwd_chan"] = dict(
            flops=units * 10 * C * C * Dk,
            bytes=2 * B * T * Hk * Dk * es + gin + units * (2 * C * C * 4 + 5 * C * Dk * 4 + Dk * 4)
            + B * T * Hv * Dk * es)
        # recurrent form: fp32 states every 8 steps written and read back, and
        # the per-16-column tile partials of the q / k / log-decay cotangents
        nt, NS = Dv // 16, (T + 7) // 8
        ck = BH * NS * Dk * Dv * 4
        part = BH * nt * Tp * (3 * Dk + 1) * 4
        m["kc_fwd"] = dict(flops=7.0 * tok * Dk * Dv,
                           bytes=io_in + B * T * Hv * Dv * es + 2 * BH * Dk * Dv * 4 + ck)
        m["kc_bwd"] = dict(flops=20.0 * tok * Dk * Dv,
                           bytes=io_in + 2 * B * T * Hv * Dv * es + ck + part
                           + BH * nt * Tp * (Dk + 1) * 4 + gin + 2 * BH * Dk * Dv * 4)
        m["bwd_reduce"] = dict(flops=0.0, bytes=2 * BH * Tp * Dk * 4 + 4 * B * T * Hk * Dk * es)
        m["_step"] = dict(bytes=2 * io_in + 2 * B * T * Hv * Dv * es + gin + 2 * units * Dk * Dv * img
                          + 4 * B * T * Hk * Dk * es + 4 * BH * Dk * Dv * 4,
                          flops=sum(m[k]["flops"] for k in ("kc_chunk", "kc_scan", "kc_bwd_scan",
                                                            "kc_bwd_prod", "kc_bwd_gate", "kc_bwd_chan")))
    return m


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid and not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            cmd += ["-i", uuid]
        except Exception:
            pass
        self.cmd = cmd

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU)
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def make_inputs(w, gates="ab"):
    """The workload's seeded inputs; with gates == "lb" the gates are the
    per-step log_decay and beta (torch-to-nnef page, op contract) instead of
    a, b, A_log, dt_bias."""
    x = wl.make_inputs(w)
    if gates in ("lb", "kc"):
        x.update(wl.make_lb_gates(w) if gates == "lb" else wl.make_kc_gates(w))
        for n in ("a", "b", "A_log", "dt_bias"):
            x.pop(n)
    return x


def oracle_sample(w, key_heads, gates="ab", conv_k=0):
    """Inputs of `w` restricted to the first `key_heads` key-head groups (with
    conv_k, plus the whole mixed projection and its convolution inputs).
    Returns (inputs, fraction of the workload's (b, h) units)."""
    x = make_inputs(w, gates)
    G = w.G
    nh = key_heads * G
    sub = {}
    for n, t in x.items():
        if t is None:
            sub[n] = None
        elif n in ("q", "k"):
            sub[n] = t[:, :, :key_heads]
        elif n in ("v", "d_o", "a", "b", "log_decay", "beta"):
            sub[n] = t[:, :, :nh]
        elif n in ("A_log", "dt_bias"):
            sub[n] = t[:nh]
        elif n in ("state0", "d_state_T"):
            sub[n] = t[:, :nh]
        else:
            sub[n] = t
    if conv_k:
        cvi = wl.make_conv_inputs(w.B, 2 * w.Hk * w.Dk + w.Hv * w.Dv, 1, conv_k, w.dtype,
                                  w.seed + 1)
        sub["hidden"], sub["conv_state"], sub["conv_weight"] = (cvi["hidden"], cvi["conv_state"],
                                                               cvi["weight"])
    return sub, nh / w.Hv


def run_oracle_step(sub, backward, rank=0, iters=3):
    import oracle

    t0 = time.perf_counter()
    if rank:  # rank-r compressed chunk states
        from oracle import compressed as oc

        args = [sub[n] for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")]
        om = wl.make_omega(sub["v"].shape[3], rank)
        if backward:  # the backward reruns the forward for its chunk states
            oc.backward_compressed(*args, sub["d_o"], sub["d_state_T"], om, iters)
        else:
            oc.forward_compressed(*args, om, iters)
        return time.perf_counter() - t0
    if "hidden" in sub:  # the fused decode's convolution (all channels)
        oracle.causal_conv1d_update(sub["hidden"], sub["conv_state"], sub["conv_weight"])
    if "log_decay" in sub:
        args = [sub[n] for n in ("q", "k", "v", "log_decay", "beta", "state0", "mask")]
        kc = sub["log_decay"].dim() == 4  # one decay per key channel
        (oracle.forward_kc if kc else oracle.forward_lb)(*args)
        if backward:
            (oracle.backward_kc if kc else oracle.backward_lb)(*args, sub["d_o"], sub["d_state_T"])
    else:
        args = [sub[n] for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")]
        oracle.forward(*args)
        if backward:
            oracle.backward(*args, sub["d_o"], sub["d_state_T"])
    return time.perf_counter() - t0


# fp64 work of one sample step: the whole 9B layer (B1 T2048 Hv64 Dk192 Dv128,
# about 2 s of fwd+bwd on 16 host cores); larger workloads run on as many of
# their key-head groups as fit in the same budget
ORACLE_SAMPLE_BUDGET = 1 * 2048 * 64 * 192 * 128


def sample_key_heads(w, rank=0):
    per_group = w.B * w.T * w.G * w.Dk * w.Dv
    # the compressed-state oracle's truncations run in numpy: a quarter of the budget
    budget = ORACLE_SAMPLE_BUDGET // (4 if rank else 1)
    return max(1, min(w.Hk, budget // per_group))


def _sample_text(w, kh, frac, backward):
    if kh == w.Hk:
        return (f"the whole workload ({w.B}x{w.T} tokens, {w.Hv} value heads), fp64 "
                f"{'fwd+bwd' if backward else 'fwd'}")
    return (f"{kh} of {w.Hk} key-head groups ({int(round(frac * w.Hv))} of {w.Hv} value heads), "
            f"all {w.B}x{w.T} tokens, fp64 {'fwd+bwd' if backward else 'fwd'}; tokens/s scaled "
            f"by the head fraction")


def cpu_baseline(w, backward, reps=3, gates="ab", conv_k=0, rank=0, iters=3):
    import oracle

    kh = sample_key_heads(w, rank)
    sub, frac = oracle_sample(w, kh, gates, conv_k)
    times = [run_oracle_step(sub, backward, rank, iters) for _ in range(reps)]
    t = statistics.median(times)
    tokens = w.B * w.T
    return {"value": tokens * frac / t, "unit": "tokens/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": _sample_text(w, kh, frac, backward) + f", median of {reps}"}


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    import oracle

    oracle.build()
    backward = w.backward
    kh = sample_key_heads(w, args.compress_rank)
    sub, frac = oracle_sample(w, kh, args.gates, args.fused_conv)
    for _ in range(args.warmup):
        run_oracle_step(sub, backward, args.compress_rank, args.compress_iters)
    times = [run_oracle_step(sub, backward, args.compress_rank, args.compress_iters)
             for _ in range(args.steps)]
    t = sum(times) / len(times)
    tokens = w.B * w.T
    value = tokens * frac / t
    line = {
        "impl": "reference", "metric": METRIC if backward else DECODE_METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3 / frac, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gates, args.fused_conv, args.compress_rank,
                            args.compress_iters),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": _sample_text(w, kh, frac, backward)
                         + f", mean of {args.steps} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, gates="ab", conv_k=0, rank=0, iters=3):
    cfg = _config_of(w, gates, conv_k)
    if rank:
        cfg["compressed_states"] = (f"rank {rank}, {iters} power iterations at every chunk "
                                    "boundary (gdn_forward_compressed / gdn_backward_compressed)")
    return cfg


def _config_of(w, gates="ab", conv_k=0):
    return {"workload": w.name, "B": w.B, "T": w.T, "Hk": w.Hk, "Hv": w.Hv, "Dk": w.Dk,
            "Dv": w.Dv, "chunk": C, "state": "fp32",
            "pass": ("fwd+bwd" if w.backward else
                     f"fwd (decode step, {conv_k}-tap short convolution fused in front)" if conv_k
                     else "fwd (decode step)"),
            "gates": ("log_decay, beta (gdn_forward_lb / gdn_backward_lb)" if gates == "lb"
                      else "per-key-channel log_decay [B, T, Hv, Dk], beta (gdn_forward_kc / "
                      "gdn_backward_kc: the chunked form at bf16, Dk 64 / 128 / 192, Dv 128, "
                      "else the CUDA-core recurrence)" if gates == "kc"
                      else "a, b, A_log, dt_bias"),
            "l2": "flushed between timed steps (256 MiB write outside the events)",
            "phase_times": "a second pass over the same steps with per-phase CUDA events "
                           "(the timed steps carry none)"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, w, world, rank, local):
    from gated_delta_rule_06_gb300 import build as gbuild
    from gated_delta_rule_06_gb300 import ops

    gbuild.build()
    lib = ops.load_library()
    lib.gdn_launch_count.restype = ctypes.c_uint64

    class PhaseTime(ctypes.Structure):
        _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64),
                    ("total_ms", ctypes.c_double)]

    dev = torch.device("cuda", local)
    lb = args.gates in ("lb", "kc")
    kc = args.gates == "kc"
    x = make_inputs(w, args.gates)
    conv_k = args.fused_conv
    if conv_k:  # the mixed projection and its convolution replace q, k, v
        Cm = w.Hk * w.Dk * 2 + w.Hv * w.Dv
        cvi = wl.make_conv_inputs(w.B, Cm, 1, conv_k, w.dtype, w.seed + 1)
        x["hidden"] = cvi["hidden"][:, :, 0].contiguous()
        x["conv_state"] = cvi["conv_state"]
        x["conv_weight"] = cvi["weight"]
        for n in ("q", "k", "v"):
            x.pop(n)
        for n in ("a", "b", "log_decay", "beta"):
            if n in x:
                x[n] = x[n][:, 0].contiguous()
    xd = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    backward = w.backward
    B, T, Hk, Hv, Dk, Dv = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv
    # preallocated outputs / workspaces
    shape = None if conv_k else ops.make_shape(xd["q"], xd["v"], xd["mask"] is not None)
    fo = {"o": torch.empty((B, T, Hv, Dv), dtype=w.dtype, device=dev),
          "state_T": torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)}
    if conv_k:
        fo["final_conv_state"] = torch.empty_like(xd["conv_state"])
    cr, ci = args.compress_rank, args.compress_iters
    omega = wl.make_omega(Dv, cr).to(dev) if cr else None
    if backward:
        if kc:
            sv, wf, wb = ops._kc_sizes(shape)
        elif cr:
            sv, wf, wb = ops.compressed_sizes(shape, cr)
        else:
            sv, wf, wb = ops.saved_bytes(shape), ops.workspace_bytes(shape, 0), \
                ops.workspace_bytes(shape, 1)
        fo["saved"] = torch.empty(sv, dtype=torch.uint8, device=dev)
        fo["ws"] = torch.empty(wf, dtype=torch.uint8, device=dev)
        bo = {"ws": torch.empty(wb, dtype=torch.uint8, device=dev)}
        gate_grads = ((("d_log_decay", xd["log_decay"]), ("d_beta", xd["beta"])) if lb else
                      (("da", xd["a"]), ("db", xd["b"])))
        for n, ref in (("dq", xd["q"]), ("dk", xd["k"]), ("dv", xd["v"])) + gate_grads:
            bo[n] = torch.empty_like(ref)
        if not lb:
            bo["dA_log"] = torch.empty((Hv,), dtype=torch.float32, device=dev)
            bo["ddt_bias"] = torch.empty((Hv,), dtype=torch.float32, device=dev)
        bo["dstate0"] = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)

    def fwd_call(inp, keep_saved):
        if conv_k:
            gates = ({"log_decay": inp["log_decay"], "beta": inp["beta"]} if lb else
                     {"a": inp["a"], "b": inp["b"], "A_log": inp["A_log"],
                      "dt_bias": inp["dt_bias"]})
            ops.decode_conv(inp["hidden"], inp["conv_state"], inp["conv_weight"], inp["state0"],
                            mask=inp["mask"], final_conv_state=fo["final_conv_state"],
                            state_out=fo["state_T"], o=fo["o"], **gates)
        elif kc:
            ops.forward_kc(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                           inp["state0"], inp["mask"], keep_saved=keep_saved, out=fo)
        elif lb:
            ops.forward_lb(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                           inp["state0"], inp["mask"], keep_saved=keep_saved, out=fo)
        elif cr:
            ops.forward_compressed(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["A_log"],
                                   inp["dt_bias"], inp["state0"], inp["mask"], omega=omega,
                                   rank=cr, iters=ci, out=fo)
        else:
            ops.forward(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["A_log"],
                        inp["dt_bias"], inp["state0"], inp["mask"], keep_saved=keep_saved,
                        out=fo)

    def step_fwd(inp):
        fwd_call(inp, True)

    def step_bwd(inp):
        if kc:
            ops.backward_kc(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                            inp["mask"], fo["saved"], inp["d_o"], inp["d_state_T"], out=bo)
        elif lb:
            ops.backward_lb(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                            inp["mask"], fo["saved"], inp["d_o"], inp["d_state_T"], out=bo)
        elif cr:
            ops.backward_compressed(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"],
                                    inp["A_log"], inp["dt_bias"], inp["mask"], fo["saved"],
                                    inp["d_o"], inp["d_state_T"], rank=cr, out=bo)
        else:
            ops.backward(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["A_log"],
                         inp["dt_bias"], inp["mask"], fo["saved"], inp["d_o"],
                         inp["d_state_T"], out=bo)

    def step(inp):
        if backward:
            step_fwd(inp)
            step_bwd(inp)
        else:
            fwd_call(inp, False)
    step.parts = (step_fwd, step_bwd)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step(xd)
    torch.cuda.synchronize()
    # One CUDA graph per step: the step's C-ABI calls (the same kernels on the
    # same buffers) captured once and replayed, so the host's gaps between the
    # launches drop out of the step.  Eager launches where capture is refused.
    graph, per_step = None, None
    launch_mode = "eager launches (--eager)"
    if not args.eager:
        try:
            n_c = lib.gdn_launch_count()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(xd)
            per_step = int(lib.gdn_launch_count() - n_c)
            g.replay()
            torch.cuda.synchronize()
            graph = g
            launch_mode = "one CUDA graph per step (the step's C-ABI calls, captured once, replayed)"
        except Exception as ex:  # capture refused: the eager loop below times the same calls
            torch.cuda.synchronize()
            launch_mode = f"eager launches (graph capture refused: {type(ex).__name__})"

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step(xd)

    # ---- timed region (device time, CUDA events on the launching stream).  The
    # step time carries no per-phase events: recording them between the kernels
    # costs 10 - 30 us a step.  The per-phase times come from a second pass over
    # the same K steps (L2 flushed the same way) with the library's phase events.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    n0 = lib.gdn_launch_count()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = per_step * args.steps if graph is not None else int(lib.gdn_launch_count() - n0)
    barrier(world)
    # phase pass
    lib.gdn_timing_begin()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(xd)
    torch.cuda.synchronize()
    phases = (PhaseTime * 16)()
    cnt = ctypes.c_int(0)
    lib.gdn_timing_end(phases, 16, ctypes.byref(cnt))
    barrier(world)
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    ms_max = max_over_ranks(ms, world)
    tokens = w.B * w.T
    value = tokens * world / (ms_max / 1e3)

    # ---- per-phase roofline of the dominant kernel
    peaks = _peaks()
    seg_ok = shape is not None and args.gates != "kc" and not cr
    nseg = ops.segments_auto(shape) if seg_ok else 1
    nseg_bwd = ops.segments_auto(shape, backward=True) if seg_ok and backward else 1
    if cr:  # the compressed backward picks its own reverse-scan segment count
        nseg_bwd = ops.segments_auto(shape, backward=True)
    model = method_model(w, args.gates, nseg, nseg_bwd, args.fused_conv, cr, ci)
    design = design_model(w, args.fused_conv, args.gates, nseg, nseg_bwd)
    ph = {phases[i].name.decode(): (phases[i].launches, phases[i].total_ms)
          for i in range(cnt.value)}
    dom = max(ph, key=lambda k: ph[k][1])
    dl, dms = ph[dom]
    avg_s = dms / dl / 1e3
    # the model counts a phase's work per step; a phase may launch more than once
    # a step (the compressed form scans and truncates chunk by chunk)
    per_step = max(1.0, dl / args.steps)
    fl, by = model[dom]["flops"] / per_step, model[dom]["bytes"] / per_step
    t_hbm = by / (peaks["hbm_gbs"] * 1e9)
    # bf16 workloads run the chunk contractions on the tensor cores (tcgen05);
    # fp32 workloads run them as FFMA on the CUDA cores
    tensor = w.dtype == torch.bfloat16 and dom in ("fwd_chunk", "fwd_scan", "bwd_scan", "bwd_chunk",
                                                  "bwd_scan_chunk", "fwd_seg_maps", "bwd_seg_maps",
                                                  "kc_scan", "kc_bwd_scan", "kc_bwd_prod")
    cpeak = peaks["bf16_tflops"] if tensor else FP32_ALU_PEAK_TFLOPS
    t_cmp = fl / (cpeak * 1e12)
    traffic = measured_traffic(w.name, dom)
    if t_cmp > t_hbm:
        roof = {"bound": "tensor" if tensor else "alu", "achieved": fl / avg_s / 1e12,
                "peak": cpeak, "unit": "TFLOP/s", "kernel": dom,
                "peak_source": (f"{peaks['source']} bf16_tflops (burst)" if tensor else
                                "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x 2070 MHz")}
    else:
        roof = {"bound": "hbm", "achieved": by / avg_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "kernel": dom, "peak_source": f"{peaks['source']} hbm_gbs"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic
    roof["algorithmic_bytes"] = by
    roof["algorithmic_flops"] = fl
    roof["bytes_basis"] = ("the method's tensors this kernel reads or writes (inputs, outputs, "
                           "cotangents, fp32 chunk checkpoints); no intermediates")
    roof["traffic_over_algorithmic"] = (traffic / by) if traffic else None
    roof["design_bytes"] = design[dom]["bytes"] / per_step if dom in design else None
    roof["launches_per_step"] = per_step
    roof["achieved_tflops"] = fl / avg_s / 1e12
    roof["achieved_gbs"] = by / avg_s / 1e9
    roof["avg_launch_ms"] = avg_s * 1e3
    roof["share"] = dms / sum(v[1] for v in ph.values())

    step_bytes = model["_step"]["bytes"] if backward else model["decode"]["bytes"]
    step_flops = model["_step"]["flops"] if backward else model["decode"]["flops"]
    t_roof = max(step_bytes / (peaks["hbm_gbs"] * 1e9),
                 step_flops / (peaks["bf16_tflops"] * 1e12) if w.dtype == torch.bfloat16 else 0.0)
    step_roof = {"algorithmic_bytes": step_bytes, "algorithmic_flops": step_flops,
                 "achieved_gbs": step_bytes / (ms / 1e3) / 1e9,
                 "frac_of_hbm": step_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                 "roofline_ms": t_roof * 1e3, "frac": t_roof / (ms / 1e3),
                 "peak_source": f"{peaks['source']} hbm_gbs, bf16_tflops"}

    # ---- end to end through the C ABI with host buffers (pinned), copies timed
    if args.no_e2e:
        e2e = None
    elif args.fused_conv or args.gates == "kc" or cr:  # forms the host session does not take
        e2e = run_e2e(args, w, x, xd, fo, bo if backward else None, step, world)
    else:
        e2e = run_e2e_session(args, w, x, world)

    line = {
        "metric": METRIC if backward else DECODE_METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / PAGE_TOKENS_PER_S[w.name]) if w.name in PAGE_TOKENS_PER_S else None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": dict(config_of(w, args.gates, args.fused_conv, cr, ci), launch=launch_mode),
        "clocks": clocks,
        "gpu_launches": launches,
        "roofline": roof,
        "step_roofline": step_roof,
        "phases_ms_per_step": {k: v[1] / args.steps for k, v in ph.items()},
        "wall_s_timed_region": wall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cr:
        kept = ops.compressed_sizes(shape, cr)[0]
        plain = ops.saved_bytes(shape)
        img = B * Hv * ((T + C - 1) // C) * Dk * Dv * 2
        line["compressed_states"] = {
            "rank": cr, "iters": ci, "saved_bytes": kept, "saved_bytes_uncompressed": plain,
            "checkpoint_bytes": kept - (plain - img), "checkpoint_bytes_uncompressed": img,
            "checkpoint_bytes_fp32_states": 2 * img,
            "note": ("checkpoints: the initial state and rank-r factors of each boundary (fp32) "
                     "against one bf16 image per chunk state (and against fp32 states)")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        line["cpu_baseline"] = cpu_baseline(w, backward, gates=args.gates,
                                            conv_k=args.fused_conv, rank=cr, iters=ci)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measured_traffic(workload, kernel):
    """DRAM bytes per launch from a committed ncu capture of this workload, or
    None when there is none or the kernel's sources changed since it was taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            ent = json.load(f).get(workload, {}).get(kernel)
        if not ent:
            return None
        h = hashlib.sha256()
        for src in ent["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return ent["bytes"] if h.hexdigest()[:16] == ent["source_sha256_16"] else None
    except Exception:
        return None


def run_e2e_session(args, w, x, world):
    """Steps on host buffers through the library's host session (gdn_host_step,
    include/gdn_host.h): each step uploads all of its inputs from pinned host
    memory, runs the forward (and the backward) and downloads all of its
    results; the session overlaps one step's copies with its neighbours'
    compute.  Timed on the host clock from a device-wide synchronisation before
    the first step's upload to the end of the last step's download."""
    from gated_delta_rule_06_gb300 import ops

    backward = w.backward
    gates = "lb" if "log_decay" in x else "ab"
    names = ["q", "k", "v"] + (["log_decay", "beta"] if gates == "lb" else
                               ["a", "b", "A_log", "dt_bias"]) + ["state0", "mask"]
    if backward:
        names += ["d_o", "d_state_T"]
    host = {n: x[n].contiguous().pin_memory() for n in names if x.get(n) is not None}
    sess = ops.HostSession(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, w.dtype,
                           has_mask=x.get("mask") is not None, gates=gates, backward=backward)
    outs = [sess.outputs(), sess.outputs()]  # the host side double-buffers its results too
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
    for i in range(max(1, args.warmup)):
        sess.step(host, outs[i & 1])
    sess.sync()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        sess.step(host, outs[i & 1])
    sess.sync()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    sess.close()
    ms = max_over_ranks(ms, world)
    return {"value": w.B * w.T * world / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "api": "gdn_host_step (C ABI, host buffers)",
            "overlap": ("across steps: three device slots; a step's uploads run under the "
                        "previous step's compute, its downloads under the next step's"),
            "timing": "host clock between device-wide synchronisations"}


def run_e2e(args, w, x, xd, fo, bo, step, world):
    dev = fo["o"].device
    names_in = [n for n in ("q", "k", "v", "hidden", "conv_state", "conv_weight", "a", "b",
                            "A_log", "dt_bias", "log_decay", "beta", "state0", "mask", "d_o",
                            "d_state_T") if x.get(n) is not None]
    if not w.backward:
        names_in = [n for n in names_in if n not in ("d_o", "d_state_T")]
    host = {n: x[n].contiguous().pin_memory() for n in names_in}
    dev_in = {n: torch.empty_like(xd[n]) for n in names_in}
    for n in ("q", "k", "v", "hidden", "conv_state", "conv_weight", "a", "b", "A_log",
              "dt_bias", "log_decay", "beta", "state0", "mask", "d_o", "d_state_T"):
        dev_in.setdefault(n, None)
    outs = [fo["o"], fo["state_T"]]
    if "final_conv_state" in fo:
        outs.append(fo["final_conv_state"])
    if bo is not None:
        outs += [bo[n] for n in ("dq", "dk", "dv", "da", "db", "d_log_decay", "d_beta", "dA_log",
                                 "ddt_bias", "dstate0") if n in bo]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)
    stream = torch.cuda.current_stream()
    # Within a step, copies overlap compute where the data flow allows: the
    # backward-only inputs (dO, dS_T) go up while the forward runs, and o and
    # the final state come back while the backward runs.  Each step moves all of
    # its own inputs and results; nothing carries over between steps.
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in, ev_up, ev_fwd, ev_down = (torch.cuda.Event() for _ in range(4))
    bwd_only = [n for n in ("d_o", "d_state_T") if n in host]
    n_fwd_out = 2

    def e2e_step():
        for n, t in host.items():
            if n not in bwd_only:
                dev_in[n].copy_(t, non_blocking=True)
        ev_in.record(stream)
        with torch.cuda.stream(up):
            up.wait_event(ev_in)
            for n in bwd_only:
                dev_in[n].copy_(host[n], non_blocking=True)
            ev_up.record(up)
        if bo is None:
            step(dev_in)
            for h, d in zip(host_out, outs):
                h.copy_(d, non_blocking=True)
            return
        ops_fwd, ops_bwd = step.parts
        ops_fwd(dev_in)
        ev_fwd.record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_fwd)
            for h, d in zip(host_out[:n_fwd_out], outs[:n_fwd_out]):
                h.copy_(d, non_blocking=True)
            ev_down.record(down)
        stream.wait_event(ev_up)
        ops_bwd(dev_in)
        for h, d in zip(host_out[n_fwd_out:], outs[n_fwd_out:]):
            h.copy_(d, non_blocking=True)
        stream.wait_event(ev_down)  # the next step's forward rewrites o and the state

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    ms = max_over_ranks(ms, world)
    r = {"value": w.B * w.T * world / (ms / 1e3), "unit": "tokens/s",
         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms}
    if bo is not None:
        r["overlap"] = ("within a step: dO / dS_T uploaded under the forward, o / final state "
                        "downloaded under the backward")
    return r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen35_9b_layer_T2048_bf16",
                    choices=[n for n in wl.WORKLOAD_ORDER])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of one CUDA graph per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-conv", type=int, default=0, metavar="K",
                    help="decode workloads: run the step with a K-tap short convolution "
                         "fused in front (gdn_decode_conv); 0 = plain decode")
    ap.add_argument("--gates", choices=["ab", "lb", "kc"], default="ab",
                    help="gate inputs: a, b, A_log, dt_bias (default), the per-step "
                         "log_decay and beta (lb), or one log_decay per key channel (kc)")
    ap.add_argument("--compress-rank", type=int, default=0, metavar="R",
                    help="fwd+bwd workloads: truncate the state to rank R (1 .. 16) at every "
                         "chunk boundary and keep rank-R factors in place of the chunk states "
                         "(gdn_forward_compressed / gdn_backward_compressed); 0 = off")
    ap.add_argument("--compress-iters", type=int, default=3, metavar="N",
                    help="power iterations of the truncation (default 3)")
    args = ap.parse_args()
    if args.compress_rank and (not wl.WORKLOADS[args.workload].backward or args.gates != "ab"
                               or args.fused_conv or not 1 <= args.compress_rank <= 16):
        ap.error("--compress-rank R takes 1 <= R <= 16, a fwd+bwd workload and the a / b gates")
    if args.warmup < 3:
        args.warmup = 3
    if args.fused_conv and (wl.WORKLOADS[args.workload].backward or not 1 <= args.fused_conv <= 16):
        ap.error("--fused-conv K takes 1 <= K <= 16 and a decode workload")
    w = wl.WORKLOADS[args.workload]
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
