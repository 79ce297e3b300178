"""Seeded synthetic inputs for the gated delta rule (shared by tests and bench).

This module only draws random numbers with a fixed recipe; it holds none of
the method's arithmetic.  Both the CUDA path and the fp64 oracle consume the
same tensors it returns (the oracle upcasts them exactly to fp64).

Recipe (all draws on the CPU with ``torch.Generator``, in this fixed order:
q, k, v, a, b, A_log, dt_bias, state0, d_o, d_state_T; the mask is fixed by
the workload, not drawn):

* q, k, v, a, b ~ N(0, 1), cast to the workload's input dtype;
* A_log ~ U(0, ln 16) (the toy/mask workloads) or ln U(1, 16) (the layer,
  training-batch and decode workloads), fp32 per value head;
* dt_bias ~ N(0, 1), fp32 per value head;
* state0 ~ N(0, sigma^2) fp32 with sigma 0.1 (toy/mask), 0.02 (training
  batch, decode) or exactly zero (the 9B layer);
* d_o ~ N(0, 1) in the input dtype; d_state_T ~ N(0, 1) fp32 for the fp32
  workloads, absent (zero) for the bf16 ones.

The log_decay / beta gate form (torch-to-nnef page, op contract) draws its
gates with ``make_lb_gates``: log_decay = -exp(u), u ~ U(ln 0.01, ln 4) (a
decay g between 0.018 and 0.99), value head 0 at -50 (a near-reset every
step), beta ~ U(0, 1), both in the input dtype, from a generator seeded
separately (seed + 7919).

Workload shapes follow the mlx-lm page's toy gradient-check shape and its
Qwen3.5-9B GatedDeltaNet performance shape, and the torch-to-nnef page's
square-width GQA layout.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    dtype: torch.dtype
    a_log: str          # "uniform_log16" (U(0, ln16)) or "log_uniform_1_16" (ln U(1,16))
    state_sigma: float  # 0 -> zero initial state
    d_state: bool       # draw a cotangent for the final state
    mask: str = "none"  # "none" | "half_second_batch"
    clamp_head: bool = False
    backward: bool = True
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hv // self.Hk

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "toy_fp32": Workload("toy_fp32", 1, 8, 2, 4, 16, 8, torch.float32, "uniform_log16",
                         0.1, True, seed=1000),
    "chunk_mask_fp32": Workload("chunk_mask_fp32", 2, 129, 4, 8, 64, 64, torch.float32,
                                "uniform_log16", 0.1, True, mask="half_second_batch",
                                clamp_head=True, seed=1001),
    "qwen35_9b_layer_T2048_bf16": Workload("qwen35_9b_layer_T2048_bf16", 1, 2048, 16, 64,
                                           192, 128, torch.bfloat16, "log_uniform_1_16", 0.0,
                                           False, seed=1002),
    "gqa_train_B4_T4096_bf16": Workload("gqa_train_B4_T4096_bf16", 4, 4096, 16, 32, 128, 128,
                                        torch.bfloat16, "log_uniform_1_16", 0.02, False,
                                        seed=1003),
    "decode_B256_bf16": Workload("decode_B256_bf16", 256, 1, 16, 32, 128, 128, torch.bfloat16,
                                 "log_uniform_1_16", 0.02, False, backward=False, seed=1004),
    # few (batch, head) pairs over a long sequence: the case the segmented scan is for
    "long_B1_T65536_Hv8_bf16": Workload("long_B1_T65536_Hv8_bf16", 1, 65536, 4, 8, 128, 128,
                                        torch.bfloat16, "log_uniform_1_16", 0.02, False,
                                        seed=1005),
}

# index order used in docs and the bench: 0 toy, 1 mask, 2 9B layer, 3 batch, 4 decode
# (then the long-sequence case of the segmented scan)
WORKLOAD_ORDER = ["toy_fp32", "chunk_mask_fp32", "qwen35_9b_layer_T2048_bf16",
                  "gqa_train_B4_T4096_bf16", "decode_B256_bf16", "long_B1_T65536_Hv8_bf16"]


def custom(name: str, B: int, T: int, Hk: int, Hv: int, Dk: int, Dv: int,
           dtype: torch.dtype = torch.float32, seed: int = 0, state_sigma: float = 0.1,
           d_state: bool = True, mask: str = "none", clamp_head: bool = False,
           a_log: str = "uniform_log16") -> Workload:
    """A workload with an arbitrary shape and the same distributions."""
    return Workload(name, B, T, Hk, Hv, Dk, Dv, dtype, a_log, state_sigma, d_state,
                    mask=mask, clamp_head=clamp_head, seed=seed)


def _normal(gen, shape, dtype, sigma=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(dtype)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw the inputs of one workload on the CPU.

    Returns a dict with q, k, v, a, b, A_log, dt_bias, state0 (or None), mask
    (uint8 [B, T] or None), d_o and d_state_T (or None).
    """
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, T, Hk, Hv, Dk, Dv = w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv
    x = {}
    x["q"] = _normal(gen, (B, T, Hk, Dk), w.dtype)
    x["k"] = _normal(gen, (B, T, Hk, Dk), w.dtype)
    x["v"] = _normal(gen, (B, T, Hv, Dv), w.dtype)
    a = torch.randn((B, T, Hv), generator=gen, dtype=torch.float32)
    x["b"] = _normal(gen, (B, T, Hv), w.dtype)
    if w.a_log == "uniform_log16":
        A_log = torch.rand((Hv,), generator=gen, dtype=torch.float32) * math.log(16.0)
    elif w.a_log == "log_uniform_1_16":
        A_log = torch.log(1.0 + 15.0 * torch.rand((Hv,), generator=gen, dtype=torch.float32))
    else:
        raise ValueError(w.a_log)
    x["dt_bias"] = torch.randn((Hv,), generator=gen, dtype=torch.float32)
    if w.clamp_head:
        # one head on the softplus clamp path: A_log = 5, a = 15
        A_log[0] = 5.0
        a[:, :, 0] = 15.0
    x["a"] = a.to(w.dtype)
    x["A_log"] = A_log
    if w.state_sigma > 0:
        x["state0"] = torch.randn((B, Hv, Dk, Dv), generator=gen,
                                  dtype=torch.float32) * w.state_sigma
    else:
        x["state0"] = None
    x["d_o"] = _normal(gen, (B, T, Hv, Dv), w.dtype)
    x["d_state_T"] = (torch.randn((B, Hv, Dk, Dv), generator=gen, dtype=torch.float32)
                      if w.d_state else None)
    if w.mask == "none":
        x["mask"] = None
    elif w.mask == "half_second_batch":
        m = torch.ones((B, T), dtype=torch.uint8)
        if B > 1:
            m[1, 65:] = 0
        x["mask"] = m
    else:
        raise ValueError(w.mask)
    return x


def make_lb_gates(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw log_decay and beta ([B, T, Hv], input dtype) for the log_decay /
    beta gate form; the recipe is in the module docstring."""
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 7919)
    shape = (w.B, w.T, w.Hv)
    u = torch.rand(shape, generator=gen, dtype=torch.float64)
    lo, hi = math.log(0.01), math.log(4.0)
    ld = -torch.exp(lo + u * (hi - lo))
    ld[:, :, 0] = -50.0
    beta = torch.rand(shape, generator=gen, dtype=torch.float64)
    return {"log_decay": ld.to(w.dtype), "beta": beta.to(w.dtype)}


def make_kc_gates(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw per-key-channel log_decay ([B, T, Hv, Dk]) and beta ([B, T, Hv]) in
    the input dtype: log_decay = -exp(u), u ~ U(ln 0.01, ln 4) per channel, with
    channel 0 of value head 0 at -50 (that channel is cleared every step);
    beta ~ U(0, 1)."""
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 104729)
    u = torch.rand((w.B, w.T, w.Hv, w.Dk), generator=gen, dtype=torch.float64)
    lo, hi = math.log(0.01), math.log(4.0)
    ld = -torch.exp(lo + u * (hi - lo))
    ld[:, :, 0, 0] = -50.0
    beta = torch.rand((w.B, w.T, w.Hv), generator=gen, dtype=torch.float64)
    return {"log_decay": ld.to(w.dtype), "beta": beta.to(w.dtype)}


def make_conv_inputs(B: int, C: int, S: int, K: int, dtype: torch.dtype = torch.float32,
                     seed: int = 0) -> dict:
    """Inputs of the causal conv1d update: hidden [B, C, S] ~ N(0, 1), conv_state
    [B, C, K] ~ N(0, 1), weight [C, K] ~ N(0, 1/K), in this draw order, in the
    input dtype."""
    gen = torch.Generator().manual_seed(seed)
    return {"hidden": _normal(gen, (B, C, S), dtype),
            "conv_state": _normal(gen, (B, C, K), dtype),
            "weight": _normal(gen, (C, K), dtype, sigma=1.0 / math.sqrt(K))}


def make_omega(Dv: int, rank: int, seed: int = 0) -> torch.Tensor:
    """The start block of the compressed form's power iteration: [Dv, rank]
    fp32, standard normal, seeded (a random draw of the method, passed in)."""
    gen = torch.Generator().manual_seed(10_000 + seed)
    return torch.randn((Dv, rank), generator=gen, dtype=torch.float32)
