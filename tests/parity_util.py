"""Helpers shared by the GPU parity tests (CUDA path vs the fp64 oracle)."""

import numpy as np
import torch

import oracle
from gated_delta_rule_06_gb300 import ops

# Parity bar: per tensor, max|x - y| / max|y| (absolute when the reference is
# all zero), 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32
# accumulation.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}

PRIMAL_ORDER = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")


def rel_err(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    if not np.isfinite(x).all():
        return float("inf")
    s = np.abs(y).max() if y.size else 0.0
    d = np.abs(x - y).max() if y.size else 0.0
    return float(d / s) if s > 0 else float(np.abs(x).max() if x.size else 0.0)


def to_dev(x, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in x.items()}


def gpu_forward(xd, keep_saved=True):
    return ops.forward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                       xd["dt_bias"], xd["state0"], xd["mask"], keep_saved=keep_saved)


def gpu_backward(xd, saved):
    return ops.backward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                        xd["dt_bias"], xd["mask"], saved, xd["d_o"], xd["d_state_T"])


def oracle_forward(x):
    return oracle.forward(*[x[n] for n in PRIMAL_ORDER])


def oracle_backward(x):
    return oracle.backward(*[x[n] for n in PRIMAL_ORDER], x["d_o"], x["d_state_T"])


def np64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def check(name, got, ref, tol, errs=None):
    e = rel_err(np64(got) if torch.is_tensor(got) else got, ref)
    if errs is not None:
        errs[name] = e
    assert e <= tol, f"{name}: rel err {e:.3e} > {tol:.1e}"
    return e
