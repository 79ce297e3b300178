"""Helpers shared by the GPU parity tests (CUDA path vs the fp64 oracle)."""

import json
import os

import numpy as np
import torch

import oracle
from gated_delta_rule_06_gb300 import ops

# Parity bar: per tensor, max|x - y| / max|y| (absolute when the reference is
# all zero), 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32
# accumulation.  The same bar also holds on every independent slice of a tensor
# on its own (one batch row and one head), so a head or a batch row whose
# values are small next to the rest cannot hide an error behind the largest
# slice's scale.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}

PRIMAL_ORDER = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")

# Axes that index independent (batch, head) slices, by tensor name:
# [B, T, H, D] -> batch and head; [B, T, H] -> batch and head;
# [B, H, Dk, Dv] -> batch and head; [H] -> head.
SLICE_AXES = {
    "o": (0, 2), "dq": (0, 2), "dk": (0, 2), "dv": (0, 2), "da": (0, 2), "db": (0, 2),
    "d_log_decay": (0, 2), "d_beta": (0, 2),
    "state_T": (0, 1), "dstate0": (0, 1),
    "dA_log": (0,), "ddt_bias": (0,),
}


def rel_err(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    if not np.isfinite(x).all():
        return float("inf")
    s = np.abs(y).max() if y.size else 0.0
    d = np.abs(x - y).max() if y.size else 0.0
    return float(d / s) if s > 0 else float(np.abs(x).max() if x.size else 0.0)


def slice_errs(x, y, axes):
    """rel_err of every slice that fixes the given axes; returns (worst error,
    index of the worst slice)."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    lead = [x.shape[a] for a in axes]
    dst = list(range(len(axes)))
    xs = np.moveaxis(x, axes, dst).reshape(int(np.prod(lead)), -1)
    ys = np.moveaxis(y, axes, dst).reshape(int(np.prod(lead)), -1)
    worst, where = 0.0, None
    for i in range(xs.shape[0]):
        e = rel_err(xs[i], ys[i])
        if e > worst or where is None:
            worst, where = e, np.unravel_index(i, lead)
    return worst, tuple(int(v) for v in where) if where is not None else ()


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


def _log(record):
    """Append one error record to the JSON-lines file named by GDN_PARITY_LOG
    (unset: nothing is written)."""
    path = os.environ.get("GDN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")


def check(name, got, ref, tol, errs=None, slices=True):
    """Whole-tensor relative error, then (for the tensors named in SLICE_AXES,
    unless slices is False) the same error on every (batch, head) slice."""
    x = np64(got) if torch.is_tensor(got) else np.asarray(got, dtype=np.float64)
    e = rel_err(x, ref)
    if errs is not None:
        errs[name] = e
    assert e <= tol, f"{name}: rel err {e:.3e} > {tol:.1e}"
    rec = {"name": name, "shape": list(np.shape(ref)), "tol": tol, "err": e}
    axes = SLICE_AXES.get(name) if slices else None
    if axes is not None and np.ndim(ref) > 0:
        es, where = slice_errs(x, ref, axes)
        rec.update(slice_err=es, worst_slice=list(where))
        if errs is not None:
            errs[name + "@slice"] = es
        _log(rec)
        assert es <= tol, f"{name}: slice {where} rel err {es:.3e} > {tol:.1e}"
    else:
        _log(rec)
    return e
