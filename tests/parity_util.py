"""Helpers shared by the GPU parity tests (CUDA path vs the fp64 oracle)."""

import json
import os

import numpy as np
import torch

import oracle
from gated_delta_rule_06_gb300 import ops

# Parity bar: per tensor, max|x - y| / max|y| (absolute when the reference is
# all zero), 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32
# accumulation.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}

# Per-slice bar.  Every independent (batch, head) slice of a tensor is also
# checked on its own: max|x - y| over the slice divided by the larger of the
# slice's own max|y| and SLICE_FLOOR times the tensor's max|y|.  A slice at
# least a tenth of the tensor's scale is thus held to the bar at its own scale,
# and a smaller one to an absolute error ten times below what the per-tensor
# bar allows, so an error confined to one head or one batch row shows up
# even where that slice's values are small.  (Without a floor, a slice whose
# exact values vanish, e.g. the log-decay cotangent of a head whose state
# resets every step, would be compared against rounding noise.)
SLICE_FLOOR = 0.1
# The gate cotangents (da, db, their log_decay / beta forms, and the per-head
# sums dA_log, ddt_bias) come from sums with heavy cancellation: per step,
# g <S_bar', S> and its chunked pieces; per head, a sum of those over (b, t).
# The tensor-core path feeds these sums from bf16 operand images of the
# chunk-start state, the chunk-end state cotangent and Delta_bar, so a head
# whose gate cotangents are small next to the terms they are summed from
# carries a larger relative error than the tensor as a whole.  With bf16
# inputs their per-slice bar is 8e-2 (measured worst 6.6e-2, on a head whose
# ddt_bias is under 1 % of the largest head's; every such case stays within
# 2e-2 per tensor).
GATE_COTANGENTS = ("da", "db", "d_log_decay", "d_beta", "dA_log", "ddt_bias")
SLICE_TOL_BF16_GATES = 8e-2

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


def slice_stats(x, y, axes):
    """Per slice that fixes the given axes: (max|x - y|, max|y|), as two arrays
    indexed like the slices, plus the slices' shape."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    lead = [x.shape[a] for a in axes]
    dst = list(range(len(axes)))
    n = int(np.prod(lead))
    xs = np.moveaxis(x, axes, dst).reshape(n, -1)
    ys = np.moveaxis(y, axes, dst).reshape(n, -1)
    if xs.shape[1] == 0:
        return np.zeros(n), np.zeros(n), lead
    d = np.where(np.isfinite(xs).all(axis=1), np.abs(xs - ys).max(axis=1), np.inf)
    return d, np.abs(ys).max(axis=1), lead


def slice_errs(x, y, axes, floor=SLICE_FLOOR):
    """Per-slice error of every slice that fixes the given axes: max|x - y|
    over the slice / max(max|y| over the slice, floor * max|y| over the whole
    tensor), absolute where both are zero.  Returns (worst error, index of the
    worst slice)."""
    d, m, lead = slice_stats(x, y, axes)
    den = np.maximum(m, floor * (float(np.abs(np.asarray(y)).max()) if np.size(y) else 0.0))
    e = np.where(den > 0, d / np.where(den > 0, den, 1.0), d)
    i = int(np.argmax(e))
    return float(e[i]), tuple(int(v) for v in np.unravel_index(i, lead))


def slice_tol(name, tol):
    if name in GATE_COTANGENTS and tol == TOL[torch.bfloat16]:
        return SLICE_TOL_BF16_GATES
    return tol


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
    """Whole-tensor relative error against tol, then (for the tensors named in
    SLICE_AXES, unless slices is False) the per-slice error of every (batch,
    head) slice against slice_tol(name, tol)."""
    x = np64(got) if torch.is_tensor(got) else np.asarray(got, dtype=np.float64)
    e = rel_err(x, ref)
    if errs is not None:
        errs[name] = e
    assert e <= tol, f"{name}: rel err {e:.3e} > {tol:.1e}"
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", ""), "name": name,
           "shape": list(np.shape(ref)), "tol": tol, "err": e,
           "max_ref": float(np.abs(ref).max()) if np.size(ref) else 0.0}
    axes = SLICE_AXES.get(name) if slices else None
    if axes is not None and np.ndim(ref) > 0:
        es, where = slice_errs(x, ref, axes)
        d, m, _ = slice_stats(x, ref, axes)
        rec.update(slice_err=es, worst_slice=list(where), slice_absdiff=d.tolist(),
                   slice_maxref=m.tolist())
        if errs is not None:
            errs[name + "@slice"] = es
        stol = slice_tol(name, tol)
        rec["slice_tol"] = stol
        _log(rec)
        assert es <= stol, f"{name}: slice {where} rel err {es:.3e} > {stol:.1e}"
    else:
        _log(rec)
    return e
