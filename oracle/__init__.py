"""fp64 CPU oracle for the gated delta rule (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library and
the CUDA library never imports it; the two share only the seeded input
generator, which holds none of the method's arithmetic.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, OpenMP over
independent (batch, value-head) pairs).  This module compiles it on first use
(``build()``) and wraps it with ctypes.  Every function takes and returns
float64 numpy arrays in the op contract's layouts (torch-to-nnef page,
"custom_extractors/gdn", op contract):

    q, k [B, T, Hk, Dk];  v [B, T, Hv, Dv];  a, b [B, T, Hv];
    A_log, dt_bias [Hv];  state [B, Hv, Dk, Dv];  mask [B, T] (bool / uint8);
    o [B, T, Hv, Dv].

The ``*_lb`` functions take the op contract's other gate form instead of
(a, b, A_log, dt_bias): log_decay = log g and beta, both [B, T, Hv].

Inputs may be any real dtype; they are upcast exactly to float64 (bf16 and
fp32 values are representable in fp64), so input rounding is not counted as
oracle error.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

SEGMENT = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into oracle/_build/."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64 = ctypes.c_int64
        dp = ctypes.c_void_p
        lib.gdn_oracle_forward.argtypes = [i64] * 6 + [dp] * 11
        lib.gdn_oracle_forward.restype = ctypes.c_int
        lib.gdn_oracle_forward_chunked.argtypes = [i64] * 7 + [dp] * 11
        lib.gdn_oracle_forward_chunked.restype = ctypes.c_int
        lib.gdn_oracle_forward_monoid.argtypes = [i64] * 7 + [dp] * 11
        lib.gdn_oracle_forward_monoid.restype = ctypes.c_int
        lib.gdn_oracle_backward.argtypes = [i64] * 6 + [dp] * 19
        lib.gdn_oracle_backward.restype = ctypes.c_int
        lib.gdn_oracle_forward_lb.argtypes = [i64] * 6 + [dp] * 9
        lib.gdn_oracle_forward_lb.restype = ctypes.c_int
        lib.gdn_oracle_backward_lb.argtypes = [i64] * 6 + [dp] * 15
        lib.gdn_oracle_backward_lb.restype = ctypes.c_int
        lib.gdn_oracle_forward_kc.argtypes = [i64] * 6 + [dp] * 9
        lib.gdn_oracle_forward_kc.restype = ctypes.c_int
        lib.gdn_oracle_backward_kc.argtypes = [i64] * 6 + [dp] * 15
        lib.gdn_oracle_backward_kc.restype = ctypes.c_int
        lib.gdn_oracle_causal_conv1d_update.argtypes = [i64] * 4 + [dp] * 5
        lib.gdn_oracle_causal_conv1d_update.restype = ctypes.c_int
        lib.gdn_oracle_threads.argtypes = []
        lib.gdn_oracle_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().gdn_oracle_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact fp64 copy on the CPU
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _u8(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x).astype(np.uint8))


def _ptr(x):
    return None if x is None else x.ctypes.data


def _dims(q, v):
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    return B, T, Hk, Hv, Dk, Dv


def forward(q, k, v, a, b, A_log, dt_bias, state0=None, mask=None):
    """Sequential recurrence.  Returns (o, state_T) as float64 arrays."""
    q, k, v, a, b, A_log, dt_bias, state0 = map(_f64, (q, k, v, a, b, A_log, dt_bias, state0))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    o = np.zeros((B, T, Hv, Dv))
    sT = np.zeros((B, Hv, Dk, Dv))
    rc = _load().gdn_oracle_forward(B, T, Hk, Hv, Dk, Dv, *map(_ptr, (
        q, k, v, a, b, A_log, dt_bias, state0, mask, o, sT)))
    if rc:
        raise ValueError(f"oracle forward rejected the shapes (code {rc})")
    return o, sT


def forward_chunked(q, k, v, a, b, A_log, dt_bias, state0=None, mask=None, chunk=64):
    """WY/UT chunked form of the same recurrence.  Returns (o, state_T)."""
    q, k, v, a, b, A_log, dt_bias, state0 = map(_f64, (q, k, v, a, b, A_log, dt_bias, state0))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    o = np.zeros((B, T, Hv, Dv))
    sT = np.zeros((B, Hv, Dk, Dv))
    rc = _load().gdn_oracle_forward_chunked(B, T, Hk, Hv, Dk, Dv, int(chunk), *map(_ptr, (
        q, k, v, a, b, A_log, dt_bias, state0, mask, o, sT)))
    if rc:
        raise ValueError(f"oracle chunked forward rejected the shapes (code {rc})")
    return o, sT


def forward_monoid(q, k, v, a, b, A_log, dt_bias, state0=None, mask=None, seg_len=64):
    """The same recurrence evaluated through its associative form (mlx-lm page,
    "Post-initial-submission extensions", Extension 5): per-step affine maps of
    the state composed into runs of seg_len steps, an exclusive tree prefix over
    the run maps for the run start states, each run replayed from its start.
    Returns (o, state_T)."""
    q, k, v, a, b, A_log, dt_bias, state0 = map(_f64, (q, k, v, a, b, A_log, dt_bias, state0))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    o = np.zeros((B, T, Hv, Dv))
    sT = np.zeros((B, Hv, Dk, Dv))
    rc = _load().gdn_oracle_forward_monoid(B, T, Hk, Hv, Dk, Dv, int(seg_len), *map(_ptr, (
        q, k, v, a, b, A_log, dt_bias, state0, mask, o, sT)))
    if rc:
        raise ValueError(f"oracle monoid forward rejected the arguments (code {rc})")
    return o, sT


def backward(q, k, v, a, b, A_log, dt_bias, state0, mask, d_o, d_state_T=None):
    """Hand-derived sequential VJP.

    Returns a dict with dq, dk, dv, da, db, dA_log, ddt_bias, dstate0
    (float64 arrays, shapes of the corresponding primal inputs).
    """
    q, k, v, a, b, A_log, dt_bias, state0, d_o, d_state_T = map(
        _f64, (q, k, v, a, b, A_log, dt_bias, state0, d_o, d_state_T))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    out = dict(
        dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape),
        da=np.zeros(a.shape), db=np.zeros(b.shape), dA_log=np.zeros(Hv),
        ddt_bias=np.zeros(Hv), dstate0=np.zeros((B, Hv, Dk, Dv)))
    rc = _load().gdn_oracle_backward(B, T, Hk, Hv, Dk, Dv, *map(_ptr, (
        q, k, v, a, b, A_log, dt_bias, state0, mask, d_o, d_state_T,
        out["dq"], out["dk"], out["dv"], out["da"], out["db"], out["dA_log"],
        out["ddt_bias"], out["dstate0"])))
    if rc:
        raise ValueError(f"oracle backward rejected the shapes (code {rc})")
    return out


GRAD_NAMES = ("dq", "dk", "dv", "da", "db", "dA_log", "ddt_bias", "dstate0")


def forward_lb(q, k, v, log_decay, beta, state0=None, mask=None):
    """Sequential recurrence with the gates given as log_decay = log g and beta
    ([B, T, Hv]).  Returns (o, state_T)."""
    q, k, v, log_decay, beta, state0 = map(_f64, (q, k, v, log_decay, beta, state0))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    o = np.zeros((B, T, Hv, Dv))
    sT = np.zeros((B, Hv, Dk, Dv))
    rc = _load().gdn_oracle_forward_lb(B, T, Hk, Hv, Dk, Dv, *map(_ptr, (
        q, k, v, log_decay, beta, state0, mask, o, sT)))
    if rc:
        raise ValueError(f"oracle forward_lb rejected the shapes (code {rc})")
    return o, sT


def backward_lb(q, k, v, log_decay, beta, state0, mask, d_o, d_state_T=None):
    """VJP of forward_lb.  Returns a dict with dq, dk, dv, d_log_decay, d_beta,
    dstate0 (the gate cotangents [B, T, Hv], zero on masked steps)."""
    q, k, v, log_decay, beta, state0, d_o, d_state_T = map(
        _f64, (q, k, v, log_decay, beta, state0, d_o, d_state_T))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    out = dict(
        dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape),
        d_log_decay=np.zeros(log_decay.shape), d_beta=np.zeros(beta.shape),
        dstate0=np.zeros((B, Hv, Dk, Dv)))
    rc = _load().gdn_oracle_backward_lb(B, T, Hk, Hv, Dk, Dv, *map(_ptr, (
        q, k, v, log_decay, beta, state0, mask, d_o, d_state_T,
        out["dq"], out["dk"], out["dv"], out["d_log_decay"], out["d_beta"], out["dstate0"])))
    if rc:
        raise ValueError(f"oracle backward_lb rejected the shapes (code {rc})")
    return out


GRAD_NAMES_LB = ("dq", "dk", "dv", "d_log_decay", "d_beta", "dstate0")


def forward_kc(q, k, v, log_decay, beta, state0=None, mask=None):
    """Sequential recurrence with one decay per key channel (the mlx-lm page's
    vectorised gating, g.ndim == 4): log_decay [B, T, Hv, Dk], beta [B, T, Hv].
    An applied step scales row i of the state by exp(log_decay[..., i]).
    Returns (o, state_T)."""
    q, k, v, log_decay, beta, state0 = map(_f64, (q, k, v, log_decay, beta, state0))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    o = np.zeros((B, T, Hv, Dv))
    sT = np.zeros((B, Hv, Dk, Dv))
    rc = _load().gdn_oracle_forward_kc(B, T, Hk, Hv, Dk, Dv, *map(_ptr, (
        q, k, v, log_decay, beta, state0, mask, o, sT)))
    if rc:
        raise ValueError(f"oracle forward_kc rejected the shapes (code {rc})")
    return o, sT


def backward_kc(q, k, v, log_decay, beta, state0, mask, d_o, d_state_T=None):
    """VJP of forward_kc.  Returns a dict with dq, dk, dv, d_log_decay
    ([B, T, Hv, Dk]), d_beta ([B, T, Hv]) and dstate0; gate cotangents are zero
    on masked steps."""
    q, k, v, log_decay, beta, state0, d_o, d_state_T = map(
        _f64, (q, k, v, log_decay, beta, state0, d_o, d_state_T))
    mask = _u8(mask)
    B, T, Hk, Hv, Dk, Dv = _dims(q, v)
    out = dict(
        dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape),
        d_log_decay=np.zeros(log_decay.shape), d_beta=np.zeros(beta.shape),
        dstate0=np.zeros((B, Hv, Dk, Dv)))
    rc = _load().gdn_oracle_backward_kc(B, T, Hk, Hv, Dk, Dv, *map(_ptr, (
        q, k, v, log_decay, beta, state0, mask, d_o, d_state_T,
        out["dq"], out["dk"], out["dv"], out["d_log_decay"], out["d_beta"], out["dstate0"])))
    if rc:
        raise ValueError(f"oracle backward_kc rejected the shapes (code {rc})")
    return out


GRAD_NAMES_KC = GRAD_NAMES_LB


def causal_conv1d_update(hidden, conv_state, weight):
    """Depthwise causal conv1d + SiLU with a K-sample carry state (torch-to-nnef
    page, CausalConvUpdateReified).  hidden [B, C, S], conv_state [B, C, K],
    weight [C, K].  Returns (out [B, C, S], final_state [B, C, K])."""
    hidden, conv_state, weight = map(_f64, (hidden, conv_state, weight))
    B, C, S = hidden.shape
    K = weight.shape[1]
    out = np.zeros((B, C, S))
    fs = np.zeros((B, C, K))
    rc = _load().gdn_oracle_causal_conv1d_update(B, C, S, K, *map(_ptr, (
        hidden, conv_state, weight, out, fs)))
    if rc:
        raise ValueError(f"oracle causal_conv1d_update rejected the shapes (code {rc})")
    return out, fs
