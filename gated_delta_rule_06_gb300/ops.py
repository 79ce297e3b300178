"""Thin ctypes binding over libgdn.so (include/gdn.h).

Every step of the computation runs in the library's CUDA kernels; this module
only checks tensors, allocates outputs/workspaces with PyTorch and passes raw
device pointers plus the current CUDA stream.  There is no fallback: if the
library has not been built (``__graft_entry__.build()`` or ``python -m
gated_delta_rule_06_gb300.build``) every call raises.

Layouts (torch-to-nnef "custom_extractors/gdn", op contract; mlx-lm PR "Add
gated_delta_update VJP", signature of gated_delta_update_vjp):
    q, k [B, T, Hk, Dk];  v [B, T, Hv, Dv];  a, b [B, T, Hv];
    A_log, dt_bias [Hv] fp32;  state [B, Hv, Dk, Dv] fp32;  mask [B, T] bool/uint8.
q, k, v, a, b share one dtype: float32 or bfloat16.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgdn.so")

GDN_OK = 0
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


class GdnError(RuntimeError):
    pass


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("Hk", ctypes.c_int64),
                ("Hv", ctypes.c_int64), ("Dk", ctypes.c_int64), ("Dv", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("has_mask", ctypes.c_int32)]


class GdnHostInputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias",
                                               "state0", "mask", "d_o", "d_state_T")]


class GdnHostOutputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("o", "state_T", "dq", "dk", "dv", "da", "db",
                                               "dA_log", "ddt_bias", "dstate0")]


_lock = threading.Lock()
_lib = None

EXPORTS = ("gdn_status_string", "gdn_last_cuda_error", "gdn_workspace_bytes",
           "gdn_saved_bytes", "gdn_forward", "gdn_backward")


def load_library(path: str = LIB_PATH):
    """Load libgdn.so (raises if it is missing) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise GdnError(f"{path} is missing: build the CUDA library first "
                           "(python -m gated_delta_rule_06_gb300.build)")
        lib = ctypes.CDLL(path)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        shp = ctypes.POINTER(GdnShape)
        lib.gdn_status_string.argtypes = [i32]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_last_cuda_error.argtypes = []
        lib.gdn_last_cuda_error.restype = ctypes.c_char_p
        lib.gdn_workspace_bytes.argtypes = [shp, i32, ctypes.POINTER(sz)]
        lib.gdn_workspace_bytes.restype = i32
        lib.gdn_saved_bytes.argtypes = [shp, ctypes.POINTER(sz)]
        lib.gdn_saved_bytes.restype = i32
        lib.gdn_forward.argtypes = [shp] + [vp] * 11 + [vp, sz, vp, sz, vp]
        lib.gdn_forward.restype = i32
        lib.gdn_backward.argtypes = [shp] + [vp] * 9 + [sz] + [vp] * 10 + [vp, sz, vp]
        lib.gdn_backward.restype = i32
        lib.gdn_forward_lb.argtypes = [shp] + [vp] * 9 + [vp, sz, vp, sz, vp]
        lib.gdn_forward_lb.restype = i32
        lib.gdn_forward_segmented.argtypes = [shp, i32] + [vp] * 11 + [vp, sz, vp, sz, vp]
        lib.gdn_forward_segmented.restype = i32
        lib.gdn_backward_segmented.argtypes = [shp, i32] + [vp] * 9 + [sz] + [vp] * 10 + [vp, sz, vp]
        lib.gdn_backward_segmented.restype = i32
        lib.gdn_segment_bytes.argtypes = [shp, i32, ctypes.POINTER(sz)]
        lib.gdn_segment_bytes.restype = i32
        lib.gdn_segments_auto.argtypes = [shp, ctypes.POINTER(i32)]
        lib.gdn_segments_auto.restype = i32
        lib.gdn_backward_segments_auto.argtypes = [shp, ctypes.POINTER(i32)]
        lib.gdn_backward_segments_auto.restype = i32
        lib.gdn_backward_lb.argtypes = [shp] + [vp] * 7 + [sz] + [vp] * 8 + [vp, sz, vp]
        lib.gdn_backward_lb.restype = i32
        lib.gdn_causal_conv1d_update.argtypes = [ctypes.c_int64] * 4 + [i32] + [vp] * 6
        lib.gdn_causal_conv1d_update.restype = i32
        lib.gdn_decode_conv.argtypes = [shp, i32, ctypes.c_int64] + [vp] * 13
        lib.gdn_decode_conv.restype = i32
        lib.gdn_kc_saved_bytes.argtypes = [shp, ctypes.POINTER(sz)]
        lib.gdn_kc_saved_bytes.restype = i32
        lib.gdn_kc_workspace_bytes.argtypes = [shp, i32, ctypes.POINTER(sz)]
        lib.gdn_kc_workspace_bytes.restype = i32
        lib.gdn_forward_kc.argtypes = [shp] + [vp] * 9 + [vp, sz, vp, sz, vp]
        lib.gdn_forward_kc.restype = i32
        lib.gdn_backward_kc.argtypes = [shp] + [vp] * 7 + [sz] + [vp] * 8 + [vp, sz, vp]
        lib.gdn_backward_kc.restype = i32
        lib.gdn_compressed_bytes.argtypes = [shp, i32] + [ctypes.POINTER(sz)] * 3
        lib.gdn_compressed_bytes.restype = i32
        lib.gdn_forward_compressed.argtypes = [shp, i32, i32, vp] + [vp] * 11 + [vp, sz, vp, sz, vp]
        lib.gdn_forward_compressed.restype = i32
        lib.gdn_backward_compressed.argtypes = [shp, i32] + [vp] * 9 + [sz] + [vp] * 10 + [vp, sz, vp]
        lib.gdn_backward_compressed.restype = i32
        lib.gdn_host_session_bytes.argtypes = [shp, i32, ctypes.POINTER(sz)]
        lib.gdn_host_session_bytes.restype = i32
        lib.gdn_host_session_create.argtypes = [shp, i32, i32, vp, sz, vp, ctypes.POINTER(vp)]
        lib.gdn_host_session_create.restype = i32
        lib.gdn_host_step.argtypes = [vp, ctypes.POINTER(GdnHostInputs),
                                      ctypes.POINTER(GdnHostOutputs)]
        lib.gdn_host_step.restype = i32
        lib.gdn_host_session_sync.argtypes = [vp]
        lib.gdn_host_session_sync.restype = i32
        lib.gdn_host_session_destroy.argtypes = [vp]
        lib.gdn_host_session_destroy.restype = i32
        _lib = lib
        return lib


def _check(rc: int):
    if rc != GDN_OK:
        lib = load_library()
        msg = lib.gdn_status_string(rc).decode()
        if "CUDA" in msg:
            msg += f" ({lib.gdn_last_cuda_error().decode()})"
        raise GdnError(msg)


def make_shape(q: torch.Tensor, v: torch.Tensor, has_mask: bool) -> GdnShape:
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    if q.dtype not in _DTYPES:
        raise GdnError(f"unsupported dtype {q.dtype}")
    return GdnShape(B, T, Hk, Hv, Dk, Dv, _DTYPES[q.dtype], int(bool(has_mask)))


def saved_bytes(shape: GdnShape) -> int:
    n = ctypes.c_size_t()
    _check(load_library().gdn_saved_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return n.value


def workspace_bytes(shape: GdnShape, pass_: int) -> int:
    """pass_ 0: training forward, 1: backward, 2: inference forward (no saved)."""
    n = ctypes.c_size_t()
    _check(load_library().gdn_workspace_bytes(ctypes.byref(shape), pass_, ctypes.byref(n)))
    return n.value


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _cuda(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise GdnError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise GdnError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise GdnError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _mask_u8(mask):
    if mask is None:
        return None
    m = mask if mask.dtype == torch.uint8 else mask.to(torch.uint8)
    return _cuda(m.contiguous(), "mask")


def _buf(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def segment_bytes(shape, segments: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().gdn_segment_bytes(ctypes.byref(shape), int(segments), ctypes.byref(n)))
    return n.value


def segments_auto(shape, backward: bool = False) -> int:
    n = ctypes.c_int(0)
    lib = load_library()
    fn = lib.gdn_backward_segments_auto if backward else lib.gdn_segments_auto
    _check(fn(ctypes.byref(shape), ctypes.byref(n)))
    return n.value


def forward(q, k, v, a, b, A_log, dt_bias, state0=None, mask=None, *, keep_saved=True,
            out=None, segments=None):
    """Run gdn_forward (the scan split into segments when the library's
    automatic choice says so).  Returns (o, state_T, saved) with saved=None when
    keep_saved is False (inference).  ``out`` may pass preallocated
    dict(o=, state_T=, saved=, ws=) buffers.  An integer ``segments`` runs
    gdn_forward_segmented with that count instead (1: the plain scan, 0: the
    automatic count); its saved buffer is the same, and ws then also holds the
    segment buffers of that count."""
    dt = q.dtype
    for n, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _cuda(t, n, dt)
    _cuda(A_log, "A_log", torch.float32)
    _cuda(dt_bias, "dt_bias", torch.float32)
    _cuda(state0, "state0", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    out = out or {}
    o = out.get("o")
    if o is None:
        o = torch.empty((B, T, Hv, Dv), dtype=dt, device=q.device)
    sT = out.get("state_T")
    if sT is None:
        sT = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    saved = None
    if keep_saved:
        saved = out.get("saved")
        if saved is None:
            saved = _buf(saved_bytes(shape), q.device)
        ws = out.get("ws")
        if ws is None:
            extra = segment_bytes(shape, segments) if segments is not None else 0
            ws = _buf(workspace_bytes(shape, 0) + extra, q.device)
    else:
        # T == 1 runs the single-step decode kernel, which needs no workspace
        # (it handles Dk * Dv <= 32768 with Dv % 4 == 0); otherwise the chunked
        # forward runs with its intermediates in an inference workspace.
        ws = out.get("ws")
        if ws is None and not (T == 1 and Dk * Dv <= 32768 and Dv % 4 == 0):
            extra = segment_bytes(shape, segments) if segments is not None else 0
            ws = _buf(workspace_bytes(shape, 2) + extra, q.device)
    lib = load_library()
    args = (_p(q), _p(k), _p(v), _p(a), _p(b), _p(A_log), _p(dt_bias),
            _p(state0), _p(m), _p(o), _p(sT), _p(saved),
            ctypes.c_size_t(saved.numel() if saved is not None else 0), _p(ws),
            ctypes.c_size_t(ws.numel() if ws is not None else 0), _stream())
    if segments is None:
        rc = lib.gdn_forward(ctypes.byref(shape), *args)
    else:
        rc = lib.gdn_forward_segmented(ctypes.byref(shape), int(segments), *args)
    _check(rc)
    return o, sT, saved


def decode(q, k, v, a, b, A_log, dt_bias, state, mask=None, *, state_out=None, o=None):
    """One T = 1 step (inference).  ``state_out`` may be ``state`` (in place)."""
    if q.shape[1] != 1:
        raise GdnError("decode takes T == 1")
    outd = {"state_T": state_out, "o": o, "ws": None}
    o, sT, _ = forward(q, k, v, a, b, A_log, dt_bias, state, mask, keep_saved=False,
                       out={k_: v_ for k_, v_ in outd.items() if v_ is not None})
    return o, sT


def backward(q, k, v, a, b, A_log, dt_bias, mask, saved, d_o, d_state_T=None, *, out=None,
             segments=None):
    """Run gdn_backward.  Returns dict(dq, dk, dv, da, db, dA_log, ddt_bias, dstate0).
    An integer ``segments`` runs gdn_backward_segmented with that count instead
    (1: one reverse pass, 0: the automatic count); ws then also holds the
    segment buffers of that count."""
    dt = q.dtype
    _cuda(d_o, "d_o", dt)
    _cuda(d_state_T, "d_state_T", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    out = dict(out or {})
    dev = q.device
    g = {
        "dq": out.get("dq", None), "dk": out.get("dk", None), "dv": out.get("dv", None),
        "da": out.get("da", None), "db": out.get("db", None),
        "dA_log": out.get("dA_log", None), "ddt_bias": out.get("ddt_bias", None),
        "dstate0": out.get("dstate0", None),
    }
    if g["dq"] is None:
        g["dq"] = torch.empty_like(q)
    if g["dk"] is None:
        g["dk"] = torch.empty_like(k)
    if g["dv"] is None:
        g["dv"] = torch.empty_like(v)
    if g["da"] is None:
        g["da"] = torch.empty_like(a)
    if g["db"] is None:
        g["db"] = torch.empty_like(b)
    if g["dA_log"] is None:
        g["dA_log"] = torch.empty((Hv,), dtype=torch.float32, device=dev)
    if g["ddt_bias"] is None:
        g["ddt_bias"] = torch.empty((Hv,), dtype=torch.float32, device=dev)
    if g["dstate0"] is None:
        g["dstate0"] = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)
    ws = out.get("ws")
    if ws is None:
        extra = segment_bytes(shape, segments) if segments is not None else 0
        ws = _buf(workspace_bytes(shape, 1) + extra, dev)
    lib = load_library()
    args = (_p(q), _p(k), _p(v), _p(a), _p(b), _p(A_log), _p(dt_bias),
            _p(m), _p(saved), ctypes.c_size_t(saved.numel()), _p(d_o), _p(d_state_T),
            _p(g["dq"]), _p(g["dk"]), _p(g["dv"]), _p(g["da"]), _p(g["db"]), _p(g["dA_log"]),
            _p(g["ddt_bias"]), _p(g["dstate0"]), _p(ws), ctypes.c_size_t(ws.numel()), _stream())
    if segments is None:
        rc = lib.gdn_backward(ctypes.byref(shape), *args)
    else:
        rc = lib.gdn_backward_segmented(ctypes.byref(shape), int(segments), *args)
    _check(rc)
    return g


# ---- rank-r compressed chunk states --------------------------------------------

def compressed_sizes(shape, rank: int):
    """(saved, forward workspace, backward workspace) bytes of the compressed form."""
    n = [ctypes.c_size_t(0) for _ in range(3)]
    _check(load_library().gdn_compressed_bytes(ctypes.byref(shape), int(rank),
                                               *[ctypes.byref(x) for x in n]))
    return tuple(x.value for x in n)


def forward_compressed(q, k, v, a, b, A_log, dt_bias, state0=None, mask=None, *, omega, rank,
                       iters=3, out=None):
    """Run gdn_forward_compressed: the state truncated to rank `rank` by `iters`
    power iterations from the start block omega ([Dv, rank] fp32) at every
    chunk boundary.  Returns (o, state_T, saved); saved holds rank-r factors
    in place of the chunk states.  ``out`` may pass dict(o=, state_T=, saved=,
    ws=)."""
    dt = q.dtype
    for n, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _cuda(t, n, dt)
    _cuda(A_log, "A_log", torch.float32)
    _cuda(dt_bias, "dt_bias", torch.float32)
    _cuda(state0, "state0", torch.float32)
    _cuda(omega, "omega", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    if tuple(omega.shape) != (Dv, rank):
        raise GdnError(f"omega must be [{Dv}, {rank}], got {tuple(omega.shape)}")
    sv, wf, _ = compressed_sizes(shape, rank)
    out = out or {}
    o = out.get("o")
    if o is None:
        o = torch.empty((B, T, Hv, Dv), dtype=dt, device=q.device)
    sT = out.get("state_T")
    if sT is None:
        sT = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    saved = out.get("saved")
    if saved is None:
        saved = _buf(sv, q.device)
    ws = out.get("ws")
    if ws is None:
        ws = _buf(wf, q.device)
    rc = load_library().gdn_forward_compressed(
        ctypes.byref(shape), int(rank), int(iters), _p(omega), _p(q), _p(k), _p(v), _p(a), _p(b),
        _p(A_log), _p(dt_bias), _p(state0), _p(m), _p(o), _p(sT), _p(saved),
        ctypes.c_size_t(saved.numel()), _p(ws), ctypes.c_size_t(ws.numel()), _stream())
    _check(rc)
    return o, sT, saved


def backward_compressed(q, k, v, a, b, A_log, dt_bias, mask, saved, d_o, d_state_T=None, *, rank,
                        out=None):
    """Run gdn_backward_compressed on the saved buffer of forward_compressed
    (same rank).  Returns dict(dq, dk, dv, da, db, dA_log, ddt_bias, dstate0)."""
    dt = q.dtype
    _cuda(d_o, "d_o", dt)
    _cuda(d_state_T, "d_state_T", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    out = dict(out or {})
    dev = q.device
    g = {n: out.get(n) for n in ("dq", "dk", "dv", "da", "db", "dA_log", "ddt_bias", "dstate0")}
    for n, ref in (("dq", q), ("dk", k), ("dv", v), ("da", a), ("db", b)):
        if g[n] is None:
            g[n] = torch.empty_like(ref)
    for n in ("dA_log", "ddt_bias"):
        if g[n] is None:
            g[n] = torch.empty((Hv,), dtype=torch.float32, device=dev)
    if g["dstate0"] is None:
        g["dstate0"] = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)
    ws = out.get("ws")
    if ws is None:
        ws = _buf(compressed_sizes(shape, rank)[2], dev)
    rc = load_library().gdn_backward_compressed(
        ctypes.byref(shape), int(rank), _p(q), _p(k), _p(v), _p(a), _p(b), _p(A_log), _p(dt_bias),
        _p(m), _p(saved), ctypes.c_size_t(saved.numel()), _p(d_o), _p(d_state_T), _p(g["dq"]),
        _p(g["dk"]), _p(g["dv"]), _p(g["da"]), _p(g["db"]), _p(g["dA_log"]), _p(g["ddt_bias"]),
        _p(g["dstate0"]), _p(ws), ctypes.c_size_t(ws.numel()), _stream())
    _check(rc)
    return g


class GatedDeltaRule(torch.autograd.Function):
    """Autograd wrapper: (o, final_state) = gated_delta_rule(q, k, v, a, b,
    A_log, dt_bias, state0, mask), with gradients for every floating input."""

    @staticmethod
    def forward(ctx, q, k, v, a, b, A_log, dt_bias, state0, mask):
        q, k, v, a, b = (t.contiguous() for t in (q, k, v, a, b))
        o, sT, saved = forward(q, k, v, a, b, A_log.contiguous(), dt_bias.contiguous(),
                               None if state0 is None else state0.contiguous(), mask)
        ctx.save_for_backward(q, k, v, a, b, A_log, dt_bias, saved)
        ctx.mask = mask
        ctx.has_state0 = state0 is not None
        return o, sT

    @staticmethod
    def backward(ctx, d_o, d_sT):
        q, k, v, a, b, A_log, dt_bias, saved = ctx.saved_tensors
        if d_o is None:
            d_o = torch.zeros_like(v)
        g = backward(q, k, v, a, b, A_log.contiguous(), dt_bias.contiguous(), ctx.mask, saved,
                     d_o.contiguous(), None if d_sT is None else d_sT.contiguous())
        return (g["dq"], g["dk"], g["dv"], g["da"], g["db"], g["dA_log"], g["ddt_bias"],
                g["dstate0"] if ctx.has_state0 else None, None)


def gated_delta_rule(q, k, v, a, b, A_log, dt_bias, state0=None, mask=None):
    """Differentiable gated delta rule (the C-ABI forward + VJP)."""
    return GatedDeltaRule.apply(q, k, v, a, b, A_log, dt_bias, state0, mask)


# ---- log_decay / beta gate form ----------------------------------------------

def forward_lb(q, k, v, log_decay, beta, state0=None, mask=None, *, keep_saved=True, out=None):
    """Run gdn_forward_lb: the gates given as log_decay = log g (finite, <= 0)
    and beta, both [B, T, Hv] in the dtype of q.  Returns (o, state_T, saved)
    as forward does."""
    dt = q.dtype
    for n, t in (("q", q), ("k", k), ("v", v), ("log_decay", log_decay), ("beta", beta)):
        _cuda(t, n, dt)
    _cuda(state0, "state0", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    out = out or {}
    o = out.get("o")
    if o is None:
        o = torch.empty((B, T, Hv, Dv), dtype=dt, device=q.device)
    sT = out.get("state_T")
    if sT is None:
        sT = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    saved = None
    ws = out.get("ws")
    if keep_saved:
        saved = out.get("saved")
        if saved is None:
            saved = _buf(saved_bytes(shape), q.device)
        if ws is None:
            ws = _buf(workspace_bytes(shape, 0), q.device)
    elif ws is None and not (T == 1 and Dk * Dv <= 32768 and Dv % 4 == 0):
        ws = _buf(workspace_bytes(shape, 2), q.device)
    rc = load_library().gdn_forward_lb(
        ctypes.byref(shape), _p(q), _p(k), _p(v), _p(log_decay), _p(beta), _p(state0), _p(m),
        _p(o), _p(sT), _p(saved), ctypes.c_size_t(saved.numel() if saved is not None else 0),
        _p(ws), ctypes.c_size_t(ws.numel() if ws is not None else 0), _stream())
    _check(rc)
    return o, sT, saved


def backward_lb(q, k, v, log_decay, beta, mask, saved, d_o, d_state_T=None, *, out=None):
    """Run gdn_backward_lb.  Returns dict(dq, dk, dv, d_log_decay, d_beta, dstate0)."""
    dt = q.dtype
    _cuda(d_o, "d_o", dt)
    _cuda(d_state_T, "d_state_T", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    out = dict(out or {})
    dev = q.device
    g = {n: out.get(n) for n in ("dq", "dk", "dv", "d_log_decay", "d_beta", "dstate0")}
    for n, ref in (("dq", q), ("dk", k), ("dv", v), ("d_log_decay", log_decay), ("d_beta", beta)):
        if g[n] is None:
            g[n] = torch.empty_like(ref)
    if g["dstate0"] is None:
        g["dstate0"] = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)
    ws = out.get("ws")
    if ws is None:
        ws = _buf(workspace_bytes(shape, 1), dev)
    rc = load_library().gdn_backward_lb(
        ctypes.byref(shape), _p(q), _p(k), _p(v), _p(log_decay), _p(beta), _p(m), _p(saved),
        ctypes.c_size_t(saved.numel()), _p(d_o), _p(d_state_T), _p(g["dq"]), _p(g["dk"]),
        _p(g["dv"]), _p(g["d_log_decay"]), _p(g["d_beta"]), _p(g["dstate0"]), _p(ws),
        ctypes.c_size_t(ws.numel()), _stream())
    _check(rc)
    return g


class GatedDeltaRuleLB(torch.autograd.Function):
    """Autograd wrapper of the log_decay / beta form: (o, final_state) =
    gated_delta_rule_lb(q, k, v, log_decay, beta, state0, mask)."""

    @staticmethod
    def forward(ctx, q, k, v, log_decay, beta, state0, mask):
        q, k, v, log_decay, beta = (t.contiguous() for t in (q, k, v, log_decay, beta))
        o, sT, saved = forward_lb(q, k, v, log_decay, beta,
                                  None if state0 is None else state0.contiguous(), mask)
        ctx.save_for_backward(q, k, v, log_decay, beta, saved)
        ctx.mask = mask
        ctx.has_state0 = state0 is not None
        return o, sT

    @staticmethod
    def backward(ctx, d_o, d_sT):
        q, k, v, log_decay, beta, saved = ctx.saved_tensors
        if d_o is None:
            d_o = torch.zeros_like(v)
        g = backward_lb(q, k, v, log_decay, beta, ctx.mask, saved, d_o.contiguous(),
                        None if d_sT is None else d_sT.contiguous())
        return (g["dq"], g["dk"], g["dv"], g["d_log_decay"], g["d_beta"],
                g["dstate0"] if ctx.has_state0 else None, None)


def gated_delta_rule_lb(q, k, v, log_decay, beta, state0=None, mask=None):
    """Differentiable gated delta rule with the gates given as log_decay, beta."""
    return GatedDeltaRuleLB.apply(q, k, v, log_decay, beta, state0, mask)


# ---- causal conv1d update ----------------------------------------------------

def causal_conv1d_update(hidden, conv_state, weight, *, out=None, final_state=None):
    """Depthwise causal conv1d + SiLU with a K-sample carry state
    (gdn_causal_conv1d_update): hidden [B, C, S], conv_state [B, C, K], weight
    [C, K], all of one dtype.  Returns (out [B, C, S], final_state [B, C, K]);
    pass final_state=conv_state to update the state in place."""
    dt = hidden.dtype
    for n, t in (("hidden", hidden), ("conv_state", conv_state), ("weight", weight)):
        _cuda(t, n, dt)
    B, C, S = hidden.shape
    K = weight.shape[1]
    if tuple(conv_state.shape) != (B, C, K) or tuple(weight.shape) != (C, K):
        raise GdnError("causal_conv1d_update: conv_state must be [B, C, K], weight [C, K]")
    if out is None:
        out = torch.empty_like(hidden)
    if final_state is None:
        final_state = torch.empty_like(conv_state)
    rc = load_library().gdn_causal_conv1d_update(
        B, C, S, K, 1 if dt == torch.bfloat16 else 0, _p(hidden), _p(conv_state), _p(weight),
        _p(out), _p(final_state), _stream())
    _check(rc)
    return out, final_state


def decode_conv(hidden, conv_state, conv_weight, state, *, a=None, b=None, A_log=None,
                dt_bias=None, log_decay=None, beta=None, mask=None, final_conv_state=None,
                state_out=None, o=None):
    """One T = 1 step with the short convolution fused in front (gdn_decode_conv).

    hidden [B, C] or [B, C, 1] is the mixed projection q | k | v (C = 2 Hk Dk +
    Hv Dv), conv_state [B, C, K], conv_weight [C, K], state [B, Hv, Dk, Dv]
    (fp32 or None for zeros).  Gates: a, b, A_log, dt_bias, or log_decay, beta
    ([B, Hv] or [B, 1, Hv]).  Returns (o [B, 1, Hv, Dv], state_T,
    final_conv_state); state_out may be state (in place), final_conv_state
    must be a separate buffer."""
    dt = hidden.dtype
    if hidden.dim() == 3:
        hidden = hidden[:, :, 0]
    hidden = hidden.contiguous()
    for n, t in (("hidden", hidden), ("conv_state", conv_state), ("conv_weight", conv_weight)):
        _cuda(t, n, dt)
    lb = log_decay is not None
    ga, gb = (log_decay, beta) if lb else (a, b)
    if ga is None or gb is None:
        raise GdnError("decode_conv: pass a, b, A_log, dt_bias or log_decay, beta")
    _cuda(ga, "a / log_decay", dt)
    _cuda(gb, "b / beta", dt)
    if not lb:
        _cuda(A_log, "A_log", torch.float32)
        _cuda(dt_bias, "dt_bias", torch.float32)
    _cuda(state, "state", torch.float32)
    B, C = hidden.shape
    K = conv_weight.shape[1]
    Hv = ga.shape[-1]
    if state is None and state_out is None:
        raise GdnError("decode_conv: pass state or state_out to give Dk, Dv")
    ref = state if state is not None else state_out
    Dk, Dv = ref.shape[2], ref.shape[3]
    if (C - Hv * Dv) % (2 * Dk) or C <= Hv * Dv:
        raise GdnError("decode_conv: hidden width must be 2 Hk Dk + Hv Dv")
    Hk = (C - Hv * Dv) // (2 * Dk)
    m = _mask_u8(mask)
    shape = GdnShape(B, 1, Hk, Hv, Dk, Dv, _DTYPES[dt], int(m is not None))
    if o is None:
        o = torch.empty((B, 1, Hv, Dv), dtype=dt, device=hidden.device)
    if state_out is None:
        state_out = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=hidden.device)
    if final_conv_state is None:
        final_conv_state = torch.empty_like(conv_state)
    rc = load_library().gdn_decode_conv(
        ctypes.byref(shape), 1 if lb else 0, K, _p(hidden), _p(conv_state), _p(conv_weight),
        _p(final_conv_state), _p(ga), _p(gb), _p(A_log), _p(dt_bias), _p(state), _p(m), _p(o),
        _p(state_out), _stream())
    _check(rc)
    return o, state_out, final_conv_state


def _kc_sizes(shape):
    lib = load_library()
    n = ctypes.c_size_t()
    _check(lib.gdn_kc_saved_bytes(ctypes.byref(shape), ctypes.byref(n)))
    saved = n.value
    _check(lib.gdn_kc_workspace_bytes(ctypes.byref(shape), 0, ctypes.byref(n)))
    wf = n.value
    _check(lib.gdn_kc_workspace_bytes(ctypes.byref(shape), 1, ctypes.byref(n)))
    return saved, wf, n.value


def forward_kc(q, k, v, log_decay, beta, state0=None, mask=None, *, keep_saved=True,
               out=None):
    """gdn_forward_kc: one decay per key channel, log_decay [B, T, Hv, Dk] and
    beta [B, T, Hv] in q's dtype.  Returns (o, state_T, saved) (saved None when
    keep_saved is False).  ``out`` may pass preallocated dict(o=, state_T=,
    saved=, ws=) buffers."""
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_decay, "log_decay"), (beta, "beta")):
        _cuda(t, n, dt)
    _cuda(state0, "state0", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    saved_n, wf, _ = _kc_sizes(shape)
    out = out or {}
    o = out.get("o")
    if o is None:
        o = torch.empty((B, T, Hv, Dv), dtype=dt, device=q.device)
    sT = out.get("state_T")
    if sT is None:
        sT = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    saved = (out.get("saved") if out.get("saved") is not None else _buf(saved_n, q.device)) \
        if keep_saved else None
    ws = out.get("ws") if out.get("ws") is not None else _buf(wf, q.device)
    rc = load_library().gdn_forward_kc(
        ctypes.byref(shape), _p(q), _p(k), _p(v), _p(log_decay), _p(beta), _p(state0), _p(m),
        _p(o), _p(sT), _p(saved), saved_n if keep_saved else 0, _p(ws), wf, _stream())
    _check(rc)
    return o, sT, saved


def backward_kc(q, k, v, log_decay, beta, mask, saved, d_o, d_state_T=None, *, out=None):
    """gdn_backward_kc.  Returns a dict with dq, dk, dv, d_log_decay, d_beta
    (q's dtype) and dstate0 (fp32).  ``out`` may pass preallocated tensors of
    those names and the workspace ``ws``."""
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (log_decay, "log_decay"), (beta, "beta"),
                 (d_o, "d_o")):
        _cuda(t, n, dt)
    _cuda(d_state_T, "d_state_T", torch.float32)
    m = _mask_u8(mask)
    shape = make_shape(q, v, m is not None)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    saved_n, _, wb = _kc_sizes(shape)
    out = out or {}
    g = dict(dq=out.get("dq"), dk=out.get("dk"), dv=out.get("dv"),
             d_log_decay=out.get("d_log_decay"), d_beta=out.get("d_beta"),
             dstate0=out.get("dstate0"))
    for n, ref in (("dq", q), ("dk", k), ("dv", v), ("d_log_decay", log_decay),
                   ("d_beta", beta)):
        if g[n] is None:
            g[n] = torch.empty_like(ref)
    if g["dstate0"] is None:
        g["dstate0"] = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    ws = out.get("ws") if out.get("ws") is not None else _buf(wb, q.device)
    rc = load_library().gdn_backward_kc(
        ctypes.byref(shape), _p(q), _p(k), _p(v), _p(log_decay), _p(beta), _p(m), _p(saved),
        saved_n, _p(d_o), _p(d_state_T), _p(g["dq"]), _p(g["dk"]), _p(g["dv"]),
        _p(g["d_log_decay"]), _p(g["d_beta"]), _p(g["dstate0"]), _p(ws), wb, _stream())
    _check(rc)
    return g


class HostSession:
    """Steps on HOST tensors through gdn_host_step (include/gdn_host.h): the
    library uploads each step's inputs, runs the forward (and the backward) and
    downloads the results, overlapping one step's copies with the compute of
    the steps next to it.  The device arena is a PyTorch allocation owned by
    this object; compute runs on the current CUDA stream at construction.

    ``step(inputs, outputs)`` takes dicts of contiguous CPU tensors (pinned for
    asynchronous copies): inputs q, k, v, a, b (or log_decay, beta when
    ``gates="lb"``), A_log, dt_bias, state0, mask, d_o, d_state_T; outputs o,
    state_T and, for a backward session, dq, dk, dv, da, db (or d_log_decay,
    d_beta), dA_log, ddt_bias, dstate0.  It only enqueues: the step's tensors
    are kept alive here and must be left alone until ``sync()``."""

    _IN = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask", "d_o", "d_state_T")
    _OUT = ("o", "state_T", "dq", "dk", "dv", "da", "db", "dA_log", "ddt_bias", "dstate0")
    _ALIAS = {"log_decay": "a", "beta": "b", "d_log_decay": "da", "d_beta": "db"}

    def __init__(self, B, T, Hk, Hv, Dk, Dv, dtype, *, has_mask=False, gates="ab",
                 backward=True, device="cuda"):
        if dtype not in _DTYPES:
            raise GdnError(f"unsupported dtype {dtype}")
        if gates not in ("ab", "lb"):
            raise GdnError("gates must be 'ab' or 'lb'")
        lib = load_library()
        self._h = None
        self.dtype, self.gates, self.backward = dtype, gates, bool(backward)
        self.shape = GdnShape(B, T, Hk, Hv, Dk, Dv, _DTYPES[dtype], int(bool(has_mask)))
        n = ctypes.c_size_t()
        _check(lib.gdn_host_session_bytes(ctypes.byref(self.shape), int(self.backward),
                                          ctypes.byref(n)))
        self.arena_bytes = n.value
        self._arena = torch.empty(n.value, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        _check(lib.gdn_host_session_create(
            ctypes.byref(self.shape), 1 if gates == "lb" else 0, int(self.backward),
            ctypes.c_void_p(self._arena.data_ptr()), n,
            ctypes.c_void_p(torch.cuda.current_stream(self._arena.device).cuda_stream),
            ctypes.byref(h)))
        self._h = h
        self._inflight = []
        f32, dt = torch.float32, dtype
        self._spec = {
            "q": ((B, T, Hk, Dk), dt), "k": ((B, T, Hk, Dk), dt), "v": ((B, T, Hv, Dv), dt),
            "a": ((B, T, Hv), dt), "b": ((B, T, Hv), dt), "A_log": ((Hv,), f32),
            "dt_bias": ((Hv,), f32), "state0": ((B, Hv, Dk, Dv), f32), "mask": ((B, T), torch.uint8),
            "d_o": ((B, T, Hv, Dv), dt), "d_state_T": ((B, Hv, Dk, Dv), f32),
            "o": ((B, T, Hv, Dv), dt), "state_T": ((B, Hv, Dk, Dv), f32),
            "dq": ((B, T, Hk, Dk), dt), "dk": ((B, T, Hk, Dk), dt), "dv": ((B, T, Hv, Dv), dt),
            "da": ((B, T, Hv), dt), "db": ((B, T, Hv), dt), "dA_log": ((Hv,), f32),
            "ddt_bias": ((Hv,), f32), "dstate0": ((B, Hv, Dk, Dv), f32)}

    def _host(self, name, t):
        shape, dt = self._spec[name]
        if t.is_cuda or not t.is_contiguous() or t.dtype != dt or tuple(t.shape) != shape:
            raise GdnError(f"{name}: expected a contiguous CPU tensor {dt} {shape}, got "
                           f"{t.device} {t.dtype} {tuple(t.shape)}")
        return ctypes.c_void_p(t.data_ptr())

    def outputs(self, pin=True):
        """Fresh host output tensors for one step (page-locked by default)."""
        names = self._OUT if self.backward else ("o", "state_T")
        rename = {}
        if self.gates == "lb":
            names = [n for n in names if n not in ("dA_log", "ddt_bias")]
            rename = {"da": "d_log_decay", "db": "d_beta"}
        return {rename.get(n, n): torch.empty(self._spec[n][0], dtype=self._spec[n][1],
                                              pin_memory=pin) for n in names}

    def step(self, inputs: dict, outputs: dict):
        if self._h is None:
            raise GdnError("session is closed")
        ins, outs = GdnHostInputs(), GdnHostOutputs()
        for k, t in inputs.items():
            if t is None:
                continue
            n = "mask" if k == "mask" else self._ALIAS.get(k, k)
            if n not in self._IN:
                raise GdnError(f"unknown input {k}")
            if n == "mask" and t.dtype != torch.uint8:
                raise GdnError("mask: expected a uint8 host tensor")
            setattr(ins, n, self._host(n, t))
        for k, t in outputs.items():
            n = self._ALIAS.get(k, k)
            if n not in self._OUT:
                raise GdnError(f"unknown output {k}")
            setattr(outs, n, self._host(n, t))
        _check(load_library().gdn_host_step(self._h, ctypes.byref(ins), ctypes.byref(outs)))
        self._inflight.append((inputs, outputs))

    def sync(self):
        """Wait for every enqueued step; their output tensors are then complete."""
        if self._h is not None:
            _check(load_library().gdn_host_session_sync(self._h))
        self._inflight.clear()

    def close(self):
        if self._h is not None:
            h, self._h = self._h, None
            _check(load_library().gdn_host_session_destroy(h))
        self._inflight.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
