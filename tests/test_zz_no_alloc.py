"""gdn_forward_noalloc: the forward for callers that cannot allocate device memory.

Inference runtimes and plugin hosts that forbid allocation while work is being
enqueued, or code recording a CUDA stream capture (where cudaMalloc is not
allowed), need an entry point that takes only inputs and outputs.  This one
keeps its scratch in a fixed device array inside the library.  These tests
call it through the C ABI, twice in a row on different inputs (the array keeps
the previous call's contents).  It runs the same kernels in the same order as
gdn_forward's inference path, so each result must equal that path's bit for
bit; the shape whose automatic segment buffers alone overflow the array runs
the single-pass scan and must equal gdn_forward_segmented with one segment,
and the fp64 oracle within the parity tolerance.  A shape too large for the
array is refused before anything runs.

The file is named so that pytest collects it after every other test file.
"""

import ctypes

import pytest
import torch

from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, oracle_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build, ops

    build.build()
    L = ops.load_library()
    vp = ctypes.c_void_p
    L.gdn_forward_noalloc.argtypes = [ctypes.POINTER(ops.GdnShape)] + [vp] * 12
    L.gdn_forward_noalloc.restype = ctypes.c_int
    L.gdn_noalloc_scratch_bytes.argtypes = []
    L.gdn_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return L


def _noalloc_forward(lib, xd):
    from gated_delta_rule_06_gb300 import ops

    q, v = xd["q"], xd["v"]
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    o = torch.full((B, T, Hv, Dv), float("nan"), dtype=q.dtype, device="cuda")
    sT = torch.full((B, Hv, Dk, Dv), float("nan"), dtype=torch.float32, device="cuda")
    m = xd["mask"]
    shape = ops.make_shape(q, v, m is not None)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.gdn_forward_noalloc(ctypes.byref(shape), p(xd["q"]), p(xd["k"]), p(xd["v"]),
                                 p(xd["a"]), p(xd["b"]), p(xd["A_log"]), p(xd["dt_bias"]),
                                 p(xd["state0"]), p(m), p(o), p(sT),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o, sT


def _reference_forward(xd, segments=None):
    from gated_delta_rule_06_gb300 import ops

    o, sT, _ = ops.forward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                           xd["dt_bias"], xd["state0"], xd["mask"], keep_saved=False,
                           segments=segments)
    return o, sT


@pytest.mark.parametrize("dtype,Dk,Dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 32)])
def test_two_calls_match_gdn_forward(lib, dtype, Dk, Dv):
    for seed in (11, 12):  # two calls in a row, different inputs, shared scratch
        w = wl.custom("noalloc", 2, 200, 2, 4, Dk, Dv, dtype=dtype, seed=seed,
                      mask="half_second_batch", clamp_head=True)
        xd = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
        rc, o, sT = _noalloc_forward(lib, xd)
        assert rc == 0
        o_ref, s_ref = _reference_forward(xd)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(sT, s_ref)


def _fallback_T(lib):
    """The shortest T (B1 Hk1 Hv1 D128 bf16) whose inference workspace exceeds
    the array only through the automatic segment count's buffers."""
    from gated_delta_rule_06_gb300 import ops

    cap = lib.gdn_noalloc_scratch_bytes()
    for T in range(8192, 65536 + 1, 256):
        shape = ops.GdnShape(1, T, 1, 1, 128, 128, 1, 0)
        need = ops.workspace_bytes(shape, 2)
        seg = ops.segment_bytes(shape, 0)
        if need > cap >= need - seg:
            return T
    return None


def test_single_pass_fallback_when_segment_buffers_overflow(lib):
    T = _fallback_T(lib)
    assert T is not None, "no shape reaches the single-pass fallback"
    for seed in (21, 22):  # two calls in a row
        w = wl.custom("noalloc_fb", 1, T, 1, 1, 128, 128, dtype=torch.bfloat16, seed=seed,
                      state_sigma=0.02)
        x = wl.make_inputs(w)
        xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
        rc, o, sT = _noalloc_forward(lib, xd)
        assert rc == 0
        o_ref, s_ref = _reference_forward(xd, segments=1)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(sT, s_ref)
        o_r, s_r = oracle_forward(x)
        check("o", o, o_r, TOL[torch.bfloat16])
        check("state_T", sT, s_r, TOL[torch.bfloat16])


def test_shape_beyond_scratch_is_refused(lib):
    from gated_delta_rule_06_gb300 import ops

    cap = lib.gdn_noalloc_scratch_bytes()
    assert cap == 64 << 20
    # B*Hv = 64 heads, T = 4096, 128 x 128 state: the checkpoints alone exceed 64 MiB
    shape = ops.GdnShape(1, 4096, 16, 64, 128, 128, 1, 0)
    assert ops.workspace_bytes(shape, 2) > cap
    dummy = ctypes.c_void_p(256)  # never dereferenced: the call returns before any launch
    rc = lib.gdn_forward_noalloc(ctypes.byref(shape), dummy, dummy, dummy, dummy, dummy, dummy,
                                 dummy, None, None, dummy, dummy, None)
    assert rc == 3  # GDN_ERR_WORKSPACE_TOO_SMALL
