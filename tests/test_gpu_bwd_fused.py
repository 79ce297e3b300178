"""The two launch forms of the tensor-core backward against the fp64 oracle.

* Fused: the reverse scan and the per-chunk gradients in one cooperative launch
  (the scan CTAs publish finished chunks, gradient items wait for theirs) when
  the scan's value tiles leave SMs free.
* Separate launches when the scan's tiles would fill the GPU.

The library's phase timing names the launches that ran, so each case also checks
which form it exercised.  Tolerance: bf16 inputs, 2e-2 per tensor
(max|x - y| / max|y|).
"""

import ctypes

import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, gpu_backward, gpu_forward, to_dev

pytestmark = pytest.mark.gpu


class PhaseTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _run(w, seed):
    from gated_delta_rule_06_gb300 import ops

    lib = ops.load_library()
    lib.gdn_timing_end.argtypes = [ctypes.POINTER(PhaseTime), ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_int)]
    x = wl.make_inputs(w, seed=seed)
    xd = to_dev(x)
    o, sT, saved = gpu_forward(xd)
    assert lib.gdn_timing_begin() == 0
    g = gpu_backward(xd, saved)
    torch.cuda.synchronize()
    buf = (PhaseTime * 16)()
    n = ctypes.c_int(0)
    assert lib.gdn_timing_end(buf, 16, ctypes.byref(n)) == 0
    phases = [buf[i].name.decode() for i in range(n.value)]
    gr = oracle.backward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                         x["state0"], x["mask"], x["d_o"], x["d_state_T"])
    for name in oracle.GRAD_NAMES:
        check(name, g[name], gr[name], TOL[w.dtype])
    return phases


def test_fused_masked_batches():
    w = wl.custom("fz", 2, 130, 2, 4, 64, 128, dtype=torch.bfloat16, seed=501,
                  mask="half_second_batch")
    phases = _run(w, seed=502)
    assert "bwd_scan_chunk" in phases and "bwd_chunk" not in phases, phases


def test_separate_launches_when_scan_tiles_fill_the_gpu():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = sms // 16 + 1  # B * 16 value heads * one tile each > SMs - 8
    w = wl.custom("fzsep", B, 70, 4, 16, 64, 128, dtype=torch.bfloat16, seed=511)
    phases = _run(w, seed=512)
    assert "bwd_scan" in phases and "bwd_chunk" in phases, phases


def test_fused_deterministic_bitwise():
    """Items are taken dynamically, but every output has one writer and a fixed
    order of accumulation: two runs agree bit for bit."""
    w = wl.custom("fzdet", 1, 300, 4, 16, 128, 128, dtype=torch.bfloat16, seed=521)
    xd = to_dev(wl.make_inputs(w))
    outs = []
    for _ in range(2):
        o, sT, saved = gpu_forward(xd)
        g = gpu_backward(xd, saved)
        outs.append([g[n].clone() for n in oracle.GRAD_NAMES])
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
