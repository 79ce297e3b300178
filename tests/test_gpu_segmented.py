"""The segmented (associative) forward scan, gdn_forward_segmented, against the
fp64 oracle.

The chunks are cut into runs; every run's composed affine map but the last is
formed in parallel, the run start states are chained, then every run is scanned
from its start state (mlx-lm page, "Post-initial-submission extensions",
Extension 5: the recurrence as an associative monoid).  The results are those
of the sequential recurrence, so the reference is the oracle's plain forward;
the saved buffer is the plain forward's, so the backward from it is checked
against the oracle's VJP too.

Tolerance: bf16 inputs, per tensor max|x - y| / max|y| <= 2e-2.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, gpu_backward, np64, oracle_backward, oracle_forward, to_dev

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


def _ops():
    from gated_delta_rule_06_gb300 import ops

    return ops


def _fwd(xd, segments, keep_saved=True):
    return _ops().forward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                          xd["dt_bias"], xd["state0"], xd["mask"], keep_saved=keep_saved,
                          segments=segments)


def _phases(fn):
    lib = _ops().load_library()
    lib.gdn_timing_end.argtypes = [ctypes.POINTER(PhaseTime), ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_int)]
    assert lib.gdn_timing_begin() == 0
    out = fn()
    torch.cuda.synchronize()
    buf = (PhaseTime * 16)()
    n = ctypes.c_int(0)
    assert lib.gdn_timing_end(buf, 16, ctypes.byref(n)) == 0
    return out, [buf[i].name.decode() for i in range(n.value)]


@pytest.mark.parametrize("Dk,segments", [(128, 2), (128, 5), (128, 14), (64, 3), (192, 4)])
def test_segmented_forward_parity(Dk, segments):
    """NC = 14 with a ragged tail of 5 steps; batch 1 masked from t = 65; a nonzero
    initial state; runs of 7, 3 (last 2), 1, 5 (last 4) and 4 (last 2) chunks."""
    w = wl.custom("seg", 2, 64 * 13 + 5, 2, 4, Dk, 128, dtype=torch.bfloat16,
                  seed=700 + Dk + segments, mask="half_second_batch")
    x = wl.make_inputs(w)
    assert x["state0"] is not None and float(x["state0"].abs().max()) > 0
    xd = to_dev(x)
    (o, sT, saved), phases = _phases(lambda: _fwd(xd, segments))
    assert "fwd_seg_maps" in phases and "fwd_seg_chain" in phases, phases
    o_r, s_r = oracle_forward(x)
    check("o", o, o_r, TOL[w.dtype])
    check("state_T", sT, s_r, TOL[w.dtype])


def test_backward_from_segmented_saved():
    """The saved buffer of the segmented forward feeds gdn_backward unchanged."""
    w = wl.custom("segb", 1, 64 * 9 + 17, 2, 4, 128, 128, dtype=torch.bfloat16, seed=731)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, saved = _fwd(xd, 3)
    g = gpu_backward(xd, saved)
    torch.cuda.synchronize()
    gr = oracle_backward(x)
    for name in oracle.GRAD_NAMES:
        check(name, g[name], gr[name], TOL[w.dtype])


def test_segmented_matches_plain_and_is_deterministic():
    """Segmented and plain scans agree to the bf16 operand rounding of the state
    products; two segmented runs agree bit for bit."""
    w = wl.custom("segd", 1, 64 * 20, 2, 2, 128, 128, dtype=torch.bfloat16, seed=741)
    xd = to_dev(wl.make_inputs(w))
    o1, s1, _ = _fwd(xd, 1)
    o2, s2, sv2 = _fwd(xd, 6)
    o3, s3, sv3 = _fwd(xd, 6)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3) and torch.equal(s2, s3) and torch.equal(sv2, sv3)
    d = np.abs(np64(o2) - np64(o1)).max() / np.abs(np64(o1)).max()
    assert d <= TOL[w.dtype], d


def test_inference_and_automatic_count():
    """keep_saved=False (the inference workspace plus the segment buffers) and
    segments = 0 (the library's choice, whatever it is on this GPU)."""
    w = wl.custom("segi", 1, 64 * 40 + 3, 1, 2, 128, 128, dtype=torch.bfloat16, seed=751)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o_r, s_r = oracle_forward(x)
    for segments in (8, 0):
        o, sT, saved = _fwd(xd, segments, keep_saved=False)
        assert saved is None
        check("o", o, o_r, TOL[w.dtype])
        check("state_T", sT, s_r, TOL[w.dtype])
    shape = _ops().make_shape(xd["q"], xd["v"], False)
    assert _ops().segments_auto(shape) >= 1


def _bwd(xd, saved, segments):
    return _ops().backward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                           xd["dt_bias"], xd["mask"], saved, xd["d_o"], xd["d_state_T"],
                           segments=segments)


@pytest.mark.parametrize("Dk,fwd_seg,bwd_seg", [(128, 1, 2), (128, 3, 5), (64, 4, 14),
                                                (192, 2, 3)])
def test_segmented_backward_parity(Dk, fwd_seg, bwd_seg):
    """The reverse scan in segments (from the end of the sequence; the first one
    shorter): maps, the chain from a nonzero d_state_T, every segment's scan,
    then the per-chunk gradients.  NC = 14 with a ragged tail, batch 1 masked from
    t = 65, a nonzero initial state; the forward's and the backward's segment
    counts differ."""
    w = wl.custom("segbw", 2, 64 * 13 + 5, 2, 4, Dk, 128, dtype=torch.bfloat16,
                  seed=760 + Dk + bwd_seg, mask="half_second_batch")
    x = wl.make_inputs(w)
    assert float(x["d_state_T"].abs().max()) > 0
    xd = to_dev(x)
    o, sT, saved = _fwd(xd, fwd_seg)
    g, phases = _phases(lambda: _bwd(xd, saved, bwd_seg))
    assert "bwd_seg_maps" in phases and "bwd_seg_chain" in phases and "bwd_chunk" in phases, phases
    gr = oracle_backward(x)
    for name in oracle.GRAD_NAMES:
        check(name, g[name], gr[name], TOL[w.dtype])


def test_segmented_backward_deterministic_and_automatic():
    """Two segmented backward runs agree bit for bit; the automatic count (the
    library's gdn_backward) also meets the bar on a few-heads shape."""
    w = wl.custom("segbd", 1, 64 * 24, 1, 2, 128, 128, dtype=torch.bfloat16, seed=771)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, saved = _fwd(xd, None)
    g1 = _bwd(xd, saved, 6)
    g2 = _bwd(xd, saved, 6)
    torch.cuda.synchronize()
    for name in oracle.GRAD_NAMES:
        assert torch.equal(g1[name], g2[name]), name
    g3, phases = _phases(lambda: _bwd(xd, saved, None))
    gr = oracle_backward(x)
    for name in oracle.GRAD_NAMES:
        check(name, g3[name], gr[name], TOL[w.dtype])


def test_segmented_long_runs():
    """Runs of 33 chunks (NC = 97, three segments forward and backward), the
    length the automatic counts pick for long sequences: the bf16 maps are
    composed over dozens of chunks before the chain uses them."""
    w = wl.custom("seglong", 1, 64 * 96 + 17, 2, 4, 128, 128, dtype=torch.bfloat16, seed=781,
                  state_sigma=0.02)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, saved = _fwd(xd, 3)
    g = _bwd(xd, saved, 3)
    torch.cuda.synchronize()
    o_r, s_r = oracle_forward(x)
    check("o", o, o_r, TOL[w.dtype])
    check("state_T", sT, s_r, TOL[w.dtype])
    gr = oracle_backward(x)
    for name in oracle.GRAD_NAMES:
        check(name, g[name], gr[name], TOL[w.dtype])


def test_automatic_counts_on_this_gpu():
    """The cost models keep the single-pass scans (and the fused backward) at the
    9B layer shape, and split both scans for few heads over a long sequence."""
    ops = _ops()
    nine = ops.GdnShape(1, 2048, 16, 64, 192, 128, 1, 0)
    assert ops.segments_auto(nine) == 1 and ops.segments_auto(nine, backward=True) == 1
    long_ = ops.GdnShape(1, 65536, 4, 8, 128, 128, 1, 0)
    assert ops.segments_auto(long_) > 1 and ops.segments_auto(long_, backward=True) > 1
    n = ctypes.c_size_t()
    lib = ops.load_library()
    assert lib.gdn_segment_bytes(ctypes.byref(nine), 0, ctypes.byref(n)) == 0 and n.value == 0
