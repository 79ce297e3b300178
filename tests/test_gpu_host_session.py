"""Steps on host buffers (gdn_host_step, include/gdn_host.h) against the fp64
oracle, element by element, at the parity tolerances of the device entry
points (per tensor max|x - y| / max|y|: 1e-4 for fp32 inputs, 2e-2 for bf16).

Each session runs several steps on different seeded inputs, so every device
slot is used and a step whose copies or compute touched its neighbour's slot
would fail its own comparison.  A plumbing check also asks that a session step
give bit-for-bit the results of gdn_forward / gdn_backward on the same inputs
(the session only moves data around those calls).
"""

import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, gpu_backward, gpu_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _ops():
    from gated_delta_rule_06_gb300 import ops

    return ops


def _session(w, gates="ab", backward=True):
    return _ops().HostSession(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, w.dtype,
                              has_mask=w.mask != "none", gates=gates, backward=backward)


def _pinned(x):
    return {k: (None if v is None else v.contiguous().pin_memory()) for k, v in x.items()}


def _oracle_ab(x, backward=True):
    o, s = oracle.forward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                          x["state0"], x["mask"])
    ref = {"o": o, "state_T": s}
    if backward:
        ref.update(oracle.backward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                                   x["dt_bias"], x["state0"], x["mask"], x["d_o"],
                                   x["d_state_T"]))
    return ref


@pytest.mark.parametrize("dtype,Dk,Dv", [(torch.bfloat16, 64, 64), (torch.bfloat16, 192, 128),
                                         (torch.float32, 32, 16)])
def test_training_steps_match_oracle(dtype, Dk, Dv):
    """Four training steps in a row (slots 0, 1, 2, 0), each on its own inputs."""
    w = wl.custom("hs", 2, 130, 2, 4, Dk, Dv, dtype=dtype, seed=301 + Dk,
                  mask="half_second_batch")
    sess = _session(w)
    steps = []
    for i in range(4):
        x = _pinned(wl.make_inputs(w, seed=311 + 7 * i))
        out = sess.outputs()
        sess.step(x, out)
        steps.append((x, out))
    sess.sync()
    tol = TOL[dtype]
    for x, out in steps:
        ref = _oracle_ab(x)
        for n in ("o", "state_T") + oracle.GRAD_NAMES:
            check(n, out[n], ref[n], tol)
    sess.close()


def test_session_step_equals_device_calls():
    """Bit-for-bit the results of gdn_forward / gdn_backward on the same data."""
    w = wl.custom("hseq", 1, 200, 2, 4, 128, 128, dtype=torch.bfloat16, seed=341)
    x = wl.make_inputs(w)
    sess = _session(w)
    out = sess.outputs()
    for _ in range(2):  # the second step runs in slot 1
        sess.step(_pinned(x), out)
    sess.sync()
    xd = to_dev(x)
    o, sT, saved = gpu_forward(xd)
    g = gpu_backward(xd, saved)
    torch.cuda.synchronize()
    assert torch.equal(out["o"], o.cpu()) and torch.equal(out["state_T"], sT.cpu())
    for n in oracle.GRAD_NAMES:
        assert torch.equal(out[n], g[n].cpu()), n
    sess.close()


def test_lb_gates_and_pageable_buffers():
    """The log_decay / beta form, with ordinary (pageable) host tensors."""
    w = wl.custom("hslb", 2, 100, 1, 2, 64, 32, dtype=torch.bfloat16, seed=351,
                  mask="half_second_batch")
    sess = _session(w, gates="lb")
    steps = []
    for i in range(2):
        x = wl.make_inputs(w, seed=361 + i)
        x.update(wl.make_lb_gates(w, seed=371 + i))
        for n in ("a", "b", "A_log", "dt_bias"):
            x.pop(n)
        out = sess.outputs(pin=False)
        sess.step(x, out)
        steps.append((x, out))
    sess.sync()
    for x, out in steps:
        o, s = oracle.forward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                                 x["mask"])
        check("o", out["o"], o, TOL[w.dtype])
        check("state_T", out["state_T"], s, TOL[w.dtype])
        gr = oracle.backward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                                x["mask"], x["d_o"], x["d_state_T"])
        for n in oracle.GRAD_NAMES_LB:
            check(n, out[n], gr[n], TOL[w.dtype])
    sess.close()


@pytest.mark.parametrize("T", [1, 70])
def test_inference_session(T):
    """Forward-only sessions: T = 1 runs the decode kernel, T = 70 the chunked
    forward without a saved buffer."""
    w = wl.custom("hsinf", 4, T, 2, 4, 64, 64, dtype=torch.bfloat16, seed=381 + T,
                  state_sigma=0.05)
    sess = _session(w, backward=False)
    steps = []
    for i in range(3):
        x = _pinned(wl.make_inputs(w, seed=391 + i))
        out = sess.outputs()
        assert set(out) == {"o", "state_T"}
        sess.step(x, out)
        steps.append((x, out))
    sess.sync()
    for x, out in steps:
        ref = _oracle_ab(x, backward=False)
        check("o", out["o"], ref["o"], TOL[w.dtype])
        check("state_T", out["state_T"], ref["state_T"], 1e-4 if T == 1 else TOL[w.dtype])
    sess.close()


def test_step_rejects_wrong_host_tensors():
    ops = _ops()
    w = wl.custom("hsbad", 1, 64, 1, 2, 32, 32, dtype=torch.bfloat16, seed=401)
    sess = _session(w)
    x = wl.make_inputs(w)
    out = sess.outputs(pin=False)
    with pytest.raises(ops.GdnError):
        sess.step({**x, "q": x["q"].float()}, out)  # dtype
    with pytest.raises(ops.GdnError):
        sess.step({**x, "v": x["v"].cuda()}, out)  # device tensor
    with pytest.raises(ops.GdnError):
        sess.step({**x, "q": None}, out)  # a required input (status from the library)
    sess.close()
    with pytest.raises(ops.GdnError):
        sess.step(x, out)  # closed
