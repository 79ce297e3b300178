"""The log_decay / beta gate form (torch-to-nnef page, op contract: log_decay
and beta [b, S, hv]) through the C ABI (gdn_forward_lb / gdn_backward_lb)
against the fp64 oracle's forward_lb / backward_lb, element by element.

Tolerances are those of the a / b form: per tensor max|x - y| / max|y|, 1e-4
for fp32 inputs and 2e-2 for bf16 inputs.  q, k, v, the state, the
cotangents, the mask and the gates (``make_lb_gates``: log_decay = -exp(u),
u ~ U(ln 0.01, ln 4), value head 0 at -50, beta ~ U(0, 1)) come from the
shared seeded generator.
"""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, np64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _lb_inputs(w, seed):
    x = wl.make_inputs(w)
    x.update(wl.make_lb_gates(w, seed))
    for n in ("a", "b", "A_log", "dt_bias"):
        x.pop(n)
    return x


def _ops():
    from gated_delta_rule_06_gb300 import ops

    return ops


def _parity(w, seed, backward=True):
    ops = _ops()
    x = _lb_inputs(w, seed)
    xd = to_dev(x)
    tol = TOL[w.dtype]
    o, sT, saved = ops.forward_lb(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                  xd["state0"], xd["mask"])
    torch.cuda.synchronize()
    o_r, s_r = oracle.forward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"],
                                 x["state0"], x["mask"])
    errs = {}
    check("o", o, o_r, tol, errs)
    check("state_T", sT, s_r, tol, errs)
    if backward:
        g = ops.backward_lb(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["mask"],
                            saved, xd["d_o"], xd["d_state_T"])
        torch.cuda.synchronize()
        gr = oracle.backward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                                x["mask"], x["d_o"], x["d_state_T"])
        for n in oracle.GRAD_NAMES_LB:
            check(n, g[n], gr[n], tol, errs)
        if x["mask"] is not None:  # masked steps carry no gate cotangent
            off = (x["mask"] == 0).to("cuda")
            assert torch.all(g["d_log_decay"][off] == 0) and torch.all(g["d_beta"][off] == 0)
    return errs


def test_lb_fp32_masked_gqa():
    """fp32 (CUDA-core path): B2 T129 Hk2 Hv4 Dk32 Dv16, batch 1 masked from t = 65."""
    w = wl.custom("lb32", 2, 129, 2, 4, 32, 16, seed=51, mask="half_second_batch")
    _parity(w, seed=52)


@pytest.mark.parametrize("T", [1, 65, 200])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (192, 128)])
def test_lb_bf16_tensor_core(T, Dk, Dv):
    """bf16 on the tensor-core kernels (Dk, Dv multiples of 32), several chunks
    and a ragged tail."""
    w = wl.custom("lbtc", 2, T, 2, 4, Dk, Dv, dtype=torch.bfloat16, seed=61 + T + Dk)
    _parity(w, seed=62 + T)


def test_lb_bf16_masked_outside_tensor_core_range():
    """bf16 with Dk = 40 (not a multiple of 32): the CUDA-core kernels, masked."""
    w = wl.custom("lbff", 2, 100, 1, 2, 40, 24, dtype=torch.bfloat16, seed=71,
                  mask="half_second_batch")
    _parity(w, seed=72)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_lb_decode(dtype):
    """T = 1 without a saved buffer (the fused single-step kernel), masked rows."""
    ops = _ops()
    w = wl.custom("lbdec", 8, 1, 2, 4, 128, 128, dtype=dtype, seed=81, state_sigma=0.02)
    x = _lb_inputs(w, seed=82)
    x["mask"] = torch.tensor([[1], [0], [1], [1], [0], [1], [1], [1]], dtype=torch.uint8)
    xd = to_dev(x)
    o, sT, saved = ops.forward_lb(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                  xd["state0"], xd["mask"], keep_saved=False)
    assert saved is None
    o_r, s_r = oracle.forward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"],
                                 x["state0"], x["mask"])
    check("o", o, o_r, TOL[dtype])
    check("state_T", sT, s_r, 1e-4)  # fp32 state update


def test_lb_deterministic_bitwise():
    ops = _ops()
    w = wl.custom("lbdet", 1, 150, 2, 4, 128, 128, dtype=torch.bfloat16, seed=91)
    xd = to_dev(_lb_inputs(w, seed=92))
    outs = []
    for _ in range(2):
        o, sT, saved = ops.forward_lb(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                      xd["state0"], xd["mask"])
        g = ops.backward_lb(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["mask"],
                            saved, xd["d_o"], xd["d_state_T"])
        outs.append([o, sT] + [g[n] for n in oracle.GRAD_NAMES_LB])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_lb_autograd_function():
    ops = _ops()
    w = wl.custom("lbag", 1, 90, 2, 4, 32, 16, seed=101)
    x = _lb_inputs(w, seed=102)
    xd = to_dev(x)
    leaves = {n: xd[n].clone().requires_grad_(True)
              for n in ("q", "k", "v", "log_decay", "beta", "state0")}
    o, sT = ops.gated_delta_rule_lb(leaves["q"], leaves["k"], leaves["v"], leaves["log_decay"],
                                    leaves["beta"], leaves["state0"], None)
    loss = (o * xd["d_o"]).sum() + (sT * xd["d_state_T"]).sum()
    loss.backward()
    gr = oracle.backward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                            None, x["d_o"], x["d_state_T"])
    for n, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("log_decay", "d_log_decay"),
                     ("beta", "d_beta"), ("state0", "dstate0")):
        check(gname, leaves[n].grad, gr[gname], 1e-4)

