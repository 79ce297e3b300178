"""The decode step with the short convolution fused in front (gdn_decode_conv)
against the composition of the oracle's causal_conv1d_update and its T = 1
forward: the mixed projection's channels hold q | k | v, head-major.

Tolerances: o at the input dtype's bar (1e-4 fp32, 2e-2 bf16); the fp32
state at 1e-4 (the convolution outputs stay fp32 inside the kernel); the
carried conv state is a copy of input samples and must match exactly.  A
masked row keeps both carried states.
"""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _case(B, Hk, Hv, Dk, Dv, K, dtype, lb, masked, seed):
    from gated_delta_rule_06_gb300 import ops

    w = wl.custom("dconv", B, 1, Hk, Hv, Dk, Dv, dtype=dtype, seed=seed, state_sigma=0.05)
    x = wl.make_inputs(w)
    if lb:
        x.update(wl.make_lb_gates(w, seed))
    C = 2 * Hk * Dk + Hv * Dv
    cv = wl.make_conv_inputs(B, C, 1, K, dtype, seed + 1)
    mask = None
    if masked:
        mask = torch.ones((B, 1), dtype=torch.uint8)
        mask[1::3] = 0
    dev = {n: t.cuda() for n, t in cv.items()}
    gates = ({"log_decay": x["log_decay"][:, 0].cuda(), "beta": x["beta"][:, 0].cuda()} if lb else
             {"a": x["a"][:, 0].cuda(), "b": x["b"][:, 0].cuda(), "A_log": x["A_log"].cuda(),
              "dt_bias": x["dt_bias"].cuda()})
    st = x["state0"].cuda()
    o, sT, fcs = ops.decode_conv(dev["hidden"], dev["conv_state"], dev["weight"], st,
                                 mask=None if mask is None else mask.cuda(), **gates)
    torch.cuda.synchronize()
    # reference: the oracle's convolution, then its recurrence on the split channels
    y, fs_r = oracle.causal_conv1d_update(cv["hidden"], cv["conv_state"], cv["weight"])
    y = y[:, :, 0]
    q = y[:, :Hk * Dk].reshape(B, 1, Hk, Dk)
    k = y[:, Hk * Dk:2 * Hk * Dk].reshape(B, 1, Hk, Dk)
    v = y[:, 2 * Hk * Dk:].reshape(B, 1, Hv, Dv)
    if lb:
        o_r, s_r = oracle.forward_lb(q, k, v, x["log_decay"], x["beta"], x["state0"], mask)
    else:
        o_r, s_r = oracle.forward(q, k, v, x["a"], x["b"], x["A_log"], x["dt_bias"],
                                  x["state0"], mask)
    if mask is not None:
        off = mask[:, 0].numpy() == 0
        fs_r[off] = np64(cv["conv_state"])[off]
    check("o", o, o_r, TOL[dtype])
    check("state_T", sT, s_r, 1e-4)
    np.testing.assert_array_equal(np64(fcs), fs_r)


@pytest.mark.parametrize("lb", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_conv(dtype, lb):
    _case(6, 2, 4, 128, 128, 4, dtype, lb, masked=False, seed=7 + lb)


def test_decode_conv_masked_rows_and_other_widths():
    _case(7, 1, 3, 64, 32, 3, torch.bfloat16, False, masked=True, seed=17)
    _case(5, 2, 2, 96, 64, 1, torch.float32, True, masked=True, seed=27)


def test_decode_conv_rejects_overlapping_conv_state():
    from gated_delta_rule_06_gb300 import ops

    B, Hk, Hv, D, K = 2, 1, 2, 64, 4
    C = 2 * Hk * D + Hv * D
    cv = {n: t.cuda() for n, t in wl.make_conv_inputs(B, C, 1, K, torch.float32, 3).items()}
    z = torch.zeros((B, Hv), device="cuda")
    st = torch.zeros((B, Hv, D, D), device="cuda")
    with pytest.raises(ops.GdnError):
        ops.decode_conv(cv["hidden"], cv["conv_state"], cv["weight"], st, log_decay=z, beta=z,
                        final_conv_state=cv["conv_state"])
