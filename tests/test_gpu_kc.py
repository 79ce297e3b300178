"""Per-key-channel gates (the mlx-lm page's vectorised gating, g.ndim == 4) through
the C ABI (gdn_forward_kc / gdn_backward_kc) against the fp64 oracle's forward_kc
/ backward_kc, element by element.

Tolerances as for the other gate forms: per tensor max|x - y| / max|y|, 1e-4
for fp32 inputs and 2e-2 for bf16 inputs.  q, k, v, the state, the cotangents
and the mask come from the shared seeded generator; the per-channel log-decays
from ``make_kc_gates`` (log_decay = -exp(u), u ~ U(ln 0.01, ln 4), channel 0 of
value head 0 at -50: a channel reset every step).
"""

import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import TOL, check, to_dev

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


def _kc_inputs(w, seed):
    x = wl.make_inputs(w)
    x.update(wl.make_kc_gates(w, seed))
    for n in ("a", "b", "A_log", "dt_bias"):
        x.pop(n)
    return x


def _parity(w, seed):
    ops = _ops()
    x = _kc_inputs(w, seed)
    xd = to_dev(x)
    tol = TOL[w.dtype]
    o, sT, saved = ops.forward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                  xd["state0"], xd["mask"])
    g = ops.backward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["mask"],
                        saved, xd["d_o"], xd["d_state_T"])
    torch.cuda.synchronize()
    o_r, s_r = oracle.forward_kc(x["q"], x["k"], x["v"], x["log_decay"], x["beta"],
                                 x["state0"], x["mask"])
    check("o", o, o_r, tol)
    check("state_T", sT, s_r, tol)
    gr = oracle.backward_kc(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                            x["mask"], x["d_o"], x["d_state_T"])
    for n in oracle.GRAD_NAMES_KC:
        check(n, g[n], gr[n], tol)
    if x["mask"] is not None:  # masked steps carry no gate cotangent
        off = (x["mask"] == 0).to("cuda")
        assert torch.all(g["d_log_decay"][off] == 0) and torch.all(g["d_beta"][off] == 0)


@pytest.mark.parametrize("T", [1, 9, 70])
def test_kc_fp32_masked_gqa(T):
    """fp32: B2 Hk2 Hv4 Dk32 Dv32 (two value tiles), batch 1 masked from t = 65,
    T over one step, a partial checkpoint segment and several segments."""
    w = wl.custom("kc32", 2, T, 2, 4, 32, 32, seed=601 + T, mask="half_second_batch")
    _parity(w, seed=602 + T)


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (192, 128)])
def test_kc_bf16(Dk, Dv):
    """bf16 at the 9B layer's head sizes and a smaller one."""
    w = wl.custom("kcbf", 1, 77, 2, 4, Dk, Dv, dtype=torch.bfloat16, seed=611 + Dk)
    _parity(w, seed=612 + Dk)


def test_kc_inference_without_saved():
    """keep_saved=False: the forward alone, no checkpoints written."""
    ops = _ops()
    w = wl.custom("kcinf", 2, 30, 1, 2, 32, 16, seed=621)
    x = _kc_inputs(w, 622)
    xd = to_dev(x)
    o, sT, saved = ops.forward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                  xd["state0"], xd["mask"], keep_saved=False)
    assert saved is None
    o_r, s_r = oracle.forward_kc(x["q"], x["k"], x["v"], x["log_decay"], x["beta"],
                                 x["state0"], x["mask"])
    check("o", o, o_r, TOL[w.dtype])
    check("state_T", sT, s_r, TOL[w.dtype])


def test_kc_deterministic_bitwise():
    ops = _ops()
    w = wl.custom("kcdet", 1, 40, 2, 4, 64, 32, dtype=torch.bfloat16, seed=631)
    xd = to_dev(_kc_inputs(w, 632))
    outs = []
    for _ in range(2):
        o, sT, saved = ops.forward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                      xd["state0"], xd["mask"])
        g = ops.backward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["mask"],
                            saved, xd["d_o"], xd["d_state_T"])
        outs.append([o, sT] + [g[n] for n in oracle.GRAD_NAMES_KC])
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_kc_rejects_unsupported_head_sizes():
    ops = _ops()
    w = wl.custom("kcbad", 1, 8, 1, 2, 24, 16, seed=641)  # Dk not a multiple of 16
    xd = to_dev(_kc_inputs(w, 642))
    with pytest.raises(ops.GdnError):
        ops.forward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["state0"])
