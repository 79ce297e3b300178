"""Per-key-channel gates (the mlx-lm page's vectorised gating, g.ndim == 4) through
the C ABI (gdn_forward_kc / gdn_backward_kc) against the fp64 oracle's forward_kc
/ backward_kc, element by element.  bf16 inputs with Dk 64 / 128 / 192 and
Dv 128 take the chunked form (tensor-core scans and products, CUDA-core decayed
Grams); every other shape the recurrent one.  The library's phase timing names
the launches that ran, so each case also checks which form it exercised.

Tolerances as for the other gate forms: per tensor max|x - y| / max|y|, 1e-4
for fp32 inputs and 2e-2 for bf16 inputs.  q, k, v, the state, the cotangents
and the mask come from the shared seeded generator; the per-channel log-decays
from ``make_kc_gates`` (log_decay = -exp(u), u ~ U(ln 0.01, ln 4), channel 0 of
value head 0 at -50: a channel reset every step).
"""

import ctypes

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


class PhaseTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


def _with_phases(fn):
    """fn() under the library's phase timing: (its result, the phase names)."""
    lib = _ops().load_library()
    lib.gdn_timing_end.argtypes = [ctypes.POINTER(PhaseTime), ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_int)]
    assert lib.gdn_timing_begin() == 0
    r = fn()
    torch.cuda.synchronize()
    buf = (PhaseTime * 16)()
    n = ctypes.c_int(0)
    assert lib.gdn_timing_end(buf, 16, ctypes.byref(n)) == 0
    return r, [buf[i].name.decode() for i in range(n.value)]


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
    (o, sT, saved), pf = _with_phases(lambda: ops.forward_kc(
        xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["state0"], xd["mask"]))
    g, pb = _with_phases(lambda: ops.backward_kc(
        xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["mask"], saved, xd["d_o"],
        xd["d_state_T"]))
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
    return pf + pb


@pytest.mark.parametrize("T", [1, 9, 70])
def test_kc_fp32_masked_gqa(T):
    """fp32: B2 Hk2 Hv4 Dk32 Dv32 (two value tiles), batch 1 masked from t = 65,
    T over one step, a partial checkpoint segment and several segments."""
    w = wl.custom("kc32", 2, T, 2, 4, 32, 32, seed=601 + T, mask="half_second_batch")
    _parity(w, seed=602 + T)


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (192, 128)])
def test_kc_bf16(Dk, Dv):
    """bf16 at the 9B layer's head sizes (chunked form) and a smaller one (Dv 64:
    the recurrent form)."""
    w = wl.custom("kcbf", 1, 77, 2, 4, Dk, Dv, dtype=torch.bfloat16, seed=611 + Dk)
    phases = _parity(w, seed=612 + Dk)
    chunked = Dv == 128
    assert ("kc_chunk" in phases) == chunked and ("kc_fwd" in phases) == (not chunked)


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,mask", [
    (1, 64, 1, 1, 64, "none"),                  # one whole chunk
    (1, 150, 2, 4, 192, "none"),                # GQA, three chunks, ragged tail
    (2, 130, 1, 2, 128, "half_second_batch"),   # batch 1 masked from t = 65
    (1, 1000, 1, 2, 192, "none"),               # 16 chunks
    (3, 1, 1, 2, 64, "none"),                   # a single step per sequence
])
def test_kc_chunked_form(B, T, Hk, Hv, Dk, mask):
    """The chunked form: chunk-local products, the per-channel scans and the two
    gradient passes, against the oracle's recurrence."""
    w = wl.custom("kcch", B, T, Hk, Hv, Dk, 128, dtype=torch.bfloat16, seed=650 + T + Dk,
                  mask=mask)
    phases = _parity(w, seed=651 + T + Dk)
    for name in ("kc_chunk", "kc_scan", "kc_bwd_scan", "kc_bwd_prod", "kc_bwd_gate", "kc_bwd_chan"):
        assert name in phases
    assert "kc_fwd" not in phases and "kc_bwd" not in phases


def test_kc_chunked_deterministic_bitwise():
    """The chunked form uses no atomics: two runs agree bit for bit."""
    ops = _ops()
    w = wl.custom("kcdet2", 2, 300, 2, 4, 192, 128, dtype=torch.bfloat16, seed=661,
                  mask="half_second_batch")
    xd = to_dev(_kc_inputs(w, 662))
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


@pytest.mark.slow
def test_kc_qwen35_9b_layer_sampled():
    """B1 T2048 Hk16 Hv64 Dk192 Dv128 bf16 with per-channel gates (value head 0
    carries the channel reset every step), in the bench's launch configuration;
    oracle on key heads 0 and 15 (value heads 0-3 and 60-63)."""
    ops = _ops()
    w = wl.WORKLOADS["qwen35_9b_layer_T2048_bf16"]
    x = _kc_inputs(w, None)
    xd = to_dev(x)
    o, sT, saved = ops.forward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"],
                                  xd["state0"], xd["mask"])
    g = ops.backward_kc(xd["q"], xd["k"], xd["v"], xd["log_decay"], xd["beta"], xd["mask"],
                        saved, xd["d_o"], xd["d_state_T"])
    torch.cuda.synchronize()
    tol = TOL[w.dtype]
    for j in (0, 15):
        h0, h1 = j * w.G, (j + 1) * w.G
        xs = {"q": x["q"][:, :, j:j + 1], "k": x["k"][:, :, j:j + 1], "v": x["v"][:, :, h0:h1],
              "log_decay": x["log_decay"][:, :, h0:h1], "beta": x["beta"][:, :, h0:h1],
              "state0": None if x["state0"] is None else x["state0"][:, h0:h1],
              "mask": x["mask"], "d_o": x["d_o"][:, :, h0:h1],
              "d_state_T": None if x["d_state_T"] is None else x["d_state_T"][:, h0:h1]}
        o_r, s_r = oracle.forward_kc(xs["q"], xs["k"], xs["v"], xs["log_decay"], xs["beta"],
                                     xs["state0"], xs["mask"])
        check("o", o[:, :, h0:h1], o_r, tol)
        check("state_T", sT[:, h0:h1], s_r, tol)
        gr = oracle.backward_kc(xs["q"], xs["k"], xs["v"], xs["log_decay"], xs["beta"],
                                xs["state0"], xs["mask"], xs["d_o"], xs["d_state_T"])
        sl = {"dq": g["dq"][:, :, j:j + 1], "dk": g["dk"][:, :, j:j + 1]}
        for n in oracle.GRAD_NAMES_KC:
            got = sl.get(n)
            if got is None:
                got = g[n][:, h0:h1] if n == "dstate0" else g[n][:, :, h0:h1]
            check(n, got, gr[n], tol)


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
