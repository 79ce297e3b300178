"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerances (per tensor, max|x - y| / max|y|): 1e-4 for fp32 inputs, 2e-2 for
bf16 inputs with fp32 accumulation.  Small cases span several 64-step chunks
and a ragged tail; the full-size workloads are compared on whole tensors
where the oracle is fast enough and on a subset of independent (batch,
key-head group) units otherwise.
"""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from parity_util import (TOL, check, gpu_backward, gpu_forward, np64, oracle_backward,
                         oracle_forward, to_dev)

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "da", "db", "dA_log", "ddt_bias", "dstate0")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _full_parity(w, backward=True):
    x = wl.make_inputs(w)
    xd = to_dev(x)
    tol = TOL[w.dtype]
    o, sT, saved = gpu_forward(xd)
    torch.cuda.synchronize()
    o_r, s_r = oracle_forward(x)
    errs = {}
    check("o", o, o_r, tol, errs)
    check("state_T", sT, s_r, tol, errs)
    if backward:
        g = gpu_backward(xd, saved)
        torch.cuda.synchronize()
        gr = oracle_backward(x)
        for n in GRADS:
            check(n, g[n], gr[n], tol, errs)
    return errs


def test_outputs_and_workspaces_start_poisoned():
    """The fixture in conftest.py is active: memory the binding allocates for
    outputs, saved buffers and workspaces reads as NaN until written."""
    from gated_delta_rule_06_gb300 import ops

    assert torch.isnan(torch.empty(64, device="cuda")).all()
    assert torch.isnan(torch.empty(64, dtype=torch.bfloat16, device="cuda")).all()
    assert bool((ops._buf(256, "cuda") == 255).all())


def test_toy_workload_fp32():
    """Toy gradient-check shape (B1 T8 Hk2 Hv4 Dk16 Dv8, fp32): forward and all 8 grads."""
    _full_parity(wl.WORKLOADS["toy_fp32"])


def test_chunk_mask_workload_fp32():
    """B2 T129 Hk4 Hv8 D64 fp32, batch 1 masked from t = 65, head 0 on the clamp."""
    _full_parity(wl.WORKLOADS["chunk_mask_fp32"])


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 200])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_lengths(T, dtype):
    """Edge lengths around the 64-step chunk (mlx-lm page, "Covered corner cases")."""
    w = wl.custom("len", 2, T, 2, 4, 32, 16, dtype=dtype, seed=100 + T,
                  mask="half_second_batch" if T > 65 else "none", clamp_head=True)
    _full_parity(w)


@pytest.mark.parametrize("Dk,Dv,Hk,Hv", [(8, 8, 1, 1), (16, 40, 1, 3), (48, 24, 2, 2),
                                         (192, 128, 1, 4), (256, 256, 1, 1), (128, 64, 4, 8)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_head_dims(Dk, Dv, Hk, Hv, dtype):
    """Key / value widths from the minimum to the maximum supported, Dk != Dv, GQA."""
    w = wl.custom("dims", 1, 100, Hk, Hv, Dk, Dv, dtype=dtype, seed=Dk * 7 + Dv)
    _full_parity(w)


@pytest.mark.parametrize("T", [1, 64, 65, 130, 200])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 128), (192, 128), (96, 192)])
def test_tensor_core_paths_bf16(T, Dk, Dv):
    """bf16 shapes that take the tcgen05 kernels (Dk % 32 == 0, Dv % 64 == 0):
    ragged tails, half masking, the clamp head and GQA."""
    w = wl.custom("tc", 2, T, 2, 4, Dk, Dv, dtype=torch.bfloat16, seed=7 * T + Dk + Dv,
                  mask="half_second_batch" if T > 65 else "none", clamp_head=True)
    _full_parity(w)


def test_zero_initial_state_and_no_state_cotangent():
    w = wl.custom("zs", 2, 70, 2, 4, 32, 32, dtype=torch.float32, seed=5, state_sigma=0.0,
                  d_state=False)
    _full_parity(w)


def test_all_true_mask_equals_no_mask():
    w = wl.custom("m1", 2, 70, 1, 2, 16, 16, seed=3)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o1, s1, sv1 = gpu_forward(xd)
    g1 = gpu_backward(xd, sv1)
    xd2 = dict(xd, mask=torch.ones((2, 70), dtype=torch.uint8, device="cuda"))
    o2, s2, sv2 = gpu_forward(xd2)
    g2 = gpu_backward(xd2, sv2)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


def test_deterministic_bitwise():
    """Two runs give byte-identical outputs and gradients (no atomics anywhere)."""
    w = wl.custom("det", 2, 150, 2, 4, 64, 64, dtype=torch.bfloat16, seed=9,
                  mask="half_second_batch")
    xd = to_dev(wl.make_inputs(w))
    outs = []
    for _ in range(2):
        o, sT, saved = gpu_forward(xd)
        g = gpu_backward(xd, saved)
        outs.append([o, sT] + [g[n] for n in GRADS])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_decode_kernel_matches_oracle_and_chunked():
    """T = 1 without a saved buffer runs the fused single-step kernel."""
    w = wl.custom("dec", 16, 1, 4, 8, 128, 128, dtype=torch.bfloat16, seed=17, state_sigma=0.02)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, _ = gpu_forward(xd, keep_saved=False)
    o_r, s_r = oracle_forward(x)
    check("o", o, o_r, TOL[torch.bfloat16])
    check("state_T", sT, s_r, 1e-4)  # fp32 state update, bf16 only in q/k/v
    o2, s2, _ = gpu_forward(xd, keep_saved=True)
    check("o_vs_chunked", o, np64(o2), TOL[torch.bfloat16])
    check("state_vs_chunked", sT, np64(s2), TOL[torch.bfloat16])


def test_decode_in_place_and_mask():
    from gated_delta_rule_06_gb300 import ops

    w = wl.custom("dec2", 8, 1, 2, 4, 64, 32, dtype=torch.float32, seed=23, state_sigma=0.1)
    x = wl.make_inputs(w)
    x["mask"] = torch.tensor([[1], [0], [1], [1], [0], [1], [1], [1]], dtype=torch.uint8)
    xd = to_dev(x)
    o_r, s_r = oracle_forward(x)
    st = xd["state0"].clone()
    o, s = ops.decode(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"], xd["dt_bias"],
                      st, xd["mask"], state_out=st)
    assert s.data_ptr() == st.data_ptr()
    check("o", o, o_r, 1e-4)
    check("state_T", st, s_r, 1e-4)


def test_autograd_function():
    from gated_delta_rule_06_gb300 import ops

    w = wl.custom("ag", 1, 90, 2, 4, 32, 16, dtype=torch.float32, seed=31)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    leaves = {n: xd[n].clone().requires_grad_(True)
              for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0")}
    o, sT = ops.gated_delta_rule(*[leaves[n] for n in ("q", "k", "v", "a", "b", "A_log",
                                                        "dt_bias", "state0")], None)
    loss = (o * xd["d_o"]).sum() + (sT * xd["d_state_T"]).sum()
    loss.backward()
    gr = oracle_backward(x)
    names = dict(q="dq", k="dk", v="dv", a="da", b="db", A_log="dA_log", dt_bias="ddt_bias",
                 state0="dstate0")
    for n, gname in names.items():
        check(gname, leaves[n].grad, gr[gname], 1e-4)


# ---- full-size workloads -------------------------------------------------------

def _subset(x, b_sel, j0, j1, G):
    """Inputs restricted to batches b_sel and key heads [j0, j1) (value heads
    [j0*G, j1*G)); every such unit is independent of the others."""
    h0, h1 = j0 * G, j1 * G
    y = {}
    for n, t in x.items():
        if t is None:
            y[n] = None
        elif n in ("q", "k"):
            y[n] = t[b_sel][:, :, j0:j1]
        elif n in ("v", "d_o"):
            y[n] = t[b_sel][:, :, h0:h1]
        elif n in ("a", "b"):
            y[n] = t[b_sel][:, :, h0:h1]
        elif n in ("A_log", "dt_bias"):
            y[n] = t[h0:h1]
        elif n in ("state0", "d_state_T"):
            y[n] = t[b_sel][:, h0:h1]
        elif n == "mask":
            y[n] = t[b_sel]
    return y


def _sampled_parity(w, b_sel, j0, j1, backward=True):
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, saved = gpu_forward(xd)
    g = gpu_backward(xd, saved) if backward else None
    torch.cuda.synchronize()
    xs = _subset(x, b_sel, j0, j1, w.G)
    h0, h1 = j0 * w.G, j1 * w.G
    tol = TOL[w.dtype]
    o_r, s_r = oracle_forward(xs)
    check("o", o[b_sel][:, :, h0:h1], o_r, tol)
    check("state_T", sT[b_sel][:, h0:h1], s_r, tol)
    if backward:
        gr = oracle_backward(xs)
        sl = {"dq": lambda t: t[b_sel][:, :, j0:j1], "dk": lambda t: t[b_sel][:, :, j0:j1],
              "dv": lambda t: t[b_sel][:, :, h0:h1], "da": lambda t: t[b_sel][:, :, h0:h1],
              "db": lambda t: t[b_sel][:, :, h0:h1], "dA_log": lambda t: t[h0:h1],
              "ddt_bias": lambda t: t[h0:h1], "dstate0": lambda t: t[b_sel][:, h0:h1]}
        for n in GRADS:
            check(n, sl[n](g[n]), gr[n], tol)


@pytest.mark.slow
def test_qwen35_9b_layer_T2048_sampled():
    """B1 T2048 Hk16 Hv64 Dk192 Dv128 bf16, in the bench's launch configuration;
    oracle on key heads 0, 7 and 15 (value heads 0-3, 28-31, 60-63)."""
    w = wl.WORKLOADS["qwen35_9b_layer_T2048_bf16"]
    for j in (0, 7, 15):
        _sampled_parity(w, [0], j, j + 1)


@pytest.mark.slow
def test_gqa_train_B4_T4096_sampled():
    """B4 T4096 Hk16 Hv32 D128 bf16; oracle on all batches of key heads 0 and 9."""
    w = wl.WORKLOADS["gqa_train_B4_T4096_bf16"]
    for j in (0, 9):
        _sampled_parity(w, [0, 1, 2, 3], j, j + 1)


@pytest.mark.slow
def test_long_B1_T65536_sampled():
    """B1 T65536 Hk4 Hv8 D128 bf16 (few heads over a long sequence), through
    gdn_forward / gdn_backward with the library's automatic segment counts,
    which split both scans on this shape (runs of dozens of chunks); oracle
    on key head 1 (value heads 2 and 3), every output and gradient."""
    from gated_delta_rule_06_gb300 import ops

    w = wl.WORKLOADS["long_B1_T65536_Hv8_bf16"]
    shape = ops.GdnShape(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, 1, 0)
    assert ops.segments_auto(shape) > 1 and ops.segments_auto(shape, backward=True) > 1
    _sampled_parity(w, [0], 1, 2)


def _fwd_bwd_outputs(xd):
    o, sT, saved = gpu_forward(xd)
    g = gpu_backward(xd, saved)
    torch.cuda.synchronize()
    return [o, sT] + [g[n] for n in GRADS]


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen35_9b_layer_T2048_bf16", "gqa_train_B4_T4096_bf16"])
def test_deterministic_bitwise_full_size(name):
    """At the full workloads every SM takes gradient items from the shared
    counter (2048 items at the 9B layer, 2048 at B4 T4096), so which CTA runs
    which item changes from run to run; the forward and all eight gradients
    must still agree bit for bit."""
    xd = to_dev(wl.make_inputs(wl.WORKLOADS[name]))
    first = _fwd_bwd_outputs(xd)
    second = _fwd_bwd_outputs(xd)
    for n, a, b in zip(("o", "state_T") + GRADS, first, second):
        assert torch.equal(a, b), n


@pytest.mark.slow
def test_decode_B256_full():
    """Decode step B256 Hv32 D128, bf16 q/k/v, fp32 state: every element."""
    w = wl.WORKLOADS["decode_B256_bf16"]
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, _ = gpu_forward(xd, keep_saved=False)
    torch.cuda.synchronize()
    o_r, s_r = oracle_forward(x)
    check("o", o, o_r, TOL[torch.bfloat16])
    check("state_T", sT, s_r, 1e-4)
