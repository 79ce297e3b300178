"""Rank-r compressed chunk states on the GPU (gdn_forward_compressed /
gdn_backward_compressed) against the compressed-state oracle
(oracle/compressed.py): mlx-lm page, "Post-initial-submission extensions",
Extension 1, the state truncated to rank r by power iteration at every chunk
boundary, the backward passing the state cotangent straight through the
boundaries.

Tolerance: bf16 inputs, per tensor max|x - y| / max|y| <= 2e-2, and the
per-slice bars of parity_util.
"""

import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from oracle import compressed as oc
from parity_util import TOL, check, to_dev

pytestmark = pytest.mark.gpu

GRADS = oracle.GRAD_NAMES
PRIMAL_ORDER = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build

    build.build()


def _ops():
    from gated_delta_rule_06_gb300 import ops

    return ops


def _gpu(xd, omega, rank, iters):
    ops = _ops()
    o, sT, saved = ops.forward_compressed(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                                          xd["dt_bias"], xd["state0"], xd["mask"], omega=omega,
                                          rank=rank, iters=iters)
    g = ops.backward_compressed(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                                xd["dt_bias"], xd["mask"], saved, xd["d_o"], xd["d_state_T"],
                                rank=rank)
    torch.cuda.synchronize()
    return o, sT, saved, g


def _oracle(x, omega, iters):
    args = [x[n] for n in PRIMAL_ORDER]
    o, sT, _, _, _ = oc.forward_compressed(*args, omega, iters)
    g = oc.backward_compressed(*args, x["d_o"], x["d_state_T"], omega, iters)
    return o, sT, g


def _parity(w, rank, iters=3, seed=0):
    x = wl.make_inputs(w)
    xd = to_dev(x)
    om = wl.make_omega(w.Dv, rank, seed)
    o, sT, saved, g = _gpu(xd, om.cuda(), rank, iters)
    o_r, s_r, g_r = _oracle(x, om, iters)
    tol = TOL[w.dtype]
    check("o", o, o_r, tol)
    check("state_T", sT, s_r, tol)
    for n in GRADS:
        check(n, g[n], g_r[n], tol)
    return saved


@pytest.mark.parametrize("Dk,Dv,rank", [(64, 128, 4), (128, 128, 16), (192, 128, 16),
                                        (192, 128, 1), (128, 128, 2)])
def test_compressed_matches_oracle(Dk, Dv, rank):
    """T = 200 (four chunks, three boundaries, a ragged tail), GQA, batch 1 masked
    from t = 65, the clamp head, a nonzero initial state."""
    w = wl.custom("cmp", 2, 200, 2, 4, Dk, Dv, dtype=torch.bfloat16, seed=900 + Dk + Dv + rank,
                  mask="half_second_batch", clamp_head=True)
    _parity(w, rank)


@pytest.mark.parametrize("iters", [0, 1, 5])
def test_iteration_counts(iters):
    w = wl.custom("cmpit", 1, 300, 2, 4, 128, 128, dtype=torch.bfloat16, seed=950 + iters)
    _parity(w, 8, iters=iters, seed=iters)


def test_single_chunk_equals_plain_path():
    """T <= 64: no boundary, so the compressed forward and backward run the same
    kernels on the same values as gdn_forward / gdn_backward: bit for bit."""
    ops = _ops()
    w = wl.custom("cmp1", 2, 64, 2, 4, 128, 128, dtype=torch.bfloat16, seed=961,
                  mask="half_second_batch")
    xd = to_dev(wl.make_inputs(w))
    om = wl.make_omega(128, 16).cuda()
    o, sT, _, g = _gpu(xd, om, 16, 3)
    o2, s2, sv2 = ops.forward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"],
                              xd["dt_bias"], xd["state0"], xd["mask"])
    g2 = ops.backward(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], xd["A_log"], xd["dt_bias"],
                      xd["mask"], sv2, xd["d_o"], xd["d_state_T"])
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(sT, s2)
    for n in GRADS:
        assert torch.equal(g[n], g2[n]), n


def test_deterministic_and_smaller_saved_buffer():
    ops = _ops()
    w = wl.custom("cmpd", 1, 64 * 8 + 9, 2, 4, 192, 128, dtype=torch.bfloat16, seed=971)
    xd = to_dev(wl.make_inputs(w))
    om = wl.make_omega(128, 16).cuda()
    a = _gpu(xd, om, 16, 3)
    b = _gpu(xd, om, 16, 3)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    for n in GRADS:
        assert torch.equal(a[3][n], b[3][n]), n
    shape = ops.make_shape(xd["q"], xd["v"], False)
    saved_c, _, _ = ops.compressed_sizes(shape, 16)
    assert saved_c < ops.saved_bytes(shape)


@pytest.mark.slow
def test_qwen35_9b_layer_rank16_sampled():
    """B1 T2048 Hk16 Hv64 Dk192 Dv128 at rank 16, three iterations; oracle on key
    heads 0 and 15 (value heads 0-3 and 60-63), every output and gradient."""
    from test_gpu_parity import _subset

    w = wl.WORKLOADS["qwen35_9b_layer_T2048_bf16"]
    x = wl.make_inputs(w)
    xd = to_dev(x)
    om = wl.make_omega(w.Dv, 16)
    o, sT, _, g = _gpu(xd, om.cuda(), 16, 3)
    tol = TOL[w.dtype]
    for j in (0, 15):
        xs = _subset(x, [0], j, j + 1, w.G)
        h0, h1 = j * w.G, (j + 1) * w.G
        o_r, s_r, g_r = _oracle(xs, om, 3)
        check("o", o[:, :, h0:h1], o_r, tol)
        check("state_T", sT[:, h0:h1], s_r, tol)
        sl = {"dq": lambda t: t[:, :, j:j + 1], "dk": lambda t: t[:, :, j:j + 1],
              "dv": lambda t: t[:, :, h0:h1], "da": lambda t: t[:, :, h0:h1],
              "db": lambda t: t[:, :, h0:h1], "dA_log": lambda t: t[h0:h1],
              "ddt_bias": lambda t: t[h0:h1], "dstate0": lambda t: t[:, h0:h1]}
        for n in GRADS:
            check(n, sl[n](g[n]), g_r[n], tol)
