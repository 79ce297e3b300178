"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself: every check is a central
difference, a closed form of a special case, an identity of the delta rule,
or an equivalence between two differently shaped inputs.  Each is chosen so
that a plausible slip in the oracle (a sign, the order of decay and update,
which state the output reads, the GQA head map, the q scale, the clamp) fails
at least one test.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BIG_NEG = -800.0  # exp(-800) underflows to 0 in fp64: A_log = -800 gives g = 1 exactly
BIG_POS = 800.0   # sigmoid(800) == 1 and sigmoid(-800) == 0 in fp64


def _np(x):
    return None if x is None else x.detach().to(torch.float64).numpy().copy()


def _inputs(w, seed=None):
    x = wl.make_inputs(w, seed)
    return {k: _np(v) if k != "mask" else (None if v is None else v.numpy().copy())
            for k, v in x.items()}


PRIMALS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0")
GRAD_OF = dict(q="dq", k="dk", v="dv", a="da", b="db", A_log="dA_log",
               dt_bias="ddt_bias", state0="dstate0")


def _loss(x, d_o, d_sT):
    o, sT = oracle.forward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                           x["dt_bias"], x["state0"], x["mask"])
    val = float((o * d_o).sum())
    if d_sT is not None:
        val += float((sT * d_sT).sum())
    return val


def _fd_check(x, max_elems=None, h=2.0 ** -17, rng=None):
    """Central differences of L = <o, d_o> + <S_T, d_S_T> against the VJP."""
    if x["state0"] is None:
        x = dict(x, state0=np.zeros((x["q"].shape[0], x["v"].shape[2], x["q"].shape[3],
                                     x["v"].shape[3])))
    g = oracle.backward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                        x["state0"], x["mask"], x["d_o"], x["d_state_T"])
    errs = {}
    for name in PRIMALS:
        arr = x[name]
        flat = arr.reshape(-1)
        idx = np.arange(flat.size)
        if max_elems is not None and flat.size > max_elems:
            idx = (rng or np.random.default_rng(0)).choice(flat.size, max_elems, replace=False)
        fd = np.zeros(len(idx))
        for n, i in enumerate(idx):
            old = flat[i]
            flat[i] = old + h
            lp = _loss(x, x["d_o"], x["d_state_T"])
            flat[i] = old - h
            lm = _loss(x, x["d_o"], x["d_state_T"])
            flat[i] = old
            fd[n] = (lp - lm) / (2 * h)
        an = g[GRAD_OF[name]].reshape(-1)[idx]
        scale = max(np.abs(fd).max(), 1e-30)
        errs[GRAD_OF[name]] = (np.abs(an - fd).max(), float(scale))
    return errs, g


def _assert_fd(errs, rel=1e-7):
    for name, (err, scale) in errs.items():
        assert err <= rel * max(scale, 1.0), (name, err, scale)


# -- central differences -------------------------------------------------------

def test_fd_toy_workload_all_grads():
    """mlx-lm page, "Numerical correctness": FD check of all 8 grads on the toy shape."""
    x = _inputs(wl.WORKLOADS["toy_fp32"])
    errs, _ = _fd_check(x)
    _assert_fd(errs)
    # The page's fp32 FD maxima are upper bounds; an fp64 FD must sit far below.
    with open(os.path.join(GOLDEN, "fd_table_toy_fp32.json")) as f:
        table = json.load(f)["max_abs_diff"]
    for name, (err, _) in errs.items():
        assert err < table[name] * 1e-3, (name, err, table[name])


@pytest.mark.parametrize("T", [1, 64, 65])
def test_fd_edge_lengths(T):
    """mlx-lm page, "Covered corner cases": T = 1, CHUNK_SIZE, CHUNK_SIZE + 1."""
    w = wl.custom("edge", 1, T, 1, 2, 8, 4, seed=7 + T)
    errs, _ = _fd_check(_inputs(w), max_elems=24, rng=np.random.default_rng(T))
    _assert_fd(errs)


def test_fd_masked_gqa_clamp():
    """FD through the masked path (mlx-lm page, "Numerical correctness" tests),
    with GQA (G = 3) and one head on the softplus clamp (A_log = 5, a = 15)."""
    w = wl.custom("mask", 2, 70, 1, 3, 8, 4, seed=11, mask="half_second_batch",
                  clamp_head=True)
    x = _inputs(w)
    errs, g = _fd_check(x, max_elems=30, rng=np.random.default_rng(3))
    _assert_fd(errs)
    for v in g.values():
        assert np.isfinite(v).all()


# -- closed forms and identities ----------------------------------------------

def _unit_rows(n, d, scale=1.0):
    """n distinct standard basis vectors of R^d (times scale)."""
    e = np.zeros((n, d))
    e[np.arange(n), np.arange(n)] = scale
    return e


def test_beta_zero_is_pure_decay_half():
    """beta = 0 removes the write; with A_log = 0 and a + dt_bias = 0 the gate is
    exp(-softplus(0)) = exp(-ln 2) = 1/2 per step, so S_T = 2^-T S_0 and
    o_t = 2^-(t+1) S_0^T q_hat_t."""
    rng = np.random.default_rng(0)
    B, T, Hk, Hv, Dk, Dv = 1, 5, 1, 1, 4, 3
    S0 = rng.standard_normal((B, Hv, Dk, Dv))
    q = np.zeros((B, T, Hk, Dk))
    q[0, :, 0, 1] = 3.0  # q_hat = e_1 * 3 / sqrt(9 + 1e-6) / sqrt(Dk)
    k = rng.standard_normal((B, T, Hk, Dk))
    v = rng.standard_normal((B, T, Hv, Dv))
    a = np.zeros((B, T, Hv))
    b = np.full((B, T, Hv), -BIG_POS)
    o, sT = oracle.forward(q, k, v, a, b, np.zeros(Hv), np.zeros(Hv), S0, None)
    np.testing.assert_allclose(sT, S0 * 2.0 ** -T, rtol=1e-14, atol=0)
    qs = 3.0 / math.sqrt(9.0 + 1e-6) / math.sqrt(Dk)
    for t in range(T):
        np.testing.assert_allclose(o[0, t, 0], 2.0 ** -(t + 1) * qs * S0[0, 0, 1], rtol=1e-13)


def test_gate_closed_forms():
    """g = exp(-exp(A_log) softplus(a + dt_bias)):
    A_log = ln 2, x = 0      -> g = exp(-2 ln 2) = 1/4;
    A_log = 0,    x = ln(e-1) -> softplus = 1 -> g = 1/e;
    split of x between a and dt_bias does not matter."""
    rng = np.random.default_rng(1)
    S0 = rng.standard_normal((1, 3, 2, 2))
    q = rng.standard_normal((1, 1, 1, 2))
    k = rng.standard_normal((1, 1, 1, 2))
    v = rng.standard_normal((1, 1, 3, 2))
    b = np.full((1, 1, 3), -BIG_POS)
    A_log = np.array([math.log(2.0), 0.0, 0.0])
    xe = math.log(math.e - 1.0)
    a = np.array([[[0.0, xe, 0.25]]])
    dt = np.array([0.0, 0.0, xe - 0.25])
    _, sT = oracle.forward(q, k, v, a, b, A_log, dt, S0, None)
    np.testing.assert_allclose(sT[0, 0], 0.25 * S0[0, 0], rtol=1e-14)
    np.testing.assert_allclose(sT[0, 1], S0[0, 1] / math.e, rtol=1e-13)
    np.testing.assert_allclose(sT[0, 2], S0[0, 2] / math.e, rtol=1e-13)


def test_softplus_clamp_saturates():
    """The clamped softplus stops growing at x = 20 (mlx-lm page, "Covered corner
    cases"); at x = 20 its value is 20 + log(1 + e^-20) (softplus(x) = x + softplus(-x))."""
    rng = np.random.default_rng(2)
    S0 = rng.standard_normal((1, 1, 2, 2))
    q, k = rng.standard_normal((2, 1, 1, 1, 2))
    v = rng.standard_normal((1, 1, 1, 2))
    b = np.full((1, 1, 1), -BIG_POS)
    A_log = np.array([-3.0])
    outs = []
    for x in (20.0, 25.0, 60.0):
        _, sT = oracle.forward(q, k, v, np.full((1, 1, 1), x), b, A_log, np.zeros(1), S0, None)
        outs.append(sT)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    g = math.exp(-math.exp(-3.0) * (20.0 + math.log1p(math.exp(-20.0))))
    np.testing.assert_allclose(outs[0], g * S0, rtol=1e-14)


def test_beta_one_retrieves_latest_value():
    """Delta rule with beta = 1: after a step, S_t^T k_hat_t = v_t up to the eps of
    the L2 norm, whatever the gate and the old state.  With q = k the output is
    o_t = S_t^T k_hat_t / sqrt(Dk).  This pins the sign of delta, decay-before-
    update, that o reads the updated state, and the 1/sqrt(Dk) scale."""
    rng = np.random.default_rng(3)
    B, T, Hk, Hv, Dk, Dv = 1, 6, 1, 1, 8, 5
    k = rng.standard_normal((B, T, Hk, Dk)) * 2.0
    q = k.copy()
    v = rng.standard_normal((B, T, Hv, Dv))
    a = rng.standard_normal((B, T, Hv))
    b = np.full((B, T, Hv), BIG_POS)
    S0 = rng.standard_normal((B, Hv, Dk, Dv))
    o, _ = oracle.forward(q, k, v, a, b, np.array([0.3]), np.array([0.1]), S0, None)
    np.testing.assert_allclose(o[0, :, 0] * math.sqrt(Dk), v[0, :, 0], rtol=0, atol=1e-6)


def test_orthonormal_keys_exact_memory():
    """g = 1, beta = 1, S_0 = 0 and orthogonal keys e_t: nothing interferes, so
    S_T = sum_t k_hat_t v_t^T, i.e. row t of S_T is v_t / sqrt(1 + eps)."""
    rng = np.random.default_rng(4)
    B, T, Hk, Hv, Dk, Dv = 1, 5, 1, 1, 7, 3
    k = _unit_rows(T, Dk)[None, :, None, :]
    q = rng.standard_normal((B, T, Hk, Dk))
    v = rng.standard_normal((B, T, Hv, Dv))
    a = rng.standard_normal((B, T, Hv))
    b = np.full((B, T, Hv), BIG_POS)
    _, sT = oracle.forward(q, k, v, a, b, np.array([BIG_NEG]), np.zeros(1), None, None)
    expect = np.zeros((Dk, Dv))
    expect[:T] = v[0, :, 0] / math.sqrt(1.0 + 1e-6)
    np.testing.assert_allclose(sT[0, 0], expect, rtol=1e-14, atol=1e-15)


def test_gqa_equals_repeat_interleave():
    """torch-to-nnef page, op contract: value head h reads q/k head h // G; the
    same run on q/k repeat-interleaved to Hv heads must agree, and dq/dk of the
    grouped run are the sums over each group of the repeated run's dq/dk."""
    w = wl.custom("gqa", 2, 9, 2, 6, 5, 4, seed=21)
    x = _inputs(w)
    G = 3
    xr = dict(x)
    xr["q"] = np.repeat(x["q"], G, axis=2)
    xr["k"] = np.repeat(x["k"], G, axis=2)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")
    o1, s1 = oracle.forward(*[x[n] for n in args])
    o2, s2 = oracle.forward(*[xr[n] for n in args])
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(s1, s2, rtol=1e-13, atol=1e-14)
    g1 = oracle.backward(*[x[n] for n in args], x["d_o"], x["d_state_T"])
    g2 = oracle.backward(*[xr[n] for n in args], x["d_o"], x["d_state_T"])
    for n in ("dq", "dk"):
        summed = g2[n].reshape(2, 9, 2, G, 5).sum(axis=3)
        np.testing.assert_allclose(g1[n], summed, rtol=1e-11, atol=1e-13)
    for n in ("dv", "da", "db", "dA_log", "ddt_bias", "dstate0"):
        np.testing.assert_allclose(g1[n], g2[n], rtol=1e-11, atol=1e-13)


def test_all_true_mask_equals_unmasked():
    """mlx-lm page, "Covered corner cases": an all-True mask equals no mask."""
    w = wl.custom("m", 2, 20, 1, 2, 6, 5, seed=31)
    x = _inputs(w)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0")
    ones = np.ones((2, 20), np.uint8)
    o1, s1 = oracle.forward(*[x[n] for n in args], None)
    o2, s2 = oracle.forward(*[x[n] for n in args], ones)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
    g1 = oracle.backward(*[x[n] for n in args], None, x["d_o"], x["d_state_T"])
    g2 = oracle.backward(*[x[n] for n in args], ones, x["d_o"], x["d_state_T"])
    for n in g1:
        np.testing.assert_array_equal(g1[n], g2[n])


def test_half_mask_final_state_is_prefix_state():
    """mlx-lm page, "Covered corner cases": under half-masking the final state is the
    state after the unmasked prefix.  The outputs of masked steps read that state
    (the reading taken for them): they equal the outputs of identity steps
    (beta = 0, g = 1) in place of the masked ones."""
    w = wl.custom("hm", 2, 129, 1, 2, 6, 5, seed=41, mask="half_second_batch")
    x = _inputs(w)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0")
    o, sT = oracle.forward(*[x[n] for n in args], x["mask"])
    xp = {n: x[n][1:2, :65] if n in ("q", "k", "v", "a", "b") else x[n] for n in args}
    xp["state0"] = x["state0"][1:2]
    _, sP = oracle.forward(*[xp[n] for n in args], None)
    np.testing.assert_allclose(sT[1], sP[0], rtol=1e-13, atol=1e-14)
    # identity steps in place of the masked ones (batch 1 only)
    xi = {n: x[n].copy() for n in args}
    xi["b"][1, 65:] = -BIG_POS
    xi["A_log"] = x["A_log"].copy()
    # g = 1 on those steps: a + dt_bias -> -inf through a very negative a
    xi["a"][1, 65:] = -1e6
    o2, s2 = oracle.forward(*[xi[n] for n in args], None)
    np.testing.assert_allclose(o[1], o2[1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sT[1], s2[1], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(o[0], o2[0])


def test_extreme_gates_stay_finite():
    """mlx-lm page, "Covered corner cases": A_log = 5 with a = 15 gives no NaN/Inf."""
    w = wl.WORKLOADS["chunk_mask_fp32"]
    x = _inputs(wl.custom("ex", 2, 129, 2, 4, 16, 8, seed=51, mask="half_second_batch",
                          clamp_head=True))
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")
    o, sT = oracle.forward(*[x[n] for n in args])
    assert np.isfinite(o).all() and np.isfinite(sT).all()
    g = oracle.backward(*[x[n] for n in args], x["d_o"], x["d_state_T"])
    for n, val in g.items():
        assert np.isfinite(val).all(), n
    assert w.clamp_head


@pytest.mark.parametrize("T,C", [(1, 64), (63, 64), (64, 64), (65, 64), (129, 64),
                                 (200, 16), (37, 7)])
def test_chunked_equals_sequential(T, C):
    """torch-to-nnef page: the chunked rule is the same recurrence with a different
    blocking, equal up to floating-point reordering."""
    w = wl.custom("ch", 2, T, 2, 4, 12, 6, seed=60 + T, mask="half_second_batch",
                  clamp_head=True)
    x = _inputs(w)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")
    o1, s1 = oracle.forward(*[x[n] for n in args])
    o2, s2 = oracle.forward_chunked(*[x[n] for n in args], chunk=C)
    assert np.abs(o1 - o2).max() <= 1e-12 * max(np.abs(o1).max(), 1.0)
    assert np.abs(s1 - s2).max() <= 1e-12 * max(np.abs(s1).max(), 1.0)


def test_chunked_catches_planted_slip():
    """Guard for the test above: a changed input (one value entry) must be visible."""
    w = wl.custom("ch", 1, 65, 1, 1, 8, 4, seed=99)
    x = _inputs(w)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")
    o1, _ = oracle.forward(*[x[n] for n in args])
    y = dict(x)
    y["v"] = x["v"].copy()
    y["v"][0, 64, 0] += 1e-3
    o2, _ = oracle.forward_chunked(*[y[n] for n in args], chunk=64)
    assert np.abs(o1 - o2).max() > 1e-8


@pytest.mark.parametrize("T,L", [(1, 1), (5, 1), (37, 37), (37, 100), (65, 64), (129, 16),
                                 (200, 7)])
def test_monoid_equals_sequential(T, L):
    """mlx-lm page, "Post-initial-submission extensions", Extension 5: the recurrence
    as an associative monoid of affine state maps, evaluated by a tree prefix over
    runs of L steps (run counts 1, 5 padded to 8, 3, 9, 29), equals the sequential
    recurrence up to rounding; masked batch, GQA, the clamp head, a nonzero
    initial state.  Composing the non-commuting maps in the wrong order, or
    dropping a run's offset, moves the result by far more than the bound."""
    w = wl.custom("mo", 2, T, 2, 4, 12, 6, seed=70 + T, mask="half_second_batch",
                  clamp_head=True)
    x = _inputs(w)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")
    assert np.abs(x["state0"]).max() > 0
    o1, s1 = oracle.forward(*[x[n] for n in args])
    o2, s2 = oracle.forward_monoid(*[x[n] for n in args], seg_len=L)
    assert np.abs(o1 - o2).max() <= 1e-12 * max(np.abs(o1).max(), 1.0)
    assert np.abs(s1 - s2).max() <= 1e-12 * max(np.abs(s1).max(), 1.0)


def test_monoid_run_maps_do_not_commute():
    """Guard for the test above: two runs of steps give different results in the
    two orders, so an order slip in the prefix would be seen.  Swapping the two
    halves of the sequence (the same run maps, composed the other way round)
    changes the final state."""
    w = wl.custom("mo", 1, 16, 1, 1, 8, 4, seed=98)
    x = _inputs(w)
    args = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")
    _, s1 = oracle.forward_monoid(*[x[n] for n in args], seg_len=8)
    y = dict(x)
    for n in ("q", "k", "v", "a", "b"):
        y[n] = np.concatenate([x[n][:, 8:], x[n][:, :8]], axis=1)
    _, s2 = oracle.forward_monoid(*[y[n] for n in args], seg_len=8)
    assert np.abs(s1 - s2).max() > 1e-3 * np.abs(s1).max()


# -- the log_decay / beta input form (torch-to-nnef page, op contract) ----------

def _lb_inputs(B, T, Hk, Hv, Dk, Dv, seed, masked=False):
    r = np.random.default_rng(seed)
    x = dict(q=r.standard_normal((B, T, Hk, Dk)), k=r.standard_normal((B, T, Hk, Dk)),
             v=r.standard_normal((B, T, Hv, Dv)),
             log_decay=-r.uniform(0.0, 2.0, (B, T, Hv)), beta=r.uniform(0.0, 1.0, (B, T, Hv)),
             state0=0.1 * r.standard_normal((B, Hv, Dk, Dv)), mask=None,
             d_o=r.standard_normal((B, T, Hv, Dv)), d_state_T=r.standard_normal((B, Hv, Dk, Dv)))
    if masked:
        m = np.ones((B, T), dtype=np.uint8)
        m[-1, T // 2:] = 0
        x["mask"] = m
    return x


def _lb_loss(x):
    o, sT = oracle.forward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                              x["mask"])
    return float((o * x["d_o"]).sum() + (sT * x["d_state_T"]).sum())


@pytest.mark.parametrize("masked", [False, True])
def test_lb_fd_all_grads(masked):
    """Central differences of L = <o, dO> + <S_T, dS_T> through the log_decay /
    beta form (GQA G = 2, T = 67 over two 64-step segments, optional mask)."""
    x = _lb_inputs(2, 67, 1, 2, 6, 4, seed=21 + masked, masked=masked)
    g = oracle.backward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                           x["mask"], x["d_o"], x["d_state_T"])
    h = 2.0 ** -17
    rng = np.random.default_rng(5)
    names = dict(q="dq", k="dk", v="dv", log_decay="d_log_decay", beta="d_beta",
                 state0="dstate0")
    for name, gname in names.items():
        flat = x[name].reshape(-1)
        idx = rng.choice(flat.size, min(flat.size, 24), replace=False)
        if masked and name in ("log_decay", "beta"):  # include masked steps
            idx = np.concatenate([idx, [flat.size - 1, flat.size - 3]])
        fd = np.zeros(len(idx))
        for n, i in enumerate(idx):
            old = flat[i]
            flat[i] = old + h
            lp = _lb_loss(x)
            flat[i] = old - h
            lm = _lb_loss(x)
            flat[i] = old
            fd[n] = (lp - lm) / (2 * h)
        an = g[gname].reshape(-1)[idx]
        assert np.abs(an - fd).max() <= 1e-7 * max(np.abs(fd).max(), 1.0), name


def test_lb_identity_and_reset_closed_forms():
    """log_decay = 0, beta = 0 is the identity step (S_T = S_0, o_t = S_0^T q_t);
    log_decay = -800 (g = 0 in fp64) resets the state each step, so
    S_t = k_t (beta_t v_t)^T and o_t = <q_t, k_t> beta_t v_t (normalised q, k)."""
    x = _lb_inputs(1, 9, 1, 2, 5, 3, seed=31)
    q, k, v, s0 = x["q"], x["k"], x["v"], x["state0"]
    qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) / np.sqrt(q.shape[-1])
    kh = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    zero = np.zeros_like(x["beta"])
    o, sT = oracle.forward_lb(q, k, v, zero, zero, s0)
    np.testing.assert_array_equal(sT, s0)
    for h in range(2):
        np.testing.assert_allclose(o[0, :, h], qh[0, :, 0] @ s0[0, h], rtol=0, atol=1e-13)
    reset = np.full_like(x["beta"], -800.0)
    o, sT = oracle.forward_lb(q, k, v, reset, x["beta"], s0)
    for h in range(2):
        qk = (qh[0, :, 0] * kh[0, :, 0]).sum(-1)
        want = (qk * x["beta"][0, :, h])[:, None] * v[0, :, h]
        np.testing.assert_allclose(o[0, :, h], want, rtol=0, atol=1e-13)
        np.testing.assert_allclose(sT[0, h], np.outer(kh[0, -1, 0], x["beta"][0, -1, h] * v[0, -1, h]),
                                   rtol=0, atol=1e-13)
    g = oracle.backward_lb(q, k, v, reset, x["beta"], s0, None, x["d_o"], x["d_state_T"])
    assert np.all(g["d_log_decay"] == 0.0)   # d/dl = gbar * g with g = 0
    assert np.all(g["dstate0"] == 0.0)       # the first step erases S_0


def test_lb_matches_gate_form_and_chain_rule():
    """The two gate forms describe one recurrence: with l = -exp(A_log)
    softplus(min(a + dt_bias, 20)) and beta = sigmoid(b), the log_decay / beta
    form gives the same o and S_T, and the gate cotangents of the a / b form are
    its d_log_decay, d_beta through that map (clamp head included)."""
    w = wl.custom("lbmap", 2, 70, 1, 2, 6, 4, seed=41, mask="half_second_batch",
                  clamp_head=True)
    x = _inputs(w)
    xc = x["a"] + x["dt_bias"][None, None, :]
    l = -np.exp(x["A_log"])[None, None, :] * np.log1p(np.exp(np.minimum(xc, 20.0)))
    beta = 1.0 / (1.0 + np.exp(-x["b"]))
    o1, s1 = oracle.forward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                            x["state0"], x["mask"])
    o2, s2 = oracle.forward_lb(x["q"], x["k"], x["v"], l, beta, x["state0"], x["mask"])
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-12)
    g1 = oracle.backward(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                         x["state0"], x["mask"], x["d_o"], x["d_state_T"])
    g2 = oracle.backward_lb(x["q"], x["k"], x["v"], l, beta, x["state0"], x["mask"], x["d_o"],
                            x["d_state_T"])
    for n in ("dq", "dk", "dv", "dstate0"):
        np.testing.assert_allclose(g2[n], g1[n], rtol=0, atol=1e-10 * max(1.0, np.abs(g1[n]).max()))
    sig = 1.0 / (1.0 + np.exp(-xc))
    da = g2["d_log_decay"] * (-np.exp(x["A_log"]))[None, None, :] * np.where(xc <= 20.0, sig, 0.0)
    np.testing.assert_allclose(g1["da"], da, rtol=0, atol=1e-10 * max(1.0, np.abs(da).max()))
    np.testing.assert_allclose(g1["db"], g2["d_beta"] * beta * (1 - beta), rtol=0, atol=1e-10)
    np.testing.assert_allclose(g1["dA_log"], (g2["d_log_decay"] * l).sum((0, 1)), rtol=1e-10,
                               atol=1e-10)
    if x["mask"] is not None:
        off = x["mask"] == 0
        assert np.all(g2["d_log_decay"][off] == 0) and np.all(g2["d_beta"][off] == 0)


# -- per-key-channel gates (the mlx-lm page's vectorised gating, g.ndim == 4) --

def _kc_inputs(B, T, Hk, Hv, Dk, Dv, seed, masked=False):
    x = _lb_inputs(B, T, Hk, Hv, Dk, Dv, seed, masked)
    r = np.random.default_rng(seed + 1000)
    x["log_decay"] = -r.uniform(0.0, 2.0, (B, T, Hv, Dk))
    return x


def _kc_loss(x):
    o, sT = oracle.forward_kc(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                              x["mask"])
    return float((o * x["d_o"]).sum() + (sT * x["d_state_T"]).sum())


@pytest.mark.parametrize("masked", [False, True])
def test_kc_fd_all_grads(masked):
    """Central differences of L = <o, dO> + <S_T, dS_T> through the per-channel
    form: every input, one log-decay cotangent per key channel (GQA G = 2,
    T = 67 over two 64-step segments, optional mask)."""
    x = _kc_inputs(2, 67, 1, 2, 6, 4, seed=61 + masked, masked=masked)
    g = oracle.backward_kc(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                           x["mask"], x["d_o"], x["d_state_T"])
    h = 2.0 ** -17
    rng = np.random.default_rng(7)
    names = dict(q="dq", k="dk", v="dv", log_decay="d_log_decay", beta="d_beta",
                 state0="dstate0")
    for name, gname in names.items():
        flat = x[name].reshape(-1)
        idx = rng.choice(flat.size, min(flat.size, 24), replace=False)
        if masked and name in ("log_decay", "beta"):  # include masked steps
            idx = np.concatenate([idx, [flat.size - 1, flat.size - 5]])
        fd = np.zeros(len(idx))
        for n, i in enumerate(idx):
            old = flat[i]
            flat[i] = old + h
            lp = _kc_loss(x)
            flat[i] = old - h
            lm = _kc_loss(x)
            flat[i] = old
            fd[n] = (lp - lm) / (2 * h)
        an = g[gname].reshape(-1)[idx]
        assert np.abs(an - fd).max() <= 1e-7 * max(np.abs(fd).max(), 1.0), name
    if masked:
        off = x["mask"] == 0
        assert np.all(g["d_log_decay"][off] == 0) and np.all(g["d_beta"][off] == 0)


def test_kc_equal_channels_is_the_scalar_form():
    """With the same log-decay on every key channel the per-channel recurrence is
    the scalar one (written separately in the oracle): o, S_T, dq, dk, dv, d_beta
    and dstate0 agree, and the per-channel log-decay cotangents sum to the
    scalar one."""
    x = _lb_inputs(2, 70, 2, 4, 5, 3, seed=71, masked=True)
    lk = np.repeat(x["log_decay"][..., None], 5, axis=-1)
    o1, s1 = oracle.forward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                               x["mask"])
    o2, s2 = oracle.forward_kc(x["q"], x["k"], x["v"], lk, x["beta"], x["state0"], x["mask"])
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-12)
    g1 = oracle.backward_lb(x["q"], x["k"], x["v"], x["log_decay"], x["beta"], x["state0"],
                            x["mask"], x["d_o"], x["d_state_T"])
    g2 = oracle.backward_kc(x["q"], x["k"], x["v"], lk, x["beta"], x["state0"], x["mask"],
                            x["d_o"], x["d_state_T"])
    for n in ("dq", "dk", "dv", "d_beta", "dstate0"):
        np.testing.assert_allclose(g2[n], g1[n], rtol=0, atol=1e-10 * max(1.0, np.abs(g1[n]).max()))
    np.testing.assert_allclose(g2["d_log_decay"].sum(-1), g1["d_log_decay"], rtol=0,
                               atol=1e-10 * max(1.0, np.abs(g1["d_log_decay"]).max()))


def test_kc_channel_reset_and_freeze_closed_forms():
    """Key channel 0 with log_decay = -800 (g = 0 in fp64) and the others at 0
    (g = 1), beta = 0: row 0 of the state is cleared at the first step and every
    other row keeps its start value, S_T = diag(0, 1, ..., 1) S_0."""
    x = _kc_inputs(1, 6, 1, 2, 4, 3, seed=81)
    ld = np.zeros_like(x["log_decay"])
    ld[..., 0] = -800.0
    zero = np.zeros_like(x["beta"])
    _, sT = oracle.forward_kc(x["q"], x["k"], x["v"], ld, zero, x["state0"])
    want = x["state0"].copy()
    want[:, :, 0, :] = 0.0
    np.testing.assert_array_equal(sT, want)


# -- the causal conv1d update (torch-to-nnef page, CausalConvUpdateReified) -----

def _silu(x):
    return x / (1.0 + np.exp(-x))


@pytest.mark.parametrize("S,K", [(1, 4), (5, 4), (9, 3), (2, 1)])
def test_conv1d_matches_numpy_correlation(S, K):
    """out = SiLU of the valid correlation of the k taps with [state, hidden],
    first window dropped (numpy's convolve with the taps reversed);
    final_state = the last k samples."""
    r = np.random.default_rng(100 + S * 10 + K)
    B, C = 2, 5
    hid = r.standard_normal((B, C, S))
    st = r.standard_normal((B, C, K))
    w = r.standard_normal((C, K))
    out, fs = oracle.causal_conv1d_update(hid, st, w)
    for b in range(B):
        for c in range(C):
            x = np.concatenate([st[b, c], hid[b, c]])
            corr = np.convolve(x, w[c][::-1], mode="valid")  # length S + 1
            np.testing.assert_allclose(out[b, c], _silu(corr[1:]), rtol=1e-14, atol=1e-14)
            np.testing.assert_array_equal(fs[b, c], x[-K:])


def test_conv1d_delta_taps_and_split_carry():
    """A tap on the newest sample gives out_t = SiLU(x_t); a tap on the oldest
    in the window gives SiLU(x_{t-k+1}) (a k-1 step delay through the state);
    running S1 + S2 samples at once equals two calls with the state carried."""
    r = np.random.default_rng(7)
    B, C, K = 1, 3, 4
    hid = r.standard_normal((B, C, 10))
    st = r.standard_normal((B, C, K))
    last = np.zeros((C, K)); last[:, -1] = 1.0
    out, _ = oracle.causal_conv1d_update(hid, st, last)
    np.testing.assert_allclose(out, _silu(hid), rtol=1e-15, atol=0)
    first = np.zeros((C, K)); first[:, 0] = 1.0
    out, _ = oracle.causal_conv1d_update(hid, st, first)
    delayed = np.concatenate([st[:, :, 1:], hid], axis=-1)[:, :, :10]
    np.testing.assert_allclose(out, _silu(delayed), rtol=1e-15, atol=0)
    w = r.standard_normal((C, K))
    o_all, f_all = oracle.causal_conv1d_update(hid, st, w)
    o1, f1 = oracle.causal_conv1d_update(hid[:, :, :6], st, w)
    o2, f2 = oracle.causal_conv1d_update(hid[:, :, 6:], f1, w)
    np.testing.assert_array_equal(np.concatenate([o1, o2], axis=-1), o_all)
    np.testing.assert_array_equal(f2, f_all)
