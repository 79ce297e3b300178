"""Pins of the compressed-state oracle (oracle/compressed.py): the gated delta
rule with the state truncated to rank r by power iteration at every chunk
boundary (mlx-lm page, "Post-initial-submission extensions", Extension 1).

None of these compares the oracle with itself.  The truncation is pinned by
facts of linear algebra (a state of rank <= r is left unchanged; with many
iterations the result is the Eckart-Young best rank-r approximation, i.e.
numpy's SVD truncated; the result is a projection, so applying it twice
changes nothing; no rank-r matrix is closer to S than the SVD truncation).
The recurrence with truncation is pinned by its special cases (one chunk has
no boundary and equals the plain recurrence; a rank equal to the key width
makes every truncation the identity) and its straight-through VJP by central
differences of the forward in which every boundary adds its truncation
offset P S - S held fixed, the function whose exact gradient that VJP is.
"""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_06_gb300 import workloads as wl
from oracle import compressed as oc


def _np(x):
    return None if x is None else x.detach().to(torch.float64).numpy().copy()


def _inputs(w, seed=None):
    x = wl.make_inputs(w, seed)
    return {k: _np(v) if k != "mask" else (None if v is None else v.numpy().copy())
            for k, v in x.items()}


def _omega(Dv, r, seed=0):
    return np.random.default_rng(seed).standard_normal((Dv, r))


def _graded(m, n, sv, seed=0):
    """m x n matrix with singular values sv (random orthonormal factors)."""
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.standard_normal((m, m)))
    V, _ = np.linalg.qr(rng.standard_normal((n, n)))
    k = len(sv)
    return (U[:, :k] * np.asarray(sv)) @ V[:, :k].T


def _rel(x, y):
    return float(np.abs(x - y).max() / max(np.abs(y).max(), 1e-300))


# -- the truncation -------------------------------------------------------------

@pytest.mark.parametrize("rank_S,r", [(4, 4), (2, 4), (1, 16), (0, 3)])
def test_state_of_rank_at_most_r_is_unchanged(rank_S, r):
    rng = np.random.default_rng(rank_S * 10 + r)
    S = rng.standard_normal((24, rank_S)) @ rng.standard_normal((rank_S, 20))
    St, Q, R = oc.truncate(S, _omega(20, r), 3)
    assert np.abs(St - S).max() <= 1e-12 * max(np.abs(S).max(), 1.0)
    # the kept basis is orthonormal on its nonzero columns
    nz = np.linalg.norm(Q, axis=0) > 0
    assert nz.sum() == rank_S
    assert np.allclose(Q[:, nz].T @ Q[:, nz], np.eye(rank_S), atol=1e-12)
    assert np.allclose(Q @ R, St, atol=1e-13)


def test_many_iterations_give_the_eckart_young_truncation():
    sv = [10, 8, 6, 5, 4, 3.5, 3, 2.5, 1.0, 0.8, 0.5, 0.3, 0.2, 0.1]
    S = _graded(32, 24, sv, seed=1)
    r = 8
    U, s, Vt = np.linalg.svd(S)
    best = (U[:, :r] * s[:r]) @ Vt[:r]
    St, _, _ = oc.truncate(S, _omega(24, r, seed=2), 200)
    assert _rel(St, best) <= 1e-9


def test_three_iterations_are_rank_r_and_no_closer_than_svd():
    rng = np.random.default_rng(5)
    S = rng.standard_normal((48, 40)) * np.linspace(2.0, 0.1, 40)
    r = 6
    U, s, Vt = np.linalg.svd(S)
    best = (U[:, :r] * s[:r]) @ Vt[:r]
    St, Q, _ = oc.truncate(S, _omega(40, r, seed=3), 3)
    assert np.linalg.matrix_rank(St, tol=1e-9 * s[0]) == r
    e3 = np.linalg.norm(S - St)
    eb = np.linalg.norm(S - best)
    assert e3 >= eb * (1 - 1e-12)
    assert e3 <= 1.5 * eb  # three iterations already come close to the optimum


def test_truncation_is_a_projection():
    rng = np.random.default_rng(7)
    S = rng.standard_normal((32, 16))
    om = _omega(16, 5, seed=4)
    St, Q, _ = oc.truncate(S, om, 3)
    St2, _, _ = oc.truncate(St, om, 3)
    assert _rel(St2, St) <= 1e-10
    # P = Q Q^T is symmetric and idempotent
    P = Q @ Q.T
    assert np.allclose(P, P.T, atol=1e-14) and np.allclose(P @ P, P, atol=1e-12)


# -- the recurrence with truncation -----------------------------------------------

def _args(x):
    return [x[n] for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0", "mask")]


def test_one_chunk_has_no_boundary():
    """T <= 64: no boundary, the plain recurrence exactly (a full-rank initial
    state is not truncated)."""
    w = wl.custom("c1", 2, 60, 2, 4, 16, 12, seed=11, mask="half_second_batch")
    x = _inputs(w)
    om = _omega(12, 2)
    o, sT, _, _, _ = oc.forward_compressed(*_args(x), om, 3)
    o_p, s_p = oracle.forward(*_args(x))
    assert np.array_equal(o, o_p) and np.array_equal(sT, s_p)
    g = oc.backward_compressed(*_args(x), x["d_o"], x["d_state_T"], om, 3)
    gp = oracle.backward(*_args(x), x["d_o"], x["d_state_T"])
    for n in oracle.GRAD_NAMES:
        assert np.array_equal(g[n], gp[n]), n


def test_rank_equal_to_key_width_is_the_plain_recurrence():
    """r = Dk <= Dv: every boundary projects onto the whole key space, so the
    result is the plain recurrence up to rounding (200 steps, 3 boundaries).
    The gates are set near g = 1 (a = -20) so that every chunk-end state has
    full rank Dk: with fast decay the states are numerically of lower rank, and
    the fixed-basis VJP then rightly projects the cotangent onto their range."""
    w = wl.custom("cfull", 1, 200, 1, 2, 8, 12, seed=13, clamp_head=False)
    x = _inputs(w)
    x["a"][:] = -20.0
    om = _omega(12, 8, seed=6)
    o, sT, _, _, _ = oc.forward_compressed(*_args(x), om, 3)
    o_p, s_p = oracle.forward(*_args(x))
    assert _rel(o, o_p) <= 1e-12 and _rel(sT, s_p) <= 1e-12
    g = oc.backward_compressed(*_args(x), x["d_o"], x["d_state_T"], om, 3)
    gp = oracle.backward(*_args(x), x["d_o"], x["d_state_T"])
    for n in oracle.GRAD_NAMES:
        assert _rel(g[n], gp[n]) <= 1e-10, n


def test_truncation_applies_at_boundaries_only():
    """With r = 2 on full-rank states the outputs of chunk 0 are those of the
    plain recurrence exactly and the later ones differ; each later chunk starts
    from a state of rank <= 2 equal to Q Q^T of the untruncated chunk end."""
    w = wl.custom("cb", 1, 150, 1, 2, 16, 12, seed=17)
    x = _inputs(w)
    om = _omega(12, 2, seed=8)
    o, _, states, bases, _ = oc.forward_compressed(*_args(x), om, 3)
    o_p, _ = oracle.forward(*_args(x))
    assert np.array_equal(o[:, :64], o_p[:, :64])
    assert _rel(o[:, 64:], o_p[:, 64:]) > 1e-3
    for c in (1, 2):
        for h in range(2):
            assert np.linalg.matrix_rank(states[c][0, h], tol=1e-10) <= 2
        # the chunk end before boundary c, rerun from the previous chunk state
        t0, t1 = 64 * (c - 1), 64 * c
        sl = lambda z: None if z is None else z[:, t0:t1]  # noqa: E731
        _, S_end = oracle.forward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["a"]), sl(x["b"]),
                                  x["A_log"], x["dt_bias"], states[c - 1], sl(x["mask"]))
        Q = bases[c]
        assert _rel(states[c], np.einsum("bhir,bhjr,bhjv->bhiv", Q, Q, S_end)) <= 1e-12


PRIMALS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state0")
GRAD_OF = dict(q="dq", k="dk", v="dv", a="da", b="db", A_log="dA_log", dt_bias="ddt_bias",
               state0="dstate0")


def test_straight_through_vjp_matches_central_differences():
    """L = <o, dO> + <S_T, dS_T> of the forward in which every boundary adds its
    truncation offset P S - S, held at its value at the unperturbed inputs:
    fp64 central differences of every input against backward_compressed (3
    boundaries, GQA, a masked tail, the clamp head)."""
    w = wl.custom("cfd", 2, 200, 1, 2, 8, 6, seed=19, mask="half_second_batch", clamp_head=True)
    x = _inputs(w)
    om = _omega(6, 3, seed=9)
    _, _, _, _, offs = oc.forward_compressed(*_args(x), om, 3)
    assert max(np.abs(d).max() for d in offs[1:]) > 1e-3  # the truncation does act
    g = oc.backward_compressed(*_args(x), x["d_o"], x["d_state_T"], om, 3)

    def loss():
        o, sT, _, _, _ = oc.forward_compressed(*_args(x), om, 3, offsets=offs)
        return float((o * x["d_o"]).sum() + (sT * x["d_state_T"]).sum())

    h = 2.0 ** -17
    rng = np.random.default_rng(0)
    for name in PRIMALS:
        flat = x[name].reshape(-1)
        idx = rng.choice(flat.size, min(flat.size, 12), replace=False)
        fd = np.zeros(len(idx))
        for n, i in enumerate(idx):
            old = flat[i]
            flat[i] = old + h
            lp = loss()
            flat[i] = old - h
            lm = loss()
            flat[i] = old
            fd[n] = (lp - lm) / (2 * h)
        an = g[GRAD_OF[name]].reshape(-1)[idx]
        assert np.abs(an - fd).max() <= 1e-7 * max(np.abs(fd).max(), 1.0), name


def test_offsets_reproduce_the_truncated_forward():
    """Adding the recorded offsets instead of truncating reproduces the
    compressed forward (so the finite differences above differentiate the
    compressed trajectory itself)."""
    w = wl.custom("coff", 1, 150, 1, 2, 16, 12, seed=29)
    x = _inputs(w)
    om = _omega(12, 3, seed=12)
    o, sT, _, _, offs = oc.forward_compressed(*_args(x), om, 3)
    o2, s2, _, _, _ = oc.forward_compressed(*_args(x), om, 3, offsets=offs)
    assert _rel(o2, o) <= 1e-13 and _rel(s2, sT) <= 1e-13


def test_checkpoint_values():
    kept, full = oc.checkpoint_values(1, 64, 192, 128, 2048, 16)
    # 9B layer at rank 16: S0 in full plus 31 boundaries of (192 + 128) x 16 factors
    assert kept == 64 * (192 * 128 + 31 * 320 * 16) and full == 64 * 32 * 192 * 128
    assert full / kept > 3.5
