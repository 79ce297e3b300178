"""fp64 oracle of the gated delta rule with rank-r compressed chunk states
(test infrastructure only: the tests and bench.py's CPU legs use it).

mlx-lm PR page, "Post-initial-submission extensions", Extension 1
("Compression-aware training"): the state is truncated to rank r by power
iteration at every chunk boundary, so only rank-r factors of each chunk
state need to be kept for the backward; three iterations are the page's
setting and ranks of at most 16 its working range (Extension 6).

Readings where the page is silent (each one is listed in the design notes):

* Boundaries are those between consecutive 64-step chunks, c = 1 .. NC - 1.
  The initial state enters chunk 0 as given, and the state after the last
  chunk is returned untruncated: neither is a boundary between two chunks.
  The truncation is not a step of the recurrence, so it applies whether or
  not the steps around it are masked.
* Truncation of S (Dk x Dv) to rank r: the range of S is estimated by
  subspace (power) iteration from a start block Omega (Dv x r) that the caller
  draws and passes in,
      Y = S Omega,  Q = orth(Y),  then `iters` times  Y = S (S^T Q),  Q = orth(Y),
  and S is replaced by its projection Q Q^T S onto span(Q), kept as the
  factors Q (Dk x r, orthonormal columns) and R = Q^T S (r x Dv).
  orth is Gram-Schmidt on the columns in order, each column orthogonalised
  twice against the earlier ones; a column whose remaining norm is at most
  1e-12 of its own norm (it lies in the span of the earlier ones, to
  rounding) is set to zero, so a state of rank below r keeps its whole range
  and nothing else.
* The VJP passes the state cotangent straight through each boundary: the
  backward is the chunked VJP evaluated along the compressed trajectory (each
  chunk from its truncated start state), with the truncation's own
  derivative taken as the identity.  It is the exact gradient of the forward
  in which each boundary adds the fixed offset P S - S (a stop-gradient on
  the truncation error).  Differentiating the truncation itself is
  ill-conditioned wherever the state's spectrum has no gap at r (its
  derivative divides by sigma_r^2 - sigma_{r+1}^2), which is the common case
  for states that decay over a chunk, and even with the basis held fixed the
  projected cotangent P S_bar changes by O(|S_bar|) with the choice of basis
  inside a numerically null part of the state's range.

The chunk recurrence itself is the pinned sequential oracle (`oracle.forward`
/ `oracle.backward`) run one chunk at a time from the truncated chunk state;
only the truncation and its VJP are new here, in numpy fp64.
"""

from __future__ import annotations

import numpy as np

import oracle as _o

CHUNK = 64


def gram_schmidt(Y, drop=1e-12):
    """Columns of Y orthonormalised in order (modified Gram-Schmidt with one
    reorthogonalisation pass, fp64: a single pass loses orthogonality in
    proportion to the condition of Y, which power iteration makes large); a
    column whose residual norm is <= drop x its own norm before the
    orthogonalisation (a column in the span of the earlier ones, to rounding)
    becomes zero."""
    Y = np.asarray(Y, dtype=np.float64)
    Q = np.zeros_like(Y)
    for j in range(Y.shape[1]):
        w = Y[:, j].copy()
        own = float(np.sqrt(w @ w))
        for _ in range(2):
            for i in range(j):
                w -= (Q[:, i] @ w) * Q[:, i]
        n = float(np.sqrt(w @ w))
        if own > 0 and n > drop * own:
            Q[:, j] = w / n
    return Q


def subspace_basis(S, omega, iters):
    """Orthonormal basis (Dk x r; zero columns where the range is exhausted)
    of the rank-r range estimate of S after `iters` power iterations from the
    start block omega (Dv x r)."""
    S = np.asarray(S, dtype=np.float64)
    Q = gram_schmidt(S @ omega)
    for _ in range(int(iters)):
        Q = gram_schmidt(S @ (S.T @ Q))
    return Q


def truncate(S, omega, iters):
    """Rank-r truncation of one state: returns (Q Q^T S, Q, R = Q^T S)."""
    Q = subspace_basis(S, omega, iters)
    R = Q.T @ np.asarray(S, dtype=np.float64)
    return Q @ R, Q, R


def _f64(x):
    return _o._f64(x)


def _chunks(T):
    return [(c0, min(T, c0 + CHUNK)) for c0 in range(0, T, CHUNK)]


def _sl(x, t0, t1):
    return None if x is None else x[:, t0:t1]


def forward_compressed(q, k, v, a, b, A_log, dt_bias, state0, mask, omega, iters=3,
                       offsets=None):
    """Forward with the state truncated at every chunk boundary.

    Returns (o, state_T, chunk_states, bases, offsets): chunk_states[c] is the
    state chunk c starts from ([B, Hv, Dk, Dv]: state0 for c = 0, the
    truncated state for c >= 1), bases[c] the basis Q of boundary c
    ([B, Hv, Dk, r]) and offsets[c] the truncation's change P S - S there
    (both None for c = 0).  Passing `offsets` adds those fixed offsets at the
    boundaries instead of truncating (the function whose exact gradient the
    straight-through VJP is; used to check it by finite differences)."""
    q, k, v, a, b, A_log, dt_bias, state0, omega = map(
        _f64, (q, k, v, a, b, A_log, dt_bias, state0, omega))
    mask = _o._u8(mask)
    B, T, Hk, Hv, Dk, Dv = _o._dims(q, v)
    S = np.zeros((B, Hv, Dk, Dv)) if state0 is None else state0.copy()
    o = np.zeros((B, T, Hv, Dv))
    states, bases, offs = [], [], []
    spans = _chunks(T)
    for c, (t0, t1) in enumerate(spans):
        if c > 0 and offsets is not None:
            bases.append(None)
            offs.append(offsets[c])
            S = S + offsets[c]
        elif c > 0:
            Qc = np.zeros((B, Hv, Dk, omega.shape[1]))
            St = np.zeros_like(S)
            for bb in range(B):
                for h in range(Hv):
                    Qc[bb, h] = subspace_basis(S[bb, h], omega, iters)
                    St[bb, h] = Qc[bb, h] @ (Qc[bb, h].T @ S[bb, h])
            bases.append(Qc)
            offs.append(St - S)
            S = St
        else:
            bases.append(None)
            offs.append(None)
        states.append(S.copy())
        oc, S = _o.forward(_sl(q, t0, t1), _sl(k, t0, t1), _sl(v, t0, t1), _sl(a, t0, t1),
                           _sl(b, t0, t1), A_log, dt_bias, S, _sl(mask, t0, t1))
        o[:, t0:t1] = oc
    return o, S, states, bases, offs


def backward_compressed(q, k, v, a, b, A_log, dt_bias, state0, mask, d_o, d_state_T, omega,
                        iters=3):
    """VJP of forward_compressed, the state cotangent passed straight through
    every boundary: chunk by chunk in reverse, the VJP of the recurrence from
    that chunk's (truncated) start state.

    Returns a dict with dq, dk, dv, da, db, dA_log, ddt_bias, dstate0 (the
    names and shapes of oracle.backward)."""
    q, k, v, a, b, A_log, dt_bias, state0, d_o, d_state_T, omega = map(
        _f64, (q, k, v, a, b, A_log, dt_bias, state0, d_o, d_state_T, omega))
    mask = _o._u8(mask)
    B, T, Hk, Hv, Dk, Dv = _o._dims(q, v)
    _, _, states, _, _ = forward_compressed(q, k, v, a, b, A_log, dt_bias, state0, mask,
                                            omega, iters)
    out = dict(dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape),
               da=np.zeros(a.shape), db=np.zeros(b.shape), dA_log=np.zeros(Hv),
               ddt_bias=np.zeros(Hv), dstate0=None)
    Sb = np.zeros((B, Hv, Dk, Dv)) if d_state_T is None else d_state_T.copy()
    spans = _chunks(T)
    for c in reversed(range(len(spans))):
        t0, t1 = spans[c]
        g = _o.backward(_sl(q, t0, t1), _sl(k, t0, t1), _sl(v, t0, t1), _sl(a, t0, t1),
                        _sl(b, t0, t1), A_log, dt_bias, states[c], _sl(mask, t0, t1),
                        _sl(d_o, t0, t1), Sb)
        for n in ("dq", "dk", "dv", "da", "db"):
            out[n][:, t0:t1] = g[n]
        out["dA_log"] += g["dA_log"]
        out["ddt_bias"] += g["ddt_bias"]
        Sb = g["dstate0"]  # cotangent of the state chunk c starts from, passed on
    out["dstate0"] = Sb
    return out


def checkpoint_values(B, Hv, Dk, Dv, T, rank):
    """Values kept per (b, h) between the forward and the backward: the
    initial state in full and rank-r factors (Dk + Dv) r for each of the
    NC - 1 boundaries, against Dk Dv for each of the NC chunk states
    uncompressed."""
    NC = (T + CHUNK - 1) // CHUNK
    return B * Hv * (Dk * Dv + (NC - 1) * (Dk + Dv) * rank), B * Hv * NC * Dk * Dv
