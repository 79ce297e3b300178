/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta rule (GatedDeltaNet).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes, and where each step is defined:
 *
 *  - Op contract (torch-to-nnef, "custom_extractors/gdn", op contract):
 *      q, k      [B, T, Hk, Dk]
 *      v         [B, T, Hv, Dv]     Hv = G * Hk, value head h reads q/k head h / G
 *      state     [B, Hv, Dk, Dv]
 *      output    [B, T, Hv, Dv],  final_state [B, Hv, Dk, Dv]
 *    q and k are L2-normalised with eps 1e-6 and q is scaled by 1/sqrt(Dk)
 *    inside the op.  The contract states a single width w; this oracle keeps
 *    Dk and Dv separate (the mlx-lm page's performance section uses Dk=192,
 *    Dv=128).
 *  - Gates (mlx-lm PR "Add gated_delta_update VJP", "What this PR adds" and
 *    "Covered corner cases"): g = exp(-exp(A_log) * softplus(a + dt_bias))
 *    with the softplus argument clamped, beta = sigmoid(b).  The clamp value
 *    is not printed; this oracle uses softplus(min(x, 20)) whose derivative is
 *    sigmoid(x) for x <= 20 and 0 above.
 *  - Second input form (torch-to-nnef page, op contract: log_decay and beta
 *    [b, S, hv]): the per-step log-decay l = log g and beta are given
 *    directly; its VJP returns their cotangents.  Both forms run one fp64
 *    core that takes (l, beta) per step; the a / b form computes them first.
 *  - Recurrence (the recurrent step that both pages name): per (b, h)
 *      S <- g S;  delta = beta (v - S^T k);  S <- S + k delta^T;  o = S^T q.
 *    A masked step leaves S unchanged (mlx-lm page, "Covered corner cases":
 *    the half-masked final state equals the state after the unmasked prefix);
 *    the page fixes only the state, so the output of a masked step is read as
 *    o = S^T q with the unchanged state.
 *  - VJP (mlx-lm page, "What this PR adds": gradients for q, k, v, a, b,
 *    A_log, dt_bias and state): plain reverse-mode differentiation of the
 *    sequential recurrence above, derived by hand, with the state stored
 *    every 64 steps and recomputed inside each 64-step segment (mlx-lm page,
 *    "Design notes": CHUNK_SIZE = 64 bounds memory to one chunk).
 *  - Causal conv1d update (torch-to-nnef page, CausalConvUpdateReified: a
 *    depthwise causal conv1d + SiLU with a k-sample carry state; hidden
 *    [b, C, S], conv_state [b, C, k], weight [C, k] -> out [b, C, S],
 *    final_state [b, C, k]).  Reading: per channel the k carried samples and
 *    the S new ones form one sequence x; out_t = SiLU(sum_i w_i x_{t+1+i}), the
 *    correlation of the k taps with the window that ends at new sample t (the
 *    oldest carried sample falls outside every window); final_state = the last
 *    k samples of x; no bias.
 *  - Chunked form (torch-to-nnef page: the chunked rule computes the same
 *    recurrence with different blocking; mlx-lm page, "Scope and
 *    follow-ups": chunk-parallel rewrite through a lower-triangular solve):
 *    an independent fp64 forward in the WY/UT form, used only to check that
 *    chunked equals sequential up to rounding.
 *  - Associative form (mlx-lm page, "Post-initial-submission extensions",
 *    Extension 5: the recurrence as an associative monoid): each step as an
 *    affine map of the state, runs of steps composed, a tree prefix over the
 *    runs; used only to check that this evaluation order equals the
 *    sequential recurrence up to rounding.
 *
 * Everything is fp64.  Parallelism: OpenMP over independent (b, h) pairs;
 * all cross-pair sums run afterwards in a fixed serial order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NORM_EPS 1e-6
#define SOFTPLUS_CLAMP 20.0
#define SEGMENT 64

/* ---- scalar helpers ---------------------------------------------------- */

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus with its argument clamped from above (reading of the clamp). */
static double softplus_clamped(double x) {
    double xc = x < SOFTPLUS_CLAMP ? x : SOFTPLUS_CLAMP;
    return log1p(exp(xc));
}

/* d/dx softplus(min(x, 20)) */
static double softplus_clamped_grad(double x) {
    return x <= SOFTPLUS_CLAMP ? sigmoid_d(x) : 0.0;
}

/* log-decay l = log g = -exp(A_log) * softplus(min(a + dt_bias, 20)) */
static double log_decay(double a, double A_log, double dt_bias) {
    return -exp(A_log) * softplus_clamped(a + dt_bias);
}

/* 1 / sqrt(sum x^2 + eps) over n entries */
static double inv_norm(const double* x, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += x[i] * x[i];
    return 1.0 / sqrt(s + NORM_EPS);
}

typedef struct {
    int64_t B, T, Hk, Hv, Dk, Dv;
} dims_t;

static int check_dims(const dims_t* d) {
    if (d->B < 1 || d->T < 0 || d->Hk < 1 || d->Hv < 1 || d->Dk < 1 || d->Dv < 1) return 1;
    if (d->Hv % d->Hk) return 2;
    return 0;
}

/* index helpers (row-major, contiguous) */
#define IQK(d, b, t, j) ((((b) * (d)->T + (t)) * (d)->Hk + (j)) * (d)->Dk)
#define IV(d, b, t, h) ((((b) * (d)->T + (t)) * (d)->Hv + (h)) * (d)->Dv)
#define IG(d, b, t, h) (((b) * (d)->T + (t)) * (d)->Hv + (h))
#define IS(d, b, h) (((b) * (d)->Hv + (h)) * (d)->Dk * (d)->Dv)

/* Normalised query / key of step t for value head h (GQA: key head h / G). */
static void load_qk_hat(const dims_t* d, const double* q, const double* k, int64_t b,
                        int64_t t, int64_t h, double* qh, double* kh) {
    int64_t G = d->Hv / d->Hk, j = h / G;
    const double* qp = q + IQK(d, b, t, j);
    const double* kp = k + IQK(d, b, t, j);
    double rq = inv_norm(qp, d->Dk) / sqrt((double)d->Dk);
    double rk = inv_norm(kp, d->Dk);
    for (int64_t i = 0; i < d->Dk; ++i) {
        qh[i] = qp[i] * rq;
        kh[i] = kp[i] * rk;
    }
}

/* One applied step of the recurrence on S (Dk x Dv, row-major).
 * Returns delta in dl, the prediction p = (gS)^T k in p. */
static void apply_step(int64_t Dk, int64_t Dv, double* S, double g, double beta,
                       const double* kh, const double* v, double* p, double* dl) {
    for (int64_t i = 0; i < Dk * Dv; ++i) S[i] *= g;
    for (int64_t c = 0; c < Dv; ++c) p[c] = 0.0;
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < Dv; ++c) p[c] += S[r * Dv + c] * kh[r];
    for (int64_t c = 0; c < Dv; ++c) dl[c] = beta * (v[c] - p[c]);
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < Dv; ++c) S[r * Dv + c] += kh[r] * dl[c];
}

/* o = S^T qh */
static void read_out(int64_t Dk, int64_t Dv, const double* S, const double* qh, double* o) {
    for (int64_t c = 0; c < Dv; ++c) o[c] = 0.0;
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < Dv; ++c) o[c] += S[r * Dv + c] * qh[r];
}

/* Per-step gates of the a / b form in fp64: lg = log g, bt = beta ([B, T, Hv]).
 * Returns 0, or 3 when memory runs out (both arrays then NULL). */
static int gates_ab(const dims_t* d, const double* a, const double* b, const double* A_log,
                    const double* dt_bias, double** lg, double** bt) {
    int64_t n = d->B * d->T * d->Hv;
    *lg = malloc(sizeof(double) * (n > 0 ? n : 1));
    *bt = malloc(sizeof(double) * (n > 0 ? n : 1));
    if (!*lg || !*bt) { free(*lg); free(*bt); *lg = *bt = NULL; return 3; }
    for (int64_t bb = 0; bb < d->B; ++bb)
        for (int64_t t = 0; t < d->T; ++t)
            for (int64_t h = 0; h < d->Hv; ++h) {
                int64_t ix = IG(d, bb, t, h);
                (*lg)[ix] = log_decay(a[ix], A_log[h], dt_bias[h]);
                (*bt)[ix] = sigmoid_d(b[ix]);
            }
    return 0;
}

/* ---- sequential forward -------------------------------------------------- */

static int forward_core(const dims_t* dd, const double* q, const double* k, const double* v,
                        const double* lg, const double* bt, const double* state0,
                        const uint8_t* mask, double* o, double* state_T) {
    const dims_t d = *dd;
    const int64_t B = d.B, T = d.T, Hv = d.Hv, Dk = d.Dk, Dv = d.Dv;
    int64_t npairs = B * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pr = 0; pr < npairs; ++pr) {
        int64_t bb = pr / Hv, h = pr % Hv;
        double* S = state_T + IS(&d, bb, h);
        if (state0)
            memcpy(S, state0 + IS(&d, bb, h), sizeof(double) * Dk * Dv);
        else
            memset(S, 0, sizeof(double) * Dk * Dv);
        double* qh = malloc(sizeof(double) * Dk);
        double* kh = malloc(sizeof(double) * Dk);
        double* p = malloc(sizeof(double) * Dv);
        double* dl = malloc(sizeof(double) * Dv);
        for (int64_t t = 0; t < T; ++t) {
            load_qk_hat(&d, q, k, bb, t, h, qh, kh);
            int on = mask ? (mask[bb * T + t] != 0) : 1;
            if (on) {
                double g = exp(lg[IG(&d, bb, t, h)]);
                double beta = bt[IG(&d, bb, t, h)];
                apply_step(Dk, Dv, S, g, beta, kh, v + IV(&d, bb, t, h), p, dl);
            }
            read_out(Dk, Dv, S, qh, o + IV(&d, bb, t, h));
        }
        free(qh); free(kh); free(p); free(dl);
    }
    return 0;
}

int gdn_oracle_forward(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                       const double* q, const double* k, const double* v, const double* a,
                       const double* b, const double* A_log, const double* dt_bias,
                       const double* state0, const uint8_t* mask, double* o,
                       double* state_T) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    double *lg, *bt;
    if (gates_ab(&d, a, b, A_log, dt_bias, &lg, &bt)) return 3;
    rc = forward_core(&d, q, k, v, lg, bt, state0, mask, o, state_T);
    free(lg); free(bt);
    return rc;
}

/* log_decay / beta form: l and beta per step, [B, T, Hv] */
int gdn_oracle_forward_lb(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                          const double* q, const double* k, const double* v,
                          const double* log_decay_, const double* beta, const double* state0,
                          const uint8_t* mask, double* o, double* state_T) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    return forward_core(&d, q, k, v, log_decay_, beta, state0, mask, o, state_T);
}

/* ---- chunked (WY/UT) forward: second, independent formulation ------------- */
/*
 * Inside one chunk of L steps with start state S0 (all quantities local):
 *   Gam_i = sum_{s<=i} l_s, gam_i = exp(Gam_i), M_ij = exp(Gam_i - Gam_j) (j<=i)
 *   A_ij  = beta_i M_ij <k_i, k_j>            (j < i, strictly lower)
 *   (I + A) X = R  solved by forward substitution for
 *        R = [diag(beta) V | diag(beta gam) K]  ->  X = [U | W]
 *   Delta = U - W S0
 *   O     = diag(gam) Q S0 + P Delta,   P_ij = M_ij <q_i, k_j>  (j <= i)
 *   S     = gam_L S0 + K^T diag(e) Delta,   e_j = exp(Gam_L - Gam_j)
 * Masked steps enter as l = 0, beta = 0 (an identity step).
 */
int gdn_oracle_forward_chunked(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk,
                               int64_t Dv, int64_t C, const double* q, const double* k,
                               const double* v, const double* a, const double* b,
                               const double* A_log, const double* dt_bias,
                               const double* state0, const uint8_t* mask, double* o,
                               double* state_T) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    if (C < 1) return 1;
    int64_t npairs = B * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pr = 0; pr < npairs; ++pr) {
        int64_t bb = pr / Hv, h = pr % Hv;
        double* S = state_T + IS(&d, bb, h);
        if (state0)
            memcpy(S, state0 + IS(&d, bb, h), sizeof(double) * Dk * Dv);
        else
            memset(S, 0, sizeof(double) * Dk * Dv);
        double* Q = malloc(sizeof(double) * C * Dk);
        double* K = malloc(sizeof(double) * C * Dk);
        double* V = malloc(sizeof(double) * C * Dv);
        double* lg = malloc(sizeof(double) * C);
        double* bt = malloc(sizeof(double) * C);
        double* Gm = malloc(sizeof(double) * C);
        double* A = malloc(sizeof(double) * C * C);
        double* U = malloc(sizeof(double) * C * Dv);
        double* W = malloc(sizeof(double) * C * Dk);
        double* Dl = malloc(sizeof(double) * C * Dv);
        double* Snew = malloc(sizeof(double) * Dk * Dv);
        for (int64_t t0 = 0; t0 < T; t0 += C) {
            int64_t L = (T - t0) < C ? (T - t0) : C;
            for (int64_t i = 0; i < L; ++i) {
                int64_t t = t0 + i;
                load_qk_hat(&d, q, k, bb, t, h, Q + i * Dk, K + i * Dk);
                memcpy(V + i * Dv, v + IV(&d, bb, t, h), sizeof(double) * Dv);
                int on = mask ? (mask[bb * T + t] != 0) : 1;
                lg[i] = on ? log_decay(a[IG(&d, bb, t, h)], A_log[h], dt_bias[h]) : 0.0;
                bt[i] = on ? sigmoid_d(b[IG(&d, bb, t, h)]) : 0.0;
                Gm[i] = (i ? Gm[i - 1] : 0.0) + lg[i];
            }
            /* A (strictly lower) */
            for (int64_t i = 0; i < L; ++i)
                for (int64_t j = 0; j < i; ++j) {
                    double kk = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) kk += K[i * Dk + r] * K[j * Dk + r];
                    A[i * C + j] = bt[i] * exp(Gm[i] - Gm[j]) * kk;
                }
            /* forward substitution: (I + A) [U | W] = [diag(beta) V | diag(beta gam) K] */
            for (int64_t i = 0; i < L; ++i) {
                double gi = exp(Gm[i]);
                for (int64_t c = 0; c < Dv; ++c) U[i * Dv + c] = bt[i] * V[i * Dv + c];
                for (int64_t r = 0; r < Dk; ++r) W[i * Dk + r] = bt[i] * gi * K[i * Dk + r];
                for (int64_t j = 0; j < i; ++j) {
                    double aij = A[i * C + j];
                    for (int64_t c = 0; c < Dv; ++c) U[i * Dv + c] -= aij * U[j * Dv + c];
                    for (int64_t r = 0; r < Dk; ++r) W[i * Dk + r] -= aij * W[j * Dk + r];
                }
            }
            /* Delta = U - W S0 */
            for (int64_t i = 0; i < L; ++i)
                for (int64_t c = 0; c < Dv; ++c) {
                    double ws = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) ws += W[i * Dk + r] * S[r * Dv + c];
                    Dl[i * Dv + c] = U[i * Dv + c] - ws;
                }
            /* O = diag(gam) Q S0 + P Delta */
            for (int64_t i = 0; i < L; ++i) {
                double* oi = o + IV(&d, bb, t0 + i, h);
                double gi = exp(Gm[i]);
                for (int64_t c = 0; c < Dv; ++c) {
                    double qs = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) qs += Q[i * Dk + r] * S[r * Dv + c];
                    oi[c] = gi * qs;
                }
                for (int64_t j = 0; j <= i; ++j) {
                    double qk = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) qk += Q[i * Dk + r] * K[j * Dk + r];
                    double pij = exp(Gm[i] - Gm[j]) * qk;
                    for (int64_t c = 0; c < Dv; ++c) oi[c] += pij * Dl[j * Dv + c];
                }
            }
            /* S = gam_L S0 + K^T diag(e) Delta */
            double gL = exp(Gm[L - 1]);
            for (int64_t r = 0; r < Dk; ++r)
                for (int64_t c = 0; c < Dv; ++c) Snew[r * Dv + c] = gL * S[r * Dv + c];
            for (int64_t j = 0; j < L; ++j) {
                double ej = exp(Gm[L - 1] - Gm[j]);
                for (int64_t r = 0; r < Dk; ++r) {
                    double kr = ej * K[j * Dk + r];
                    for (int64_t c = 0; c < Dv; ++c) Snew[r * Dv + c] += kr * Dl[j * Dv + c];
                }
            }
            memcpy(S, Snew, sizeof(double) * Dk * Dv);
        }
        free(Q); free(K); free(V); free(lg); free(bt); free(Gm); free(A);
        free(U); free(W); free(Dl); free(Snew);
    }
    return 0;
}

/* ---- associative (monoid) form of the forward ------------------------------
 *
 * mlx-lm page, "Post-initial-submission extensions", Extension 5: the
 * recurrence written as an associative monoid, so that it can be evaluated by a
 * scan other than one sequential pass.  Written out, an applied step
 *   S -> g S + k beta (v - (g S)^T k)^T
 * is the affine map S -> A S + M with A = g (I - beta k k^T) (Dk x Dk) and
 * M = beta k v^T (Dk x Dv); a masked step is the identity map (I, 0).  "First
 * x, then y" is x (+) y = (A_y A_x, A_y M_x + M_y), which is associative with
 * identity (I, 0).
 *
 * This form cuts the T steps into runs of seg_len, composes each run's map from
 * its steps, takes the exclusive prefix of the run maps with a balanced tree
 * (an up-sweep then a down-sweep over a power-of-two array padded with
 * identities), applies each prefix to state0 for the run's start state, and
 * replays each run from its start state for the outputs.  It exists only to
 * check that this evaluation order gives the sequential recurrence.
 */

typedef struct {
    double* A; /* Dk x Dk */
    double* M; /* Dk x Dv */
} amap_t;

static void amap_identity(int64_t Dk, int64_t Dv, amap_t* m) {
    memset(m->A, 0, sizeof(double) * Dk * Dk);
    for (int64_t i = 0; i < Dk; ++i) m->A[i * Dk + i] = 1.0;
    memset(m->M, 0, sizeof(double) * Dk * Dv);
}

/* X (Dk x n) <- g (X - beta k (k^T X)): the linear part of one step applied to X */
static void step_linear(int64_t Dk, int64_t n, double* X, double g, double beta,
                        const double* kh, double* tmp) {
    for (int64_t c = 0; c < n; ++c) tmp[c] = 0.0;
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < n; ++c) tmp[c] += kh[r] * X[r * n + c];
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < n; ++c) X[r * n + c] = g * (X[r * n + c] - beta * kh[r] * tmp[c]);
}

/* out = x (+) y = (A_y A_x, A_y M_x + M_y); out may not alias x or y */
static void amap_then(int64_t Dk, int64_t Dv, const amap_t* x, const amap_t* y, amap_t* out) {
    for (int64_t i = 0; i < Dk; ++i) {
        for (int64_t j = 0; j < Dk; ++j) {
            double s = 0.0;
            for (int64_t l = 0; l < Dk; ++l) s += y->A[i * Dk + l] * x->A[l * Dk + j];
            out->A[i * Dk + j] = s;
        }
        for (int64_t j = 0; j < Dv; ++j) {
            double s = y->M[i * Dv + j];
            for (int64_t l = 0; l < Dk; ++l) s += y->A[i * Dk + l] * x->M[l * Dv + j];
            out->M[i * Dv + j] = s;
        }
    }
}

static void amap_copy(int64_t Dk, int64_t Dv, const amap_t* x, amap_t* out) {
    memcpy(out->A, x->A, sizeof(double) * Dk * Dk);
    memcpy(out->M, x->M, sizeof(double) * Dk * Dv);
}

int gdn_oracle_forward_monoid(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk,
                              int64_t Dv, int64_t seg_len, const double* q, const double* k,
                              const double* v, const double* a, const double* b,
                              const double* A_log, const double* dt_bias, const double* state0,
                              const uint8_t* mask, double* o, double* state_T) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    if (seg_len < 1) return 1;
    double *lg, *bt;
    if (gates_ab(&d, a, b, A_log, dt_bias, &lg, &bt)) return 3;
    const int64_t nseg = T > 0 ? (T + seg_len - 1) / seg_len : 0;
    int64_t npad = 1;
    while (npad < nseg) npad *= 2;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pr = 0; pr < B * Hv; ++pr) {
        const int64_t bb = pr / Hv, h = pr % Hv;
        amap_t* x = calloc((size_t)npad, sizeof(amap_t));
        amap_t tmpm;
        double* pool = malloc(sizeof(double) * (size_t)(npad + 1) * (Dk * Dk + Dk * Dv));
        double* qh = malloc(sizeof(double) * Dk);
        double* kh = malloc(sizeof(double) * Dk);
        double* w = malloc(sizeof(double) * (Dk > Dv ? Dk : Dv));
        double* p = malloc(sizeof(double) * Dv);
        double* dl = malloc(sizeof(double) * Dv);
        double* S = malloc(sizeof(double) * Dk * Dv);
        if (!x || !pool || !qh || !kh || !w || !p || !dl || !S) {
#pragma omp atomic write
            fail = 3;
        } else {
            for (int64_t i = 0; i <= npad; ++i) {
                amap_t* m = i < npad ? &x[i] : &tmpm;
                m->A = pool + i * (Dk * Dk + Dk * Dv);
                m->M = m->A + Dk * Dk;
                amap_identity(Dk, Dv, m);
            }
            /* each run's map, composed step by step: (A, M) <- (A_t A, A_t M + M_t) */
            for (int64_t s = 0; s < nseg; ++s) {
                for (int64_t t = s * seg_len; t < T && t < (s + 1) * seg_len; ++t) {
                    if (mask && !mask[bb * T + t]) continue;
                    load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                    const double g = exp(lg[IG(&d, bb, t, h)]), beta = bt[IG(&d, bb, t, h)];
                    step_linear(Dk, Dk, x[s].A, g, beta, kh, w);
                    step_linear(Dk, Dv, x[s].M, g, beta, kh, w);
                    const double* vt = v + IV(&d, bb, t, h);
                    for (int64_t r = 0; r < Dk; ++r)
                        for (int64_t c = 0; c < Dv; ++c) x[s].M[r * Dv + c] += beta * kh[r] * vt[c];
                }
            }
            /* exclusive prefix: up-sweep, then down-sweep from the identity */
            for (int64_t st = 1; st < npad; st *= 2)
                for (int64_t i = 2 * st - 1; i < npad; i += 2 * st) {
                    amap_then(Dk, Dv, &x[i - st], &x[i], &tmpm);
                    amap_copy(Dk, Dv, &tmpm, &x[i]);
                }
            amap_identity(Dk, Dv, &x[npad - 1]);
            for (int64_t st = npad / 2; st >= 1; st /= 2)
                for (int64_t i = 2 * st - 1; i < npad; i += 2 * st) {
                    /* left child <- the parent's prefix; right child <- the parent's
                     * prefix followed by the left subtree's total */
                    amap_then(Dk, Dv, &x[i], &x[i - st], &tmpm);
                    amap_copy(Dk, Dv, &x[i], &x[i - st]);
                    amap_copy(Dk, Dv, &tmpm, &x[i]);
                }
            /* replay each run from prefix(state0) */
            const double* S0 = state0 ? state0 + IS(&d, bb, h) : NULL;
            for (int64_t s = 0; s < nseg; ++s) {
                for (int64_t r = 0; r < Dk; ++r)
                    for (int64_t c = 0; c < Dv; ++c) {
                        double acc = x[s].M[r * Dv + c];
                        if (S0)
                            for (int64_t l = 0; l < Dk; ++l) acc += x[s].A[r * Dk + l] * S0[l * Dv + c];
                        S[r * Dv + c] = acc;
                    }
                for (int64_t t = s * seg_len; t < T && t < (s + 1) * seg_len; ++t) {
                    load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                    if (!mask || mask[bb * T + t]) {
                        const double g = exp(lg[IG(&d, bb, t, h)]), beta = bt[IG(&d, bb, t, h)];
                        apply_step(Dk, Dv, S, g, beta, kh, v + IV(&d, bb, t, h), p, dl);
                    }
                    read_out(Dk, Dv, S, qh, o + IV(&d, bb, t, h));
                }
            }
            if (nseg > 0)
                memcpy(state_T + IS(&d, bb, h), S, sizeof(double) * Dk * Dv);
            else if (S0)
                memcpy(state_T + IS(&d, bb, h), S0, sizeof(double) * Dk * Dv);
            else
                memset(state_T + IS(&d, bb, h), 0, sizeof(double) * Dk * Dv);
        }
        free(x); free(pool); free(qh); free(kh); free(w); free(p); free(dl); free(S);
    }
    free(lg); free(bt);
    return fail;
}

/* ---- sequential VJP ------------------------------------------------------ */
/*
 * Reverse-mode derivative of the sequential recurrence, per (b, h).  For an
 * applied step with previous state S_prev:
 *     S_a = g S_prev,  p = S_a^T k,  delta = beta (v - p),
 *     S   = S_a + k delta^T,  o = S^T q.
 * With Sbar = dL/dS (from later steps) and obar = dL/do:
 *     Sbar  += q obar^T;          qbar  = S obar
 *     kbar   = Sbar delta;        dbar  = Sbar^T k
 *     vbar   = beta dbar;         betabar = <dbar, v - p>;   pbar = -beta dbar
 *     Sbar_a = Sbar + k pbar^T;   kbar += S_a pbar
 *     gbar   = <Sbar_a, S_prev>;  Sbar_prev = g Sbar_a;       lbar = gbar g
 * A masked step only adds q obar^T to Sbar and gives qbar = S obar.
 * Then, outside the (b, h) loop, in a fixed order:
 *   - GQA: dqhat / dkhat of key head j = sum over its G value heads (ascending h)
 *   - L2 norm: xhat = s x / n, n = sqrt(|x|^2 + eps):
 *         dx = (s / n) (xhatbar - u <u, xhatbar>),  u = x / n
 *     (s = 1/sqrt(Dk) for q, 1 for k; written without n^2 or n^3 terms)
 *   - gates: da = lbar * (-exp(A_log)) * softplus'(a + dt_bias);
 *            db = betabar * beta (1 - beta);
 *            dA_log[h] = sum_{b,t} lbar * l;  ddt_bias[h] = sum_{b,t} da
 */
/* After the per-(b, h) reverse passes: zero dv on masked steps, then the GQA
 * sum and the L2-norm backward of q and k (see the comment above
 * backward_core), per (b, t, key head) in a fixed order. */
static void qk_finish(const dims_t* dd, const double* q, const double* k, const uint8_t* mask,
                      const double* dqh, const double* dkh, double* dq, double* dk, double* dv) {
    const dims_t d = *dd;
    const int64_t B = d.B, T = d.T, Hk = d.Hk, Hv = d.Hv, Dk = d.Dk, Dv = d.Dv;
    int64_t G = Hv / Hk;
    /* v gradient is zero on masked steps */
    if (mask)
        for (int64_t bb = 0; bb < B; ++bb)
            for (int64_t t = 0; t < T; ++t)
                if (!mask[bb * T + t])
                    for (int64_t h = 0; h < Hv; ++h)
                        memset(dv + IV(&d, bb, t, h), 0, sizeof(double) * Dv);
    /* GQA sum + L2-norm backward, per (b, t, key head) */
    double* acc = malloc(sizeof(double) * Dk);
    double sq = 1.0 / sqrt((double)Dk);
    for (int64_t bb = 0; bb < B; ++bb)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t j = 0; j < Hk; ++j) {
                for (int pass = 0; pass < 2; ++pass) {
                    const double* x = (pass == 0 ? q : k) + IQK(&d, bb, t, j);
                    const double* src = pass == 0 ? dqh : dkh;
                    double* dst = (pass == 0 ? dq : dk) + IQK(&d, bb, t, j);
                    double s = pass == 0 ? sq : 1.0;
                    for (int64_t r = 0; r < Dk; ++r) acc[r] = 0.0;
                    for (int64_t h = j * G; h < (j + 1) * G; ++h) {
                        const double* y = src + ((bb * T + t) * Hv + h) * Dk;
                        for (int64_t r = 0; r < Dk; ++r) acc[r] += y[r];
                    }
                    double rn = inv_norm(x, Dk); /* 1/n */
                    double uy = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) uy += x[r] * rn * acc[r];
                    for (int64_t r = 0; r < Dk; ++r) dst[r] = s * rn * (acc[r] - x[r] * rn * uy);
                }
            }
    free(acc);
}

/* The VJP up to the gates: dq, dk, dv, dstate0 and the per-step cotangents
 * dlg of l = log g and dbt of beta ([B, T, Hv], zero on masked steps). */
static int backward_core(const dims_t* dd, const double* q, const double* k, const double* v,
                         const double* lg, const double* bt, const double* state0,
                         const uint8_t* mask, const double* d_o, const double* d_state_T,
                         double* dq, double* dk, double* dv, double* dlg, double* dbt,
                         double* dstate0) {
    const dims_t d = *dd;
    const int64_t B = d.B, T = d.T, Hv = d.Hv, Dk = d.Dk, Dv = d.Dv;
    int64_t SS = Dk * Dv;
    int64_t nseg = (T + SEGMENT - 1) / SEGMENT;
    /* per value head gradients of the normalised q / k */
    double* dqh = calloc((size_t)(B * T * Hv * Dk > 0 ? B * T * Hv * Dk : 1), sizeof(double));
    double* dkh = calloc((size_t)(B * T * Hv * Dk > 0 ? B * T * Hv * Dk : 1), sizeof(double));
    if (!dqh || !dkh) { free(dqh); free(dkh); return 3; }
    memset(dlg, 0, sizeof(double) * B * T * Hv);
    memset(dbt, 0, sizeof(double) * B * T * Hv);
    int64_t npairs = B * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pr = 0; pr < npairs; ++pr) {
        int64_t bb = pr / Hv, h = pr % Hv;
        /* states at segment starts */
        double* seg = malloc(sizeof(double) * SS * (nseg > 0 ? nseg : 1));
        /* states after every step of one segment (index 0 = segment start) */
        double* hist = malloc(sizeof(double) * SS * (SEGMENT + 1));
        double* Sb = malloc(sizeof(double) * SS);
        double* Sa = malloc(sizeof(double) * SS);
        double* qh = malloc(sizeof(double) * Dk);
        double* kh = malloc(sizeof(double) * Dk);
        double* p = malloc(sizeof(double) * Dv);
        double* dl = malloc(sizeof(double) * Dv);
        double* dbar = malloc(sizeof(double) * Dv);
        double* pbar = malloc(sizeof(double) * Dv);
        double* S = malloc(sizeof(double) * SS);
        if (state0)
            memcpy(S, state0 + IS(&d, bb, h), sizeof(double) * SS);
        else
            memset(S, 0, sizeof(double) * SS);
        /* forward pass, keeping only segment-start states */
        for (int64_t t = 0; t < T; ++t) {
            if (t % SEGMENT == 0) memcpy(seg + (t / SEGMENT) * SS, S, sizeof(double) * SS);
            int on = mask ? (mask[bb * T + t] != 0) : 1;
            if (on) {
                load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                double g = exp(lg[IG(&d, bb, t, h)]);
                double beta = bt[IG(&d, bb, t, h)];
                apply_step(Dk, Dv, S, g, beta, kh, v + IV(&d, bb, t, h), p, dl);
            }
        }
        /* seed: dL/dS_T */
        if (d_state_T)
            memcpy(Sb, d_state_T + IS(&d, bb, h), sizeof(double) * SS);
        else
            memset(Sb, 0, sizeof(double) * SS);
        for (int64_t sg = nseg - 1; sg >= 0; --sg) {
            int64_t t0 = sg * SEGMENT;
            int64_t L = (T - t0) < SEGMENT ? (T - t0) : SEGMENT;
            /* recompute states of this segment */
            memcpy(hist, seg + sg * SS, sizeof(double) * SS);
            for (int64_t i = 0; i < L; ++i) {
                int64_t t = t0 + i;
                double* Sn = hist + (i + 1) * SS;
                memcpy(Sn, hist + i * SS, sizeof(double) * SS);
                int on = mask ? (mask[bb * T + t] != 0) : 1;
                if (on) {
                    load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                    double g = exp(lg[IG(&d, bb, t, h)]);
                    double beta = bt[IG(&d, bb, t, h)];
                    apply_step(Dk, Dv, Sn, g, beta, kh, v + IV(&d, bb, t, h), p, dl);
                }
            }
            /* reverse steps */
            for (int64_t i = L - 1; i >= 0; --i) {
                int64_t t = t0 + i;
                const double* Sprev = hist + i * SS;
                const double* Scur = hist + (i + 1) * SS;
                const double* ob = d_o + IV(&d, bb, t, h);
                double* qbar = dqh + ((bb * T + t) * Hv + h) * Dk;
                double* kbar = dkh + ((bb * T + t) * Hv + h) * Dk;
                load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                /* o = S^T q */
                for (int64_t r = 0; r < Dk; ++r) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) {
                        Sb[r * Dv + c] += qh[r] * ob[c];
                        acc += Scur[r * Dv + c] * ob[c];
                    }
                    qbar[r] = acc;
                }
                int on = mask ? (mask[bb * T + t] != 0) : 1;
                if (!on) continue;
                double g = exp(lg[IG(&d, bb, t, h)]);
                double beta = bt[IG(&d, bb, t, h)];
                const double* vt = v + IV(&d, bb, t, h);
                /* S_a = g S_prev, p = S_a^T k, delta = beta (v - p) */
                for (int64_t x = 0; x < SS; ++x) Sa[x] = g * Sprev[x];
                for (int64_t c = 0; c < Dv; ++c) p[c] = 0.0;
                for (int64_t r = 0; r < Dk; ++r)
                    for (int64_t c = 0; c < Dv; ++c) p[c] += Sa[r * Dv + c] * kh[r];
                for (int64_t c = 0; c < Dv; ++c) dl[c] = beta * (vt[c] - p[c]);
                /* S = S_a + k delta^T */
                for (int64_t r = 0; r < Dk; ++r) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) acc += Sb[r * Dv + c] * dl[c];
                    kbar[r] = acc;
                }
                for (int64_t c = 0; c < Dv; ++c) {
                    double acc = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) acc += Sb[r * Dv + c] * kh[r];
                    dbar[c] = acc;
                }
                /* delta = beta (v - p) */
                double betabar = 0.0;
                double* vbar = dv + IV(&d, bb, t, h);
                for (int64_t c = 0; c < Dv; ++c) {
                    vbar[c] = beta * dbar[c];
                    betabar += dbar[c] * (vt[c] - p[c]);
                    pbar[c] = -beta * dbar[c];
                }
                /* p = S_a^T k */
                for (int64_t r = 0; r < Dk; ++r) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) {
                        Sb[r * Dv + c] += kh[r] * pbar[c];
                        acc += Sa[r * Dv + c] * pbar[c];
                    }
                    kbar[r] += acc;
                }
                /* S_a = g S_prev */
                double gbar = 0.0;
                for (int64_t x = 0; x < SS; ++x) gbar += Sb[x] * Sprev[x];
                for (int64_t x = 0; x < SS; ++x) Sb[x] *= g;
                dlg[IG(&d, bb, t, h)] = gbar * g;
                dbt[IG(&d, bb, t, h)] = betabar;
            }
        }
        memcpy(dstate0 + IS(&d, bb, h), Sb, sizeof(double) * SS);
        free(seg); free(hist); free(Sb); free(Sa); free(qh); free(kh);
        free(p); free(dl); free(dbar); free(pbar); free(S);
    }
    qk_finish(&d, q, k, mask, dqh, dkh, dq, dk, dv);
    free(dqh); free(dkh);
    return 0;
}

int gdn_oracle_backward(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                        const double* q, const double* k, const double* v, const double* a,
                        const double* b, const double* A_log, const double* dt_bias,
                        const double* state0, const uint8_t* mask, const double* d_o,
                        const double* d_state_T, double* dq, double* dk, double* dv,
                        double* da, double* db, double* dA_log, double* ddt_bias,
                        double* dstate0) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    double *lg, *bt;
    if (gates_ab(&d, a, b, A_log, dt_bias, &lg, &bt)) return 3;
    double* dlg = malloc(sizeof(double) * (B * T * Hv > 0 ? B * T * Hv : 1));
    double* dbt = malloc(sizeof(double) * (B * T * Hv > 0 ? B * T * Hv : 1));
    if (!dlg || !dbt) { free(lg); free(bt); free(dlg); free(dbt); return 3; }
    rc = backward_core(&d, q, k, v, lg, bt, state0, mask, d_o, d_state_T, dq, dk, dv, dlg, dbt,
                       dstate0);
    if (rc) { free(lg); free(bt); free(dlg); free(dbt); return rc; }
    /* gates and per-head sums (fixed order: b, then t) */
    for (int64_t h = 0; h < Hv; ++h) {
        double sA = 0.0, sdt = 0.0;
        for (int64_t bb = 0; bb < B; ++bb)
            for (int64_t t = 0; t < T; ++t) {
                int64_t ix = IG(&d, bb, t, h);
                int on = mask ? (mask[bb * T + t] != 0) : 1;
                if (!on) { da[ix] = 0.0; db[ix] = 0.0; continue; }
                double x = a[ix] + dt_bias[h];
                double lgv = log_decay(a[ix], A_log[h], dt_bias[h]);
                double dx = dlg[ix] * (-exp(A_log[h])) * softplus_clamped_grad(x);
                double beta = sigmoid_d(b[ix]);
                da[ix] = dx;
                db[ix] = dbt[ix] * beta * (1.0 - beta);
                sA += dlg[ix] * lgv;
                sdt += dx;
            }
        dA_log[h] = sA;
        ddt_bias[h] = sdt;
    }
    free(lg); free(bt); free(dlg); free(dbt);
    return 0;
}

/* log_decay / beta form: returns d_log_decay and d_beta ([B, T, Hv], zero on
 * masked steps) in place of the gate-parameter cotangents */
int gdn_oracle_backward_lb(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                           const double* q, const double* k, const double* v,
                           const double* log_decay_, const double* beta, const double* state0,
                           const uint8_t* mask, const double* d_o, const double* d_state_T,
                           double* dq, double* dk, double* dv, double* d_log_decay,
                           double* d_beta, double* dstate0) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    return backward_core(&d, q, k, v, log_decay_, beta, state0, mask, d_o, d_state_T, dq, dk,
                         dv, d_log_decay, d_beta, dstate0);
}

/* ---- per-key-channel gates ------------------------------------------------
 * The vectorised gating the mlx-lm page lists (g.ndim == 4: one decay per key
 * channel), in the op contract's log_decay form extended by the key-channel
 * axis: log_decay [B, T, Hv, Dk] holds l_{t,i} = log g_{t,i}, beta [B, T, Hv].
 * An applied step scales row i of S (key channel i) by g_{t,i}:
 *     S_a = diag(g) S_prev,  p = S_a^T k,  delta = beta (v - p),  S = S_a + k delta^T,
 * and its VJP is the scalar one above with diag(g) in place of g:
 *     Sbar_prev = diag(g) Sbar_a,   lbar_i = g_i sum_c Sbar_a[i, c] S_prev[i, c].
 * Written apart from the scalar path (not through it), so that with equal
 * channels the two agree only through the mathematics. */
#define IGK(d, b, t, h) ((((b) * (d)->T + (t)) * (d)->Hv + (h)) * (d)->Dk)

static void apply_step_kc(int64_t Dk, int64_t Dv, double* S, const double* g, double beta,
                          const double* kh, const double* v, double* p, double* dl) {
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < Dv; ++c) S[r * Dv + c] *= g[r];
    for (int64_t c = 0; c < Dv; ++c) p[c] = 0.0;
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < Dv; ++c) p[c] += S[r * Dv + c] * kh[r];
    for (int64_t c = 0; c < Dv; ++c) dl[c] = beta * (v[c] - p[c]);
    for (int64_t r = 0; r < Dk; ++r)
        for (int64_t c = 0; c < Dv; ++c) S[r * Dv + c] += kh[r] * dl[c];
}

int gdn_oracle_forward_kc(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                          const double* q, const double* k, const double* v,
                          const double* log_decay_, const double* beta, const double* state0,
                          const uint8_t* mask, double* o, double* state_T) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    int64_t npairs = B * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pr = 0; pr < npairs; ++pr) {
        int64_t bb = pr / Hv, h = pr % Hv;
        double* S = state_T + IS(&d, bb, h);
        if (state0)
            memcpy(S, state0 + IS(&d, bb, h), sizeof(double) * Dk * Dv);
        else
            memset(S, 0, sizeof(double) * Dk * Dv);
        double* qh = malloc(sizeof(double) * Dk);
        double* kh = malloc(sizeof(double) * Dk);
        double* g = malloc(sizeof(double) * Dk);
        double* p = malloc(sizeof(double) * Dv);
        double* dl = malloc(sizeof(double) * Dv);
        for (int64_t t = 0; t < T; ++t) {
            load_qk_hat(&d, q, k, bb, t, h, qh, kh);
            int on = mask ? (mask[bb * T + t] != 0) : 1;
            if (on) {
                for (int64_t r = 0; r < Dk; ++r) g[r] = exp(log_decay_[IGK(&d, bb, t, h) + r]);
                apply_step_kc(Dk, Dv, S, g, beta[IG(&d, bb, t, h)], kh, v + IV(&d, bb, t, h), p, dl);
            }
            read_out(Dk, Dv, S, qh, o + IV(&d, bb, t, h));
        }
        free(qh); free(kh); free(g); free(p); free(dl);
    }
    return 0;
}

/* d_log_decay [B, T, Hv, Dk] and d_beta [B, T, Hv] (zero on masked steps), with
 * dq, dk, dv and dstate0 as in gdn_oracle_backward. */
int gdn_oracle_backward_kc(int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                           const double* q, const double* k, const double* v,
                           const double* log_decay_, const double* beta_, const double* state0,
                           const uint8_t* mask, const double* d_o, const double* d_state_T,
                           double* dq, double* dk, double* dv, double* d_log_decay,
                           double* d_beta, double* dstate0) {
    dims_t d = {B, T, Hk, Hv, Dk, Dv};
    int rc = check_dims(&d);
    if (rc) return rc;
    int64_t SS = Dk * Dv;
    int64_t nseg = (T + SEGMENT - 1) / SEGMENT;
    double* dqh = calloc((size_t)(B * T * Hv * Dk > 0 ? B * T * Hv * Dk : 1), sizeof(double));
    double* dkh = calloc((size_t)(B * T * Hv * Dk > 0 ? B * T * Hv * Dk : 1), sizeof(double));
    if (!dqh || !dkh) { free(dqh); free(dkh); return 3; }
    memset(d_log_decay, 0, sizeof(double) * B * T * Hv * Dk);
    memset(d_beta, 0, sizeof(double) * B * T * Hv);
    int64_t npairs = B * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pr = 0; pr < npairs; ++pr) {
        int64_t bb = pr / Hv, h = pr % Hv;
        double* seg = malloc(sizeof(double) * SS * (nseg > 0 ? nseg : 1));
        double* hist = malloc(sizeof(double) * SS * (SEGMENT + 1));
        double* Sb = malloc(sizeof(double) * SS);
        double* Sa = malloc(sizeof(double) * SS);
        double* S = malloc(sizeof(double) * SS);
        double* qh = malloc(sizeof(double) * Dk);
        double* kh = malloc(sizeof(double) * Dk);
        double* g = malloc(sizeof(double) * Dk);
        double* p = malloc(sizeof(double) * Dv);
        double* dl = malloc(sizeof(double) * Dv);
        double* dbar = malloc(sizeof(double) * Dv);
        double* pbar = malloc(sizeof(double) * Dv);
        if (state0)
            memcpy(S, state0 + IS(&d, bb, h), sizeof(double) * SS);
        else
            memset(S, 0, sizeof(double) * SS);
        for (int64_t t = 0; t < T; ++t) {  /* segment-start states */
            if (t % SEGMENT == 0) memcpy(seg + (t / SEGMENT) * SS, S, sizeof(double) * SS);
            if (mask && !mask[bb * T + t]) continue;
            load_qk_hat(&d, q, k, bb, t, h, qh, kh);
            for (int64_t r = 0; r < Dk; ++r) g[r] = exp(log_decay_[IGK(&d, bb, t, h) + r]);
            apply_step_kc(Dk, Dv, S, g, beta_[IG(&d, bb, t, h)], kh, v + IV(&d, bb, t, h), p, dl);
        }
        if (d_state_T)
            memcpy(Sb, d_state_T + IS(&d, bb, h), sizeof(double) * SS);
        else
            memset(Sb, 0, sizeof(double) * SS);
        for (int64_t sg = nseg - 1; sg >= 0; --sg) {
            int64_t t0 = sg * SEGMENT;
            int64_t L = (T - t0) < SEGMENT ? (T - t0) : SEGMENT;
            memcpy(hist, seg + sg * SS, sizeof(double) * SS);
            for (int64_t i = 0; i < L; ++i) {
                int64_t t = t0 + i;
                double* Sn = hist + (i + 1) * SS;
                memcpy(Sn, hist + i * SS, sizeof(double) * SS);
                if (mask && !mask[bb * T + t]) continue;
                load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                for (int64_t r = 0; r < Dk; ++r) g[r] = exp(log_decay_[IGK(&d, bb, t, h) + r]);
                apply_step_kc(Dk, Dv, Sn, g, beta_[IG(&d, bb, t, h)], kh, v + IV(&d, bb, t, h), p, dl);
            }
            for (int64_t i = L - 1; i >= 0; --i) {
                int64_t t = t0 + i;
                const double* Sprev = hist + i * SS;
                const double* Scur = hist + (i + 1) * SS;
                const double* ob = d_o + IV(&d, bb, t, h);
                double* qbar = dqh + ((bb * T + t) * Hv + h) * Dk;
                double* kbar = dkh + ((bb * T + t) * Hv + h) * Dk;
                load_qk_hat(&d, q, k, bb, t, h, qh, kh);
                for (int64_t r = 0; r < Dk; ++r) {  /* o = S^T q */
                    double acc = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) {
                        Sb[r * Dv + c] += qh[r] * ob[c];
                        acc += Scur[r * Dv + c] * ob[c];
                    }
                    qbar[r] = acc;
                }
                if (mask && !mask[bb * T + t]) continue;
                double beta = beta_[IG(&d, bb, t, h)];
                const double* vt = v + IV(&d, bb, t, h);
                for (int64_t r = 0; r < Dk; ++r) g[r] = exp(log_decay_[IGK(&d, bb, t, h) + r]);
                /* S_a = diag(g) S_prev, p = S_a^T k, delta = beta (v - p) */
                for (int64_t r = 0; r < Dk; ++r)
                    for (int64_t c = 0; c < Dv; ++c) Sa[r * Dv + c] = g[r] * Sprev[r * Dv + c];
                for (int64_t c = 0; c < Dv; ++c) p[c] = 0.0;
                for (int64_t r = 0; r < Dk; ++r)
                    for (int64_t c = 0; c < Dv; ++c) p[c] += Sa[r * Dv + c] * kh[r];
                for (int64_t c = 0; c < Dv; ++c) dl[c] = beta * (vt[c] - p[c]);
                /* S = S_a + k delta^T */
                for (int64_t r = 0; r < Dk; ++r) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) acc += Sb[r * Dv + c] * dl[c];
                    kbar[r] = acc;
                }
                for (int64_t c = 0; c < Dv; ++c) {
                    double acc = 0.0;
                    for (int64_t r = 0; r < Dk; ++r) acc += Sb[r * Dv + c] * kh[r];
                    dbar[c] = acc;
                }
                /* delta = beta (v - p) */
                double betabar = 0.0;
                double* vbar = dv + IV(&d, bb, t, h);
                for (int64_t c = 0; c < Dv; ++c) {
                    vbar[c] = beta * dbar[c];
                    betabar += dbar[c] * (vt[c] - p[c]);
                    pbar[c] = -beta * dbar[c];
                }
                /* p = S_a^T k */
                for (int64_t r = 0; r < Dk; ++r) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) {
                        Sb[r * Dv + c] += kh[r] * pbar[c];
                        acc += Sa[r * Dv + c] * pbar[c];
                    }
                    kbar[r] += acc;
                }
                /* S_a = diag(g) S_prev: one log-decay cotangent per key channel */
                double* lbar = d_log_decay + IGK(&d, bb, t, h);
                for (int64_t r = 0; r < Dk; ++r) {
                    double gb = 0.0;
                    for (int64_t c = 0; c < Dv; ++c) gb += Sb[r * Dv + c] * Sprev[r * Dv + c];
                    lbar[r] = gb * g[r];
                    for (int64_t c = 0; c < Dv; ++c) Sb[r * Dv + c] *= g[r];
                }
                d_beta[IG(&d, bb, t, h)] = betabar;
            }
        }
        memcpy(dstate0 + IS(&d, bb, h), Sb, sizeof(double) * SS);
        free(seg); free(hist); free(Sb); free(Sa); free(S); free(qh); free(kh); free(g);
        free(p); free(dl); free(dbar); free(pbar);
    }
    qk_finish(&d, q, k, mask, dqh, dkh, dq, dk, dv);
    free(dqh); free(dkh);
    return 0;
}

/* ---- causal conv1d update ------------------------------------------------ */

int gdn_oracle_causal_conv1d_update(int64_t B, int64_t C, int64_t S, int64_t K,
                                    const double* hidden, const double* conv_state,
                                    const double* weight, double* out, double* final_state) {
    if (B < 1 || C < 1 || S < 0 || K < 1) return 1;
    double* x = malloc(sizeof(double) * (size_t)(K + S));
    if (!x) return 3;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t c = 0; c < C; ++c) {
            const int64_t bc = b * C + c;
            for (int64_t i = 0; i < K; ++i) x[i] = conv_state[bc * K + i];
            for (int64_t t = 0; t < S; ++t) x[K + t] = hidden[bc * S + t];
            for (int64_t t = 0; t < S; ++t) {
                double acc = 0.0;
                for (int64_t i = 0; i < K; ++i) acc += weight[c * K + i] * x[t + 1 + i];
                out[bc * S + t] = acc / (1.0 + exp(-acc));
            }
            for (int64_t i = 0; i < K; ++i) final_state[bc * K + i] = x[S + i];
        }
    free(x);
    return 0;
}

/* ---- threads the OpenMP runtime will use --------------------------------- */

int gdn_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
