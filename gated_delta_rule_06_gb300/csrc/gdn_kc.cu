// gdn_kc.cu -- the recurrence with one decay per key channel (the vectorised
// gating the mlx-lm page lists as g.ndim == 4 and leaves to a follow-up), on the
// CUDA cores with an fp32 state.
//
// Gates: log_decay [B, T, Hv, Dk] (l_{t,i} = log g_{t,i}, key channel i) and
// beta [B, T, Hv].  An applied step of (b, h) (torch-to-nnef page, op contract,
// with diag(g) in place of the scalar g):
//     S_a = diag(g_t) S,  p = S_a^T kh_t,  delta = beta_t (v_t - p),
//     S = S_a + kh_t delta^T,  o_t = S^T qh_t
// (a masked step leaves S unchanged and reads o_t = S^T qh_t).  Its VJP is the
// scalar one with diag(g): Sbar_prev = diag(g) Sbar_a and
// lbar_i = g_i sum_c Sbar_a[i, c] S_prev[i, c].
//
// The columns of S evolve independently, so a CTA owns a tile of KT = 16 value
// columns of one (b, h): 256 threads, thread (row group rg, column jj) keeps rows
// rg R .. rg R + R - 1 (R = Dk / 16) of its column in registers.  Sums over the
// rows of a column go through a shuffle and shared memory in a fixed order; sums
// over the 16 columns of a row (the backward's q, k and gate cotangents) through
// shuffles, per tile, into partials that later kernels add in tile order.
//   forward:  sequential over t; the state at every kSeg-th step is kept
//             (checkpoints [B, Hv, ceil(T / kSeg), Dk, Dv]) for the backward.
//   backward: reverse over the kSeg-step segments: the segment's states are
//             recomputed from its checkpoint into shared memory, then walked back.
// The q / k cotangent partials of the tiles are written as if each (h, tile) were
// its own value head, so the reduction kernel of gdn_bwd.cu (GQA sum and L2-norm
// backward) finishes them with G Dv / 16 heads per key head.
#include "gdn_internal.cuh"

namespace gdn {

namespace {

constexpr int KT = 16;             // value columns per CTA
constexpr int KG = 16;             // Dk <= KG kMaxR
constexpr int kThreads = KT * KG;  // 256
constexpr int kSeg = 8;            // steps between checkpoints
constexpr int kMaxR = 16;          // rows per thread (Dk <= 256)

struct KcArgs {
    const void* lg;      // log_decay [B, T, Hv, Dk]
    const void* beta;    // [B, T, Hv]
    float* ckpt;         // [B, Hv, NS, Dk, Dv]
    float* gpart;        // [B, Hv nt, Tp, Dk] per-tile log-decay cotangents
    float* bpart;        // [B, Hv nt, Tp] per-tile beta cotangents
    void* d_lg;          // [B, T, Hv, Dk]
    void* d_beta;        // [B, T, Hv]
};

// Per-step vectors of steps t0 .. t0 + L - 1 of (b, h) into shared memory: the
// normalised k and q rows, g per key channel, beta, the applied flag, the tile's
// v columns and (ob non-null) its d_o columns.  NB steps at a time, every global
// load of a batch issued before its first store, so a batch pays one load
// latency, not one per step (NB trades that against registers).
template <typename TI, int NB>
__device__ __forceinline__ void load_seg(const Dims& d, const Ptrs& p, const KcArgs& a,
                                         int64_t bb, int64_t h, int64_t t0, int L, int col0,
                                         float* kh, float* qh, float* g, float* v, float* ob,
                                         float* bt, int* on) {
    const int tid = threadIdx.x;
    const int64_t j = h / d.G;
    const int Dk = (int)d.Dk;
#pragma unroll 1
    for (int i0 = 0; i0 < L; i0 += NB) {
        float xk[NB], xq[NB], xg[NB], nk[NB], nq[NB], xv[NB], xo[NB], xb[NB];
        bool live[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int i = i0 + u;
            const int64_t t = t0 + i;
            const bool in = i < L;
            live[u] = in && (p.mask == nullptr || p.mask[bb * d.T + t] != 0);
            xk[u] = xq[u] = nk[u] = nq[u] = xv[u] = xo[u] = xb[u] = xg[u] = 0.f;
            if (in && tid < Dk) {
                const int64_t xi = ((bb * d.T + t) * d.Hk + j) * Dk + tid;
                const int64_t ri = (bb * d.Hk + j) * d.Tp + t;
                xk[u] = ldf((const TI*)p.k + xi);
                xq[u] = ldf((const TI*)p.q + xi);
                nk[u] = p.rk[ri];
                nq[u] = p.rq[ri];
                xg[u] = ldf((const TI*)a.lg + ((bb * d.T + t) * d.Hv + h) * Dk + tid);
            }
            if (in && tid < KT) {
                const int64_t vi = ((bb * d.T + t) * d.Hv + h) * d.Dv + col0 + tid;
                xv[u] = ldf((const TI*)p.v + vi);
                if (ob) xo[u] = ldf((const TI*)p.d_o + vi);
            }
            if (in && tid == 0) xb[u] = ldf((const TI*)a.beta + (bb * d.T + t) * d.Hv + h);
        }
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int i = i0 + u;
            if (i >= L) break;
            if (tid < Dk) {
                kh[i * Dk + tid] = xk[u] * nk[u];
                qh[i * Dk + tid] = xq[u] * nq[u] * rsqrtf((float)Dk);
                g[i * Dk + tid] = live[u] ? expf(xg[u]) : 1.f;
            }
            if (tid < KT) {
                v[i * KT + tid] = xv[u];
                if (ob) ob[i * KT + tid] = xo[u];
            }
            if (tid == 0) {
                bt[i] = live[u] ? xb[u] : 0.f;
                on[i] = live[u] ? 1 : 0;
            }
        }
    }
}

// sum over the 32 lanes of a warp (fixed xor tree)
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Forward: warp w owns columns col0 + 2 w, + 1 of the tile; lane l owns rows
// l, l + 32, ... (RR = Dk / 32 of them), so every per-step sum is a warp
// shuffle and the steps need no CTA barrier (only the segment staging does).
template <typename TI>
__global__ void __launch_bounds__(kThreads, 4) kc_fwd_kernel(Dims d, Ptrs p, KcArgs a) {
    extern __shared__ __align__(16) float kcf[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv, RR = Dk / 32;
    float* kh = kcf;                  // [kSeg][Dk]
    float* qh = kh + kSeg * Dk;       // [kSeg][Dk]
    float* gv = qh + kSeg * Dk;       // [kSeg][Dk]
    float* vv = gv + kSeg * Dk;       // [kSeg][KT]
    float* bt = vv + kSeg * KT;       // [kSeg]
    int* on = reinterpret_cast<int*>(bt + kSeg);
    const int tile = blockIdx.x;
    const int64_t h = blockIdx.y, bb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col0 = tile * KT, c0 = 2 * warp;  // the warp's columns c0, c0 + 1 of the tile
    const int64_t bh = bb * d.Hv + h;
    const int64_t NS = (d.T + kSeg - 1) / kSeg;
    float S[kMaxR / 2][2];
#pragma unroll
    for (int m = 0; m < kMaxR / 2; ++m)
#pragma unroll
        for (int c = 0; c < 2; ++c)
            S[m][c] = (m < RR && p.state0) ? p.state0[(bh * Dk + lane + 32 * m) * Dv + col0 + c0 + c] : 0.f;
    for (int64_t sg = 0; sg < NS; ++sg) {
        const int64_t t0 = sg * kSeg;
        const int L = (int)(d.T - t0 < kSeg ? d.T - t0 : kSeg);
        if (a.ckpt) {  // the state at the start of this segment
            float* ck = a.ckpt + (bh * NS + sg) * Dk * Dv + col0 + c0;
#pragma unroll
            for (int m = 0; m < kMaxR / 2; ++m)
                if (m < RR) {
                    ck[(int64_t)(lane + 32 * m) * Dv] = S[m][0];
                    ck[(int64_t)(lane + 32 * m) * Dv + 1] = S[m][1];
                }
        }
        __syncthreads();  // the previous segment's vectors have been read
        load_seg<TI, 2>(d, p, a, bb, h, t0, L, col0, kh, qh, gv, vv, nullptr, bt, on);
        __syncthreads();
        for (int i = 0; i < L; ++i) {
            const float* kk = kh + i * Dk;
            const float* gg = gv + i * Dk;
            const float* qq = qh + i * Dk;
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int m = 0; m < kMaxR / 2; ++m)
                if (m < RR) {
                    const float gk = gg[lane + 32 * m] * kk[lane + 32 * m];
                    p0 = fmaf(gk, S[m][0], p0);
                    p1 = fmaf(gk, S[m][1], p1);
                }
            p0 = warp_sum(p0);
            p1 = warp_sum(p1);
            if (on[i]) {
                const float d0 = bt[i] * (vv[i * KT + c0] - p0), d1 = bt[i] * (vv[i * KT + c0 + 1] - p1);
#pragma unroll
                for (int m = 0; m < kMaxR / 2; ++m)
                    if (m < RR) {
                        const float gi = gg[lane + 32 * m], ki = kk[lane + 32 * m];
                        S[m][0] = fmaf(ki, d0, gi * S[m][0]);
                        S[m][1] = fmaf(ki, d1, gi * S[m][1]);
                    }
            }
            float o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int m = 0; m < kMaxR / 2; ++m)
                if (m < RR) {
                    o0 = fmaf(S[m][0], qq[lane + 32 * m], o0);
                    o1 = fmaf(S[m][1], qq[lane + 32 * m], o1);
                }
            o0 = warp_sum(o0);
            o1 = warp_sum(o1);
            if (lane < 2) stf((TI*)p.o + ((bb * d.T + t0 + i) * d.Hv + h) * Dv + col0 + c0 + lane,
                              lane == 0 ? o0 : o1);
        }
    }
#pragma unroll
    for (int m = 0; m < kMaxR / 2; ++m)
        if (m < RR) {
            p.state_T[(bh * Dk + lane + 32 * m) * Dv + col0 + c0] = S[m][0];
            p.state_T[(bh * Dk + lane + 32 * m) * Dv + col0 + c0 + 1] = S[m][1];
        }
}

// Backward, in the forward's decomposition (warp w: columns c0 = 2 w, + 1 of the
// tile; lane l: rows l + 32 m).  Per segment (reverse order), in two halves of
// kSub steps (the later half first): the warp's states of a half are recomputed
// from the segment's checkpoint (the earlier half run through again for the
// later one) into the warp's own slice of shared memory, then walked back.
// Column sums are warp shuffles; the row sums over the tile's 16 columns (the
// q, k and log-decay cotangents) and the beta cotangent are per-warp register
// sums, added over the 8 warps in warp order through shared memory.  The tile's
// partials are written as if (h, tile) were value head h nt + tile of
// B x (Hv nt) heads.  Sized for two CTAs per SM.
constexpr int kSub = kSeg / 2;

template <typename TI>
__global__ void __launch_bounds__(kThreads, 2) kc_bwd_kernel(Dims d, Ptrs p, KcArgs a) {
    extern __shared__ __align__(16) float kcs[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv, RR = Dk / 32;
    constexpr int NW = kThreads / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* hw = kcs + warp * (kSub + 1) * 2 * Dk;     // this warp: [kSub + 1][2][Dk] states
    float* kh = kcs + NW * (kSub + 1) * 2 * Dk;       // [kSeg][Dk]
    float* qh = kh + kSeg * Dk;                       // [kSeg][Dk]
    float* gv = qh + kSeg * Dk;                       // [kSeg][Dk]
    float* vv = gv + kSeg * Dk;                       // [kSeg][KT]
    float* ob = vv + kSeg * KT;                       // [kSeg][KT] d_o
    float* bt = ob + kSeg * KT;                       // [kSeg]
    float* rowp = bt + kSeg;                          // [NW][3 Dk + 1] per-warp row sums
    int* on = reinterpret_cast<int*>(rowp + NW * (3 * Dk + 1));  // [kSeg]
    const int RP = 3 * Dk + 1;
    const int tile = blockIdx.x;
    const int64_t h = blockIdx.y, bb = blockIdx.z;
    const int col0 = tile * KT, c0 = 2 * warp;
    const int nt = Dv / KT;
    const int64_t bh = bb * d.Hv + h;
    const int64_t hv2 = bb * d.Hv * nt + h * nt + tile;  // virtual head of the partials
    const int64_t NS = (d.T + kSeg - 1) / kSeg;
    float Sb[kMaxR / 2][2];
#pragma unroll
    for (int m = 0; m < kMaxR / 2; ++m)
#pragma unroll
        for (int c = 0; c < 2; ++c)
            Sb[m][c] = (m < RR && p.d_state_T) ? p.d_state_T[(bh * Dk + lane + 32 * m) * Dv + col0 + c0 + c] : 0.f;
    for (int64_t sg = NS - 1; sg >= 0; --sg) {
        const int64_t t0 = sg * kSeg;
        const int L = (int)(d.T - t0 < kSeg ? d.T - t0 : kSeg);
        __syncthreads();  // the previous segment's shared memory is free
        load_seg<TI, 2>(d, p, a, bb, h, t0, L, col0, kh, qh, gv, vv, ob, bt, on);
        __syncthreads();
        const float* ck = a.ckpt + (bh * NS + sg) * Dk * Dv + col0 + c0;
#pragma unroll 1
        for (int half = 1; half >= 0; --half) {
            const int h0 = half * kSub;
            const int Lh = L - h0 < kSub ? L - h0 : kSub;
            if (Lh <= 0) continue;
            float S[kMaxR / 2][2];
#pragma unroll
            for (int m = 0; m < kMaxR / 2; ++m)
                if (m < RR) {
                    S[m][0] = ck[(int64_t)(lane + 32 * m) * Dv];
                    S[m][1] = ck[(int64_t)(lane + 32 * m) * Dv + 1];
                }
            float dls[kSub][2], pcs[kSub][2];
            // steps 0 .. h0 + Lh - 1 of the segment; the states of the half's steps kept
#pragma unroll 1
            for (int i = 0; i < h0 + Lh; ++i) {
                const float* kk = kh + i * Dk;
                const float* gg = gv + i * Dk;
                if (i == h0) {
#pragma unroll
                    for (int m = 0; m < kMaxR / 2; ++m)
                        if (m < RR) {
                            hw[lane + 32 * m] = S[m][0];
                            hw[Dk + lane + 32 * m] = S[m][1];
                        }
                }
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int m = 0; m < kMaxR / 2; ++m)
                    if (m < RR) {
                        const float gk = gg[lane + 32 * m] * kk[lane + 32 * m];
                        p0 = fmaf(gk, S[m][0], p0);
                        p1 = fmaf(gk, S[m][1], p1);
                    }
                p0 = warp_sum(p0);
                p1 = warp_sum(p1);
                float d0 = 0.f, d1 = 0.f;
                if (on[i]) {
                    d0 = bt[i] * (vv[i * KT + c0] - p0);
                    d1 = bt[i] * (vv[i * KT + c0 + 1] - p1);
#pragma unroll
                    for (int m = 0; m < kMaxR / 2; ++m)
                        if (m < RR) {
                            const float gi = gg[lane + 32 * m], ki = kk[lane + 32 * m];
                            S[m][0] = fmaf(ki, d0, gi * S[m][0]);
                            S[m][1] = fmaf(ki, d1, gi * S[m][1]);
                        }
                }
                if (i >= h0) {
                    const int u = i - h0;
#pragma unroll
                    for (int uu = 0; uu < kSub; ++uu)
                        if (uu == u) {
                            dls[uu][0] = d0;
                            dls[uu][1] = d1;
                            pcs[uu][0] = p0;
                            pcs[uu][1] = p1;
                        }
                    float* hs = hw + (u + 1) * 2 * Dk;
#pragma unroll
                    for (int m = 0; m < kMaxR / 2; ++m)
                        if (m < RR) {
                            hs[lane + 32 * m] = S[m][0];
                            hs[Dk + lane + 32 * m] = S[m][1];
                        }
                }
            }
            __syncwarp();  // the warp's own states (each lane rereads only its own rows)
            // reverse over the half's steps
#pragma unroll
            for (int u = kSub - 1; u >= 0; --u) {
                if (u >= Lh) continue;
                const int i = h0 + u;
                const int64_t t = t0 + i;
                const float* scur = hw + (u + 1) * 2 * Dk;
                const float* sprev = hw + u * 2 * Dk;
                const float* kk = kh + i * Dk;
                const float* gg = gv + i * Dk;
                const float* qq = qh + i * Dk;
                const float o0 = ob[i * KT + c0], o1 = ob[i * KT + c0 + 1];
                float* rp = rowp + warp * RP;
                float db0 = 0.f, db1 = 0.f;
#pragma unroll
                for (int m = 0; m < kMaxR / 2; ++m)
                    if (m < RR) {
                        const int r = lane + 32 * m;
                        Sb[m][0] = fmaf(qq[r], o0, Sb[m][0]);
                        Sb[m][1] = fmaf(qq[r], o1, Sb[m][1]);
                        rp[r] = fmaf(scur[r], o0, scur[Dk + r] * o1);  // q cotangent, this warp's columns
                        db0 = fmaf(Sb[m][0], kk[r], db0);
                        db1 = fmaf(Sb[m][1], kk[r], db1);
                    }
                if (on[i]) {
                    db0 = warp_sum(db0);
                    db1 = warp_sum(db1);
                    const float beta = bt[i];
                    if (lane < 2)
                        stf((TI*)p.dv + ((bb * d.T + t) * d.Hv + h) * Dv + col0 + c0 + lane,
                            beta * (lane == 0 ? db0 : db1));
                    const float pb0 = -beta * db0, pb1 = -beta * db1;
                    const float d0 = dls[u][0], d1 = dls[u][1];
                    if (lane == 0)
                        rp[3 * Dk] = fmaf(db0, vv[i * KT + c0] - pcs[u][0], db1 * (vv[i * KT + c0 + 1] - pcs[u][1]));
#pragma unroll
                    for (int m = 0; m < kMaxR / 2; ++m)
                        if (m < RR) {
                            const int r = lane + 32 * m;
                            const float gi = gg[r], ki = kk[r];
                            const float sp0 = sprev[r], sp1 = sprev[Dk + r];
                            rp[Dk + r] = fmaf(Sb[m][0], d0, gi * sp0 * pb0) + fmaf(Sb[m][1], d1, gi * sp1 * pb1);
                            Sb[m][0] = fmaf(ki, pb0, Sb[m][0]);  // Sbar_a
                            Sb[m][1] = fmaf(ki, pb1, Sb[m][1]);
                            rp[2 * Dk + r] = gi * fmaf(Sb[m][0], sp0, Sb[m][1] * sp1);
                            Sb[m][0] *= gi;
                            Sb[m][1] *= gi;
                        }
                } else {
                    if (lane < 2)
                        stf((TI*)p.dv + ((bb * d.T + t) * d.Hv + h) * Dv + col0 + c0 + lane, 0.f);
                    if (lane == 0) rp[3 * Dk] = 0.f;
#pragma unroll
                    for (int m = 0; m < kMaxR / 2; ++m)
                        if (m < RR) {
                            rp[Dk + lane + 32 * m] = 0.f;
                            rp[2 * Dk + lane + 32 * m] = 0.f;
                        }
                }
                __syncthreads();
                // the tile's row sums: the eight warps' in warp order
                const int64_t prow = (hv2 * d.Tp + t) * Dk;
                for (int e = tid; e < RP; e += kThreads) {
                    float x = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) x += rowp[w * RP + e];
                    if (e < Dk) p.dqh[prow + e] = x;
                    else if (e < 2 * Dk) p.dkh[prow + e - Dk] = x;
                    else if (e < 3 * Dk) a.gpart[prow + e - 2 * Dk] = x;
                    else a.bpart[hv2 * d.Tp + t] = x;
                }
                __syncthreads();  // rowp free for the next step
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kMaxR / 2; ++m)
        if (m < RR) {
            p.dstate0[(bh * Dk + lane + 32 * m) * Dv + col0 + c0] = Sb[m][0];
            p.dstate0[(bh * Dk + lane + 32 * m) * Dv + col0 + c0 + 1] = Sb[m][1];
        }
}

// d_log_decay and d_beta: the tiles' partials in tile order
template <typename TI>
__global__ void __launch_bounds__(256) kc_gate_kernel(Dims d, KcArgs a) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over (b, t, h, i)
    const int64_t n = d.B * d.T * d.Hv * d.Dk;
    if (e >= n) return;
    const int64_t i = e % d.Dk, h = (e / d.Dk) % d.Hv, t = (e / (d.Dk * d.Hv)) % d.T,
                  bb = e / (d.Dk * d.Hv * d.T);
    const int nt = (int)(d.Dv / KT);
    const int64_t v0 = (bb * d.Hv + h) * nt;
    float s = 0.f;
    for (int tl = 0; tl < nt; ++tl) s += a.gpart[((v0 + tl) * d.Tp + t) * d.Dk + i];
    stf((TI*)a.d_lg + e, s);
    if (i == 0) {
        float sb = 0.f;
        for (int tl = 0; tl < nt; ++tl) sb += a.bpart[(v0 + tl) * d.Tp + t];
        stf((TI*)a.d_beta + (bb * d.T + t) * d.Hv + h, sb);
    }
}

size_t fwd_smem(const Dims& d) {
    return sizeof(float) * (3 * (size_t)kSeg * d.Dk + (size_t)kSeg * KT + kSeg) + sizeof(int) * kSeg;
}

size_t bwd_smem(const Dims& d) {
    const size_t NW = kThreads / 32;
    return sizeof(float) * (NW * (kSub + 1) * 2 * (size_t)d.Dk + 3 * (size_t)kSeg * d.Dk +
                            2 * (size_t)kSeg * KT + kSeg + NW * (3 * (size_t)d.Dk + 1)) +
           sizeof(int) * kSeg;
}

template <typename TI>
cudaError_t launch_kc_fwd_t(const Dims& d, const Ptrs& p, const KcArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)(d.Dv / KT), (unsigned)d.Hv, (unsigned)d.B);
    kc_fwd_kernel<TI><<<grid, kThreads, fwd_smem(d), s>>>(d, p, a);
    count_launches(1);
    return cudaPeekAtLastError();
}

template <typename TI>
cudaError_t launch_kc_bwd_t(const Dims& d, const Ptrs& p, const KcArgs& a, cudaStream_t s) {
    const size_t smem = bwd_smem(d);
    auto kern = kc_bwd_kernel<TI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / KT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads, smem, s>>>(d, p, a);
    const int64_t n = d.B * d.T * d.Hv * d.Dk;
    kc_gate_kernel<TI><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(d, a);
    count_launches(2);
    return cudaPeekAtLastError();
}

}  // namespace

bool kc_supported(const Dims& d) {
    return d.Dk % 32 == 0 && d.Dk / KG <= kMaxR && d.Dv % KT == 0;
}
size_t kc_bwd_smem_bytes(const Dims& d) { return bwd_smem(d); }
int64_t kc_tiles(const Dims& d) { return d.Dv / KT; }
int64_t kc_segments(const Dims& d) { return (d.T + kSeg - 1) / kSeg; }

cudaError_t launch_kc_forward(const Dims& d, const Ptrs& p, const void* log_decay, const void* beta,
                              float* ckpt, cudaStream_t s) {
    KcArgs a{};
    a.lg = log_decay;
    a.beta = beta;
    a.ckpt = ckpt;
    return d.dtype == 1 ? launch_kc_fwd_t<__nv_bfloat16>(d, p, a, s) : launch_kc_fwd_t<float>(d, p, a, s);
}

cudaError_t launch_kc_backward(const Dims& d, const Ptrs& p, const void* log_decay,
                               const void* beta, const float* ckpt, float* gpart, float* bpart,
                               void* d_log_decay, void* d_beta, cudaStream_t s) {
    KcArgs a{};
    a.lg = log_decay;
    a.beta = beta;
    a.ckpt = const_cast<float*>(ckpt);
    a.gpart = gpart;
    a.bpart = bpart;
    a.d_lg = d_log_decay;
    a.d_beta = d_beta;
    return d.dtype == 1 ? launch_kc_bwd_t<__nv_bfloat16>(d, p, a, s) : launch_kc_bwd_t<float>(d, p, a, s);
}

}  // namespace gdn
