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
constexpr int KG = 16;             // row groups
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

// sum over the 16 row groups of column jj: lanes l and l + 16 of a warp hold row
// groups 2w and 2w + 1; the eight warp sums go through red[8][KT] in warp order
__device__ __forceinline__ float col_sum(float x, float (*red)[KT], int warp, int lane, int jj) {
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    if (lane < 16) red[warp][jj] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[w][jj];
    return s;
}

// sum over the 16 columns of the tile (the 16 lanes of a half warp)
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Per-step vectors of steps t0 .. t0 + L - 1 of (b, h) into shared memory: the
// normalised k and q rows, g per key channel, beta, the applied flag, the tile's
// v columns and (ob non-null) its d_o columns.  Every global load of the
// segment is issued before the first store, so the segment pays one load
// latency, not one per step.
template <typename TI>
__device__ __forceinline__ void load_seg(const Dims& d, const Ptrs& p, const KcArgs& a,
                                         int64_t bb, int64_t h, int64_t t0, int L, int col0,
                                         float* kh, float* qh, float* g, float* v, float* ob,
                                         float* bt, int* on) {
    const int tid = threadIdx.x;
    const int64_t j = h / d.G;
    const int Dk = (int)d.Dk;
    float xk[kSeg], xq[kSeg], xg[kSeg], nk[kSeg], nq[kSeg], xv[kSeg], xo[kSeg], xb[kSeg];
    bool live[kSeg];
#pragma unroll
    for (int i = 0; i < kSeg; ++i) {
        const int64_t t = t0 + i;
        const bool in = i < L;
        live[i] = in && (p.mask == nullptr || p.mask[bb * d.T + t] != 0);
        xk[i] = xq[i] = nk[i] = nq[i] = xv[i] = xo[i] = xb[i] = 0.f;
        xg[i] = 0.f;
        if (in && tid < Dk) {
            const int64_t xi = ((bb * d.T + t) * d.Hk + j) * Dk + tid;
            const int64_t ri = (bb * d.Hk + j) * d.Tp + t;
            xk[i] = ldf((const TI*)p.k + xi);
            xq[i] = ldf((const TI*)p.q + xi);
            nk[i] = p.rk[ri];
            nq[i] = p.rq[ri];
            xg[i] = ldf((const TI*)a.lg + ((bb * d.T + t) * d.Hv + h) * Dk + tid);
        }
        if (in && tid < KT) {
            const int64_t vi = ((bb * d.T + t) * d.Hv + h) * d.Dv + col0 + tid;
            xv[i] = ldf((const TI*)p.v + vi);
            if (ob) xo[i] = ldf((const TI*)p.d_o + vi);
        }
        if (in && tid == 0) xb[i] = ldf((const TI*)a.beta + (bb * d.T + t) * d.Hv + h);
    }
#pragma unroll
    for (int i = 0; i < kSeg; ++i) {
        if (i >= L) break;
        if (tid < Dk) {
            kh[i * Dk + tid] = xk[i] * nk[i];
            qh[i * Dk + tid] = xq[i] * nq[i] * rsqrtf((float)Dk);
            g[i * Dk + tid] = live[i] ? expf(xg[i]) : 1.f;
        }
        if (tid < KT) {
            v[i * KT + tid] = xv[i];
            if (ob) ob[i * KT + tid] = xo[i];
        }
        if (tid == 0) {
            bt[i] = live[i] ? xb[i] : 0.f;
            on[i] = live[i] ? 1 : 0;
        }
    }
}

template <typename TI>
__global__ void __launch_bounds__(kThreads) kc_fwd_kernel(Dims d, Ptrs p, KcArgs a) {
    extern __shared__ __align__(16) float kcf[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv, R = Dk / KG;
    float* kh = kcf;                  // [kSeg][Dk]
    float* qh = kh + kSeg * Dk;       // [kSeg][Dk]
    float* gv = qh + kSeg * Dk;       // [kSeg][Dk]
    float* vv = gv + kSeg * Dk;       // [kSeg][KT]
    float* bt = vv + kSeg * KT;       // [kSeg]
    int* on = reinterpret_cast<int*>(bt + kSeg);
    __shared__ float red[2][kThreads / 32][KT];
    const int tile = blockIdx.x;
    const int64_t h = blockIdx.y, bb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jj = tid % KT, rg = tid / KT, r0 = rg * R;
    const int col0 = tile * KT, col = col0 + jj;
    const int64_t bh = bb * d.Hv + h;
    const int64_t NS = (d.T + kSeg - 1) / kSeg;
    int nred = 0;
    float S[kMaxR];
#pragma unroll
    for (int m = 0; m < kMaxR; ++m)
        S[m] = (m < R && p.state0) ? p.state0[(bh * Dk + r0 + m) * Dv + col] : 0.f;
    for (int64_t sg = 0; sg < NS; ++sg) {
        const int64_t t0 = sg * kSeg;
        const int L = (int)(d.T - t0 < kSeg ? d.T - t0 : kSeg);
        if (a.ckpt) {  // the state at the start of this segment
            float* ck = a.ckpt + ((bh * NS + sg) * Dk + r0) * Dv + col;
#pragma unroll
            for (int m = 0; m < kMaxR; ++m)
                if (m < R) ck[(int64_t)m * Dv] = S[m];
        }
        __syncthreads();  // the previous segment's vectors have been read
        load_seg<TI>(d, p, a, bb, h, t0, L, col0, kh, qh, gv, vv, nullptr, bt, on);
        __syncthreads();
        for (int i = 0; i < L; ++i) {
            const float* kk = kh + i * Dk;
            const float* gg = gv + i * Dk;
            float pp = 0.f;
#pragma unroll
            for (int m = 0; m < kMaxR; ++m)
                if (m < R) pp = fmaf(gg[r0 + m] * S[m], kk[r0 + m], pp);
            const float pc = col_sum(pp, red[nred], warp, lane, jj);
            nred ^= 1;
            if (on[i]) {
                const float dl = bt[i] * (vv[i * KT + jj] - pc);
#pragma unroll
                for (int m = 0; m < kMaxR; ++m)
                    if (m < R) S[m] = fmaf(kk[r0 + m], dl, gg[r0 + m] * S[m]);
            }
            float po = 0.f;
#pragma unroll
            for (int m = 0; m < kMaxR; ++m)
                if (m < R) po = fmaf(S[m], qh[i * Dk + r0 + m], po);
            const float oc = col_sum(po, red[nred], warp, lane, jj);
            nred ^= 1;
            if (rg == 0) stf((TI*)p.o + ((bb * d.T + t0 + i) * d.Hv + h) * Dv + col, oc);
        }
    }
#pragma unroll
    for (int m = 0; m < kMaxR; ++m)
        if (m < R) p.state_T[(bh * Dk + r0 + m) * Dv + col] = S[m];
}

// Partials of the tile (b, h, tile) are written as if (h, tile) were value head
// h nt + tile of B x (Hv nt) heads.
template <typename TI>
__global__ void __launch_bounds__(kThreads) kc_bwd_kernel(Dims d, Ptrs p, KcArgs a) {
    extern __shared__ __align__(16) float kcs[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv, R = Dk / KG;
    float* hist = kcs;                              // [kSeg + 1][Dk][KT] states of a segment
    float* kh = hist + (kSeg + 1) * Dk * KT;        // [kSeg][Dk]
    float* qh = kh + kSeg * Dk;                     // [kSeg][Dk]
    float* gv = qh + kSeg * Dk;                     // [kSeg][Dk]
    float* vv = gv + kSeg * Dk;                     // [kSeg][KT]
    float* ob = vv + kSeg * KT;                     // [kSeg][KT] d_o
    float* dlv = ob + kSeg * KT;                    // [kSeg][KT] delta
    float* pvv = dlv + kSeg * KT;                   // [kSeg][KT] p
    float* bt = pvv + kSeg * KT;                    // [kSeg]
    int* on = reinterpret_cast<int*>(bt + kSeg);    // [kSeg]
    __shared__ float red[2][kThreads / 32][KT];
    const int tile = blockIdx.x;
    const int64_t h = blockIdx.y, bb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jj = tid % KT, rg = tid / KT, r0 = rg * R;
    const int col0 = tile * KT, col = col0 + jj;
    const int nt = Dv / KT;
    const int64_t bh = bb * d.Hv + h;
    const int64_t hv2 = bb * d.Hv * nt + h * nt + tile;  // virtual head of the partials
    const int64_t NS = (d.T + kSeg - 1) / kSeg;
    float* dqh = p.dqh;
    float* dkh = p.dkh;
    int nred = 0;
    float Sb[kMaxR];
#pragma unroll
    for (int m = 0; m < kMaxR; ++m)
        Sb[m] = (m < R && p.d_state_T) ? p.d_state_T[(bh * Dk + r0 + m) * Dv + col] : 0.f;
    for (int64_t sg = NS - 1; sg >= 0; --sg) {
        const int64_t t0 = sg * kSeg;
        const int L = (int)(d.T - t0 < kSeg ? d.T - t0 : kSeg);
        load_seg<TI>(d, p, a, bb, h, t0, L, col0, kh, qh, gv, vv, ob, bt, on);
        float S[kMaxR];
        const float* ck = a.ckpt + ((bh * NS + sg) * Dk + r0) * Dv + col;
#pragma unroll
        for (int m = 0; m < kMaxR; ++m)
            if (m < R) {
                S[m] = ck[(int64_t)m * Dv];
                hist[(r0 + m) * KT + jj] = S[m];
            }
        __syncthreads();
        // the segment's states again, with delta and p of every step
        for (int i = 0; i < L; ++i) {
            float pp = 0.f;
#pragma unroll
            for (int m = 0; m < kMaxR; ++m)
                if (m < R) pp = fmaf(gv[i * Dk + r0 + m] * S[m], kh[i * Dk + r0 + m], pp);
            const float pc = col_sum(pp, red[nred], warp, lane, jj);
            nred ^= 1;
            float dl = 0.f;
            if (on[i]) {
                dl = bt[i] * (vv[i * KT + jj] - pc);
#pragma unroll
                for (int m = 0; m < kMaxR; ++m)
                    if (m < R) S[m] = fmaf(kh[i * Dk + r0 + m], dl, gv[i * Dk + r0 + m] * S[m]);
            }
            if (rg == 0) {
                dlv[i * KT + jj] = dl;
                pvv[i * KT + jj] = pc;
            }
#pragma unroll
            for (int m = 0; m < kMaxR; ++m)
                if (m < R) hist[((i + 1) * Dk + r0 + m) * KT + jj] = S[m];
        }
        __syncthreads();
        // reverse over the segment's steps
        for (int i = L - 1; i >= 0; --i) {
            const int64_t t = t0 + i;
            const float* scur = hist + (i + 1) * Dk * KT;
            const float* sprev = hist + i * Dk * KT;
            const float oj = ob[i * KT + jj];
            const int64_t prow = (hv2 * d.Tp + t) * Dk;
#pragma unroll
            for (int m = 0; m < kMaxR; ++m)
                if (m < R) {
                    Sb[m] = fmaf(qh[i * Dk + r0 + m], oj, Sb[m]);
                    const float qb = row_sum(scur[(r0 + m) * KT + jj] * oj);
                    if (jj == 0) dqh[prow + r0 + m] = qb;
                }
            if (on[i]) {
                const float dl = dlv[i * KT + jj], pc = pvv[i * KT + jj], beta = bt[i];
                float db = 0.f;
#pragma unroll
                for (int m = 0; m < kMaxR; ++m)
                    if (m < R) db = fmaf(Sb[m], kh[i * Dk + r0 + m], db);
                const float dbar = col_sum(db, red[nred], warp, lane, jj);
                nred ^= 1;
                if (rg == 0) stf((TI*)p.dv + ((bb * d.T + t) * d.Hv + h) * Dv + col, beta * dbar);
                const float bsum = row_sum(dbar * (vv[i * KT + jj] - pc));
                if (tid == 0) a.bpart[hv2 * d.Tp + t] = bsum;
                const float pbar = -beta * dbar;
#pragma unroll
                for (int m = 0; m < kMaxR; ++m)
                    if (m < R) {
                        const float gi = gv[i * Dk + r0 + m], sp = sprev[(r0 + m) * KT + jj];
                        const float kb = row_sum(fmaf(Sb[m], dl, gi * sp * pbar));
                        Sb[m] = fmaf(kh[i * Dk + r0 + m], pbar, Sb[m]);  // Sbar_a
                        const float gb = row_sum(Sb[m] * sp);
                        Sb[m] *= gi;
                        if (jj == 0) {
                            dkh[prow + r0 + m] = kb;
                            a.gpart[prow + r0 + m] = gb * gi;
                        }
                    }
            } else {
                if (rg == 0) stf((TI*)p.dv + ((bb * d.T + t) * d.Hv + h) * Dv + col, 0.f);
                if (tid == 0) a.bpart[hv2 * d.Tp + t] = 0.f;
#pragma unroll
                for (int m = 0; m < kMaxR; ++m)
                    if (m < R && jj == 0) {
                        dkh[prow + r0 + m] = 0.f;
                        a.gpart[prow + r0 + m] = 0.f;
                    }
            }
        }
        __syncthreads();  // the segment's shared memory is free
    }
#pragma unroll
    for (int m = 0; m < kMaxR; ++m)
        if (m < R) p.dstate0[(bh * Dk + r0 + m) * Dv + col] = Sb[m];
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
    return sizeof(float) * ((size_t)(kSeg + 1) * d.Dk * KT + 3 * (size_t)kSeg * d.Dk +
                            4 * (size_t)kSeg * KT + kSeg) + sizeof(int) * kSeg;
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
    return d.Dk % KG == 0 && d.Dk / KG <= kMaxR && d.Dv % KT == 0;
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
