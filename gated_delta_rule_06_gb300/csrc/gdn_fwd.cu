// gdn_fwd.cu -- chunked forward of the gated delta rule, CUDA-core (FFMA) path.
//
// Inside one 64-step chunk with start state S (Dk x Dv) the recurrence
//     S <- g S;  delta = beta (v - S^T k);  S <- S + k delta^T;  o = S^T q
// (mlx-lm PR "Add gated_delta_update VJP", "What this PR adds"; torch-to-nnef
// "custom_extractors/gdn": the chunked rule equals the recurrent one up to
// floating-point reordering) unrolls, with Gamma the in-chunk cumulative
// log-decay, gam = exp(Gamma), M_ij = exp(Gamma_i - Gamma_j) (j <= i),
// e_j = exp(Gamma_63 - Gamma_j), into the WY/UT form through a unit
// lower-triangular solve (mlx-lm page, "Scope and follow-ups"):
//     A_ij  = beta_i M_ij <k_i, k_j>  (j < i),   T = (I + A)^-1
//     W = T diag(beta gam) K,   U = T diag(beta) V,   P = (Q K^T) o M (j <= i)
//     Delta = U - W S
//     O     = diag(gam) Q S + P Delta
//     S'    = gam_63 S + K^T diag(e) Delta
// fwd_chunk computes T, W, U, P for every (b, h, chunk) in parallel;
// fwd_scan walks the chunks in order per (b, h, Dv-tile) and writes the
// per-chunk fp32 state checkpoints, Delta and the output.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

// ---------------------------------------------------------------------------
// fwd_chunk: one CTA per (chunk, value head, batch)
// ---------------------------------------------------------------------------
template <typename TI>
__global__ void __launch_bounds__(256) fwd_chunk_kernel(Dims d, Ptrs p) {
    extern __shared__ float sm[];
    const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int Dm = Dk > Dv ? Dk : Dv;
    float* X1 = sm;                  // [64][Dm]
    float* X2 = X1 + kChunk * Dm;    // [64][Dm]
    float* Gkk = X2 + kChunk * Dm;   // [64][64]
    float* Gqk = Gkk + kChunk * kChunk;
    float* Ti = Gqk + kChunk * kChunk;
    float* bt = Ti + kChunk * kChunk;  // [64]
    float* rqv = bt + kChunk;
    float* rkv = rqv + kChunk;
    double* Gm = reinterpret_cast<double*>(rkv + kChunk);  // [64], 8-byte aligned

    const int64_t t0 = (int64_t)c * kChunk;
    const int64_t gbase = ((int64_t)bb * d.Hv + h) * d.Tp + t0;
    const int64_t rbase = ((int64_t)bb * d.Hk + j) * d.Tp + t0;
    const float qscale = rsqrtf((float)Dk);
    for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
        Gm[i] = p.gam[gbase + i];
        bt[i] = p.beta[gbase + i];
        rqv[i] = p.rq[rbase + i] * qscale;
        rkv[i] = p.rk[rbase + i];
    }
    __syncthreads();
    const TI* q = (const TI*)p.q;
    const TI* k = (const TI*)p.k;
    for (int idx = threadIdx.x; idx < kChunk * Dk; idx += blockDim.x) {
        const int i = idx / Dk, x = idx % Dk;
        const int64_t t = t0 + i;
        float kv = 0.f, qv = 0.f;
        if (t < d.T) {
            const int64_t off = (((int64_t)bb * d.T + t) * d.Hk + j) * Dk + x;
            kv = ldf(k + off) * rkv[i];
            qv = ldf(q + off) * rqv[i];
        }
        X1[i * Dk + x] = kv;
        X2[i * Dk + x] = qv;
    }
    __syncthreads();
    // Grams: K K^T and Q K^T (normalised rows)
    cta_gemm<4, 4>(kChunk, kChunk, Dk, X1, Dk, 1, X1, 1, Dk, Gkk, kChunk, 1.f, 0.f, nullptr);
    cta_gemm<4, 4>(kChunk, kChunk, Dk, X2, Dk, 1, X1, 1, Dk, Gqk, kChunk, 1.f, 0.f, nullptr);
    __syncthreads();
    // A (strictly lower, in Gkk) and P (lower incl. diagonal, in Gqk)
    TI* P = (TI*)p.P + (((int64_t)bb * d.Hv + h) * d.NC + c) * kChunk * kChunk;
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) {
        const int i = idx / kChunk, jj = idx % kChunk;
        const float m = jj <= i ? expf((float)(Gm[i] - Gm[jj])) : 0.f;
        Gkk[idx] = jj < i ? bt[i] * m * Gkk[idx] : 0.f;
        const float pv = m * Gqk[idx];
        Gqk[idx] = pv;
        stf(P + idx, pv);
    }
    __syncthreads();
    // T = (I + A)^-1 by forward substitution, one thread per column
    if (threadIdx.x < kChunk) {
        const int col = threadIdx.x;
        for (int i = 0; i < kChunk; ++i) {
            float v = (i == col) ? 1.f : 0.f;
            if (i > col) {
                for (int jj = col; jj < i; ++jj) v = fmaf(-Gkk[i * kChunk + jj], Ti[jj * kChunk + col], v);
            }
            Ti[i * kChunk + col] = v;
        }
    }
    __syncthreads();
    float* Tg = p.Tinv + (((int64_t)bb * d.Hv + h) * d.NC + c) * kChunk * kChunk;
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) Tg[idx] = Ti[idx];
    // W = T diag(beta gam) K
    for (int idx = threadIdx.x; idx < kChunk * Dk; idx += blockDim.x) {
        const int i = idx / Dk;
        X1[idx] *= bt[i] * expf((float)Gm[i]);
    }
    __syncthreads();
    cta_gemm<4, 4>(kChunk, Dk, kChunk, Ti, kChunk, 1, X1, Dk, 1, X2, Dk, 1.f, 0.f, nullptr);
    __syncthreads();
    TI* W = (TI*)p.W + gbase * Dk;
    for (int idx = threadIdx.x; idx < kChunk * Dk; idx += blockDim.x) stf(W + idx, X2[idx]);
    // U = T diag(beta) V
    const TI* v = (const TI*)p.v;
    for (int idx = threadIdx.x; idx < kChunk * Dv; idx += blockDim.x) {
        const int i = idx / Dv, x = idx % Dv;
        const int64_t t = t0 + i;
        float vv = 0.f;
        if (t < d.T) vv = ldf(v + (((int64_t)bb * d.T + t) * d.Hv + h) * Dv + x) * bt[i];
        X1[idx] = vv;
    }
    __syncthreads();
    cta_gemm<4, 4>(kChunk, Dv, kChunk, Ti, kChunk, 1, X1, Dv, 1, X2, Dv, 1.f, 0.f, nullptr);
    __syncthreads();
    float* U = p.U + gbase * Dv;
    for (int idx = threadIdx.x; idx < kChunk * Dv; idx += blockDim.x) U[idx] = X2[idx];
}

// ---------------------------------------------------------------------------
// fwd_scan: one CTA per (Dv tile, value head, batch), sequential over chunks
// ---------------------------------------------------------------------------
template <typename TI, int DVT>
__global__ void __launch_bounds__(256) fwd_scan_kernel(Dims d, Ptrs p) {
    extern __shared__ float sm[];
    const int tile = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int n0 = tile * DVT;
    float* S = sm;                       // [Dk][DVT]
    float* big = S + Dk * DVT;           // [64][Dk]
    float* Pm = big + kChunk * Dk;       // [64][64]
    float* Dl = Pm + kChunk * kChunk;    // [64][DVT]
    float* O = Dl + kChunk * DVT;        // [64][DVT]
    float* De = O + kChunk * DVT;        // [64][DVT]
    float* gm = De + kChunk * DVT;       // [64] exp(Gamma)
    float* ev = gm + kChunk;             // [64] exp(Gamma_63 - Gamma)
    float* rqv = ev + kChunk;
    float* rkv = rqv + kChunk;

    const TI* q = (const TI*)p.q;
    const TI* k = (const TI*)p.k;
    const TI* W = (const TI*)p.W;
    const float* U = p.U;
    const TI* P = (const TI*)p.P;
    float* Delta = p.Delta;
    TI* o = (TI*)p.o;
    const float qscale = rsqrtf((float)Dk);
    const int64_t sbase = ((int64_t)bb * d.Hv + h) * Dk * Dv;
    for (int idx = threadIdx.x; idx < Dk * DVT; idx += blockDim.x) {
        const int x = idx / DVT, n = idx % DVT;
        S[idx] = p.state0 ? p.state0[sbase + (int64_t)x * Dv + n0 + n] : 0.f;
    }
    for (int64_t c = 0; c < d.NC; ++c) {
        const int64_t t0 = c * kChunk;
        const int64_t gbase = ((int64_t)bb * d.Hv + h) * d.Tp + t0;
        const int64_t rbase = ((int64_t)bb * d.Hk + j) * d.Tp + t0;
        __syncthreads();  // previous chunk fully done with smem
        for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
            const double G = p.gam[gbase + i];
            gm[i] = expf((float)G);
            ev[i] = expf((float)(p.gam[gbase + kChunk - 1] - G));
            rqv[i] = p.rq[rbase + i] * qscale;
            rkv[i] = p.rk[rbase + i];
        }
        float* ck = p.ckpt + (((int64_t)bb * d.Hv + h) * d.NC + c) * Dk * Dv;
        for (int idx = threadIdx.x; idx < Dk * DVT; idx += blockDim.x) {
            const int x = idx / DVT, n = idx % DVT;
            ck[(int64_t)x * Dv + n0 + n] = S[idx];
        }
        for (int idx = threadIdx.x; idx < kChunk * Dk; idx += blockDim.x)
            big[idx] = ldf(W + gbase * Dk + idx);
        for (int idx = threadIdx.x; idx < kChunk * DVT; idx += blockDim.x) {
            const int i = idx / DVT, n = idx % DVT;
            Dl[idx] = U[(gbase + i) * Dv + n0 + n];
        }
        __syncthreads();
        // Delta = U - W S
        cta_gemm<2, 4>(kChunk, DVT, Dk, big, Dk, 1, S, DVT, 1, Dl, DVT, -1.f, 1.f, nullptr);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kChunk * DVT; idx += blockDim.x) {
            const int i = idx / DVT, n = idx % DVT;
            Delta[(gbase + i) * Dv + n0 + n] = Dl[idx];
        }
        // O = diag(gam) Q S + P Delta
        for (int idx = threadIdx.x; idx < kChunk * Dk; idx += blockDim.x) {
            const int i = idx / Dk, x = idx % Dk;
            const int64_t t = t0 + i;
            big[idx] = t < d.T ? ldf(q + (((int64_t)bb * d.T + t) * d.Hk + j) * Dk + x) * rqv[i]
                               : 0.f;
        }
        const TI* Pc = P + (((int64_t)bb * d.Hv + h) * d.NC + c) * kChunk * kChunk;
        for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) Pm[idx] = ldf(Pc + idx);
        __syncthreads();
        cta_gemm<2, 4>(kChunk, DVT, Dk, big, Dk, 1, S, DVT, 1, O, DVT, 1.f, 0.f, gm);
        __syncthreads();
        cta_gemm<2, 4>(kChunk, DVT, kChunk, Pm, kChunk, 1, Dl, DVT, 1, O, DVT, 1.f, 1.f, nullptr);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kChunk * DVT; idx += blockDim.x) {
            const int i = idx / DVT, n = idx % DVT;
            const int64_t t = t0 + i;
            if (t < d.T) stf(o + (((int64_t)bb * d.T + t) * d.Hv + h) * Dv + n0 + n, O[idx]);
        }
        // S' = gam_63 S + K^T diag(e) Delta
        for (int idx = threadIdx.x; idx < kChunk * Dk; idx += blockDim.x) {
            const int i = idx / Dk, x = idx % Dk;
            const int64_t t = t0 + i;
            big[idx] = t < d.T ? ldf(k + (((int64_t)bb * d.T + t) * d.Hk + j) * Dk + x) * rkv[i]
                               : 0.f;
        }
        for (int idx = threadIdx.x; idx < kChunk * DVT; idx += blockDim.x) De[idx] = Dl[idx] * ev[idx / DVT];
        __syncthreads();
        cta_gemm<2, 4>(Dk, DVT, kChunk, big, 1, Dk, De, DVT, 1, S, DVT, 1.f, gm[kChunk - 1], nullptr);
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < Dk * DVT; idx += blockDim.x) {
        const int x = idx / DVT, n = idx % DVT;
        p.state_T[sbase + (int64_t)x * Dv + n0 + n] = S[idx];
    }
}

template <typename TI, int DVT>
cudaError_t launch_scan_t(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = sizeof(float) * ((size_t)d.Dk * DVT + (size_t)kChunk * d.Dk +
                                         kChunk * kChunk + 3 * kChunk * DVT + 4 * kChunk);
    auto kern = fwd_scan_kernel<TI, DVT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, 256, smem, s>>>(d, p);
    count_launches(1);
    return cudaPeekAtLastError();
}

template <typename TI>
cudaError_t launch_fwd_chunk_t(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t Dm = d.Dk > d.Dv ? d.Dk : d.Dv;
    const size_t smem = sizeof(float) * (2 * kChunk * Dm + 3 * kChunk * kChunk + 3 * kChunk) +
                        sizeof(double) * kChunk;
    auto kern = fwd_chunk_kernel<TI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, 256, smem, s>>>(d, p);
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_fwd_chunk(const Dims& d, const Ptrs& p, cudaStream_t s) {
    if (tc_path(d)) return launch_fwd_chunk_tc(d, p, s);
    return d.dtype == 1 ? launch_fwd_chunk_t<__nv_bfloat16>(d, p, s)
                        : launch_fwd_chunk_t<float>(d, p, s);
}

cudaError_t launch_fwd_scan(const Dims& d, const Ptrs& p, cudaStream_t s) {
    if (tc_path(d)) return launch_fwd_scan_tc(d, p, s);
    if (d.Dv % 32 == 0)
        return d.dtype == 1 ? launch_scan_t<__nv_bfloat16, 32>(d, p, s) : launch_scan_t<float, 32>(d, p, s);
    if (d.Dv % 16 == 0)
        return d.dtype == 1 ? launch_scan_t<__nv_bfloat16, 16>(d, p, s) : launch_scan_t<float, 16>(d, p, s);
    return d.dtype == 1 ? launch_scan_t<__nv_bfloat16, 8>(d, p, s) : launch_scan_t<float, 8>(d, p, s);
}

}  // namespace gdn
