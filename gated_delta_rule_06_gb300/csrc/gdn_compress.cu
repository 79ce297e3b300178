// gdn_compress.cu -- rank-r compressed chunk states (mlx-lm PR "Add
// gated_delta_update VJP", "Post-initial-submission extensions", Extension 1:
// power-iteration rank-r truncation of the state at every chunk boundary, so
// that the backward keeps rank-r factors of each chunk state instead of the
// state itself).
//
// trunc_kernel: at boundary c, for every (b, h), the range of the chunk-end
// state S (Dk x Dv, fp32) is estimated by subspace iteration from the caller's
// start block Omega (Dv x r):
//     Y = S Omega,  Q = orth(Y),  then `iters` times  Y = S (S^T Q),  Q = orth(Y)
// and S is replaced by Q R with R = Q^T S.  orth is classical Gram-Schmidt with
// one reorthogonalisation pass, run by one warp; a column whose remaining norm
// is at most kDrop of its norm before (it lies in the span of the earlier ones
// to rounding) becomes zero, so a state of rank below r keeps exactly its
// range.  The factors Q, R go to the saved buffer; the truncated state Q R
// (fp32) is the next chunk's start state.
//
// expand_kernel: the bf16 checkpoint images of every chunk start state for the
// backward's gradient kernel, rebuilt from the factors (the initial state from
// its fp32 copy).  Every element is the same fmaf chain over q as in
// trunc_kernel, so the images equal those the forward scan formed.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRmax = 16;       // largest rank
constexpr int kCThreads = 256;  // threads per CTA
constexpr float kDrop = 1e-5f;  // own-norm relative drop threshold (fp32)

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Yc [kRmax][n] (column-major, n rows) orthonormalised in place by one warp:
// classical Gram-Schmidt, each column projected twice against the earlier ones
__device__ void orth_warp(float* Yc, int n, int r, int lane) {
    for (int j = 0; j < r; ++j) {
        float* y = Yc + j * n;
        float own = 0.f;
        for (int i = lane; i < n; i += 32) own = fmaf(y[i], y[i], own);
        own = warp_sum(own);
        for (int pass = 0; pass < 2; ++pass) {
            float h[kRmax];
#pragma unroll
            for (int t = 0; t < kRmax; ++t) {
                float acc = 0.f;
                if (t < j)
                    for (int i = lane; i < n; i += 32) acc = fmaf(Yc[t * n + i], y[i], acc);
                h[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < kRmax; ++t)
                if (t < j) h[t] = warp_sum(h[t]);
            for (int i = lane; i < n; i += 32) {
                float w = y[i];
#pragma unroll
                for (int t = 0; t < kRmax; ++t)
                    if (t < j) w = fmaf(-h[t], Yc[t * n + i], w);
                y[i] = w;
            }
            __syncwarp();
        }
        float nn = 0.f;
        for (int i = lane; i < n; i += 32) nn = fmaf(y[i], y[i], nn);
        nn = warp_sum(nn);
        const float norm = sqrtf(nn);
        const float sc = (own > 0.f && norm > kDrop * sqrtf(own)) ? 1.f / norm : 0.f;
        for (int i = lane; i < n; i += 32) y[i] *= sc;
        __syncwarp();
    }
}

// Yc[q][i] = sum_v S[i][v] X[v][q] (X [Dv][kRmax]); warp w takes rows w, w + 8, ...,
// lanes split v, fixed butterfly sums
__device__ void rows_times(const float* __restrict__ S, const float* X, float* Yc, int Dk, int Dv,
                           int warp, int lane) {
    for (int i = warp; i < Dk; i += kCThreads / 32) {
        float acc[kRmax];
#pragma unroll
        for (int q = 0; q < kRmax; ++q) acc[q] = 0.f;
        for (int v = lane; v < Dv; v += 32) {
            const float s = S[(int64_t)i * Dv + v];
#pragma unroll
            for (int q = 0; q < kRmax; ++q) acc[q] = fmaf(s, X[v * kRmax + q], acc[q]);
        }
        float mine = 0.f;
#pragma unroll
        for (int q = 0; q < kRmax; ++q) {
            const float t = warp_sum(acc[q]);
            if (lane == q) mine = t;
        }
        if (lane < kRmax) Yc[lane * Dk + i] = mine;
    }
}

// acc[q] = sum_i S[i][v] Qc[q][i] for the column v of this thread
__device__ __forceinline__ void col_times(const float* __restrict__ S, const float* Qc, int Dk, int Dv,
                                          int v, float (&acc)[kRmax]) {
#pragma unroll
    for (int q = 0; q < kRmax; ++q) acc[q] = 0.f;
    for (int i = 0; i < Dk; ++i) {
        const float s = S[(int64_t)i * Dv + v];
#pragma unroll
        for (int q = 0; q < kRmax; ++q) acc[q] = fmaf(s, Qc[q * Dk + i], acc[q]);
    }
}

// one element of Q R: the fmaf chain over q = 0 .. r - 1 ascending, from zero
__device__ __forceinline__ float qr_elem(const float* qrow, int qstride, const float* rcol, int rstride,
                                         int r) {
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kRmax; ++q)
        if (q < r) acc = fmaf(qrow[q * qstride], rcol[q * rstride], acc);
    return acc;
}

// One CTA per (value head, batch).  S_end [B][Hv][Dk][Dv] chunk-end states in,
// S_tr the truncated states out; Qf [B][Hv][NC][Dk][r], Rf [B][Hv][NC][r][Dv]
// receive slot c.
__global__ void __launch_bounds__(kCThreads) trunc_kernel(Dims d, const float* __restrict__ S_end,
                                                          const float* __restrict__ omega, int r,
                                                          int iters, float* __restrict__ S_tr,
                                                          float* __restrict__ Qf,
                                                          float* __restrict__ Rf, int64_t c) {
    extern __shared__ __align__(16) float csm[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    float* Om = csm;                 // [Dv][kRmax]
    float* Zr = Om + Dv * kRmax;     // [Dv][kRmax]
    float* Yc = Zr + Dv * kRmax;     // [kRmax][Dk], Q in place
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t bh = (int64_t)blockIdx.y * d.Hv + blockIdx.x;
    const float* S = S_end + bh * Dk * Dv;
    for (int e = tid; e < Dv * kRmax; e += kCThreads) {
        const int v = e / kRmax, q = e % kRmax;
        Om[e] = q < r ? omega[(int64_t)v * r + q] : 0.f;
    }
    __syncthreads();
    rows_times(S, Om, Yc, Dk, Dv, warp, lane);
    __syncthreads();
    if (warp == 0) orth_warp(Yc, Dk, r, lane);
    __syncthreads();
    for (int it = 0; it < iters; ++it) {
        for (int v = tid; v < Dv; v += kCThreads) {
            float acc[kRmax];
            col_times(S, Yc, Dk, Dv, v, acc);
#pragma unroll
            for (int q = 0; q < kRmax; ++q) Zr[v * kRmax + q] = acc[q];
        }
        __syncthreads();
        rows_times(S, Zr, Yc, Dk, Dv, warp, lane);
        __syncthreads();
        if (warp == 0) orth_warp(Yc, Dk, r, lane);
        __syncthreads();
    }
    // R = Q^T S and the truncated state Q R, column by column
    float* Rg = Rf + (bh * d.NC + c) * (int64_t)r * Dv;
    float* St = S_tr + bh * Dk * Dv;
    for (int v = tid; v < Dv; v += kCThreads) {
        float acc[kRmax];
        col_times(S, Yc, Dk, Dv, v, acc);
#pragma unroll
        for (int q = 0; q < kRmax; ++q)
            if (q < r) Rg[(int64_t)q * Dv + v] = acc[q];
        for (int i = 0; i < Dk; ++i) St[(int64_t)i * Dv + v] = qr_elem(Yc + i, Dk, acc, 1, r);
    }
    float* Qg = Qf + (bh * d.NC + c) * (int64_t)Dk * r;
    for (int e = tid; e < Dk * r; e += kCThreads) {
        const int i = e / r, q = e % r;
        Qg[e] = Yc[q * Dk + i];
    }
}

// Grid (NC, Hv, B): the bf16 panel image of chunk c's start state, byte
// (i / 8) Dv 16 + v 16 + 2 (i % 8) of image (b, h, c) holding S[i][v]
__global__ void __launch_bounds__(kCThreads) expand_kernel(Dims d, const float* __restrict__ S0f,
                                                           const float* __restrict__ Qf,
                                                           const float* __restrict__ Rf, int r,
                                                           uint8_t* __restrict__ img) {
    extern __shared__ __align__(16) float esm[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int64_t c = blockIdx.x;
    const int64_t bh = (int64_t)blockIdx.z * d.Hv + blockIdx.y;
    float* Qs = esm;                  // [Dk][kRmax]
    float* Rs = Qs + Dk * kRmax;      // [kRmax][Dv]
    const int tid = threadIdx.x;
    uint8_t* out = img + (bh * d.NC + c) * (int64_t)Dk * Dv * 2;
    if (c == 0) {
        const float* S = S0f + bh * Dk * Dv;
        for (int e = tid; e < (Dk / 8) * Dv; e += kCThreads) {
            const int gi = e / Dv, v = e % Dv;
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(S[(int64_t)(8 * gi + 2 * u) * Dv + v],
                                                                 S[(int64_t)(8 * gi + 2 * u + 1) * Dv + v]);
                w[u] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(out + (int64_t)gi * Dv * 16 + (int64_t)v * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        return;
    }
    const float* Qg = Qf + (bh * d.NC + c) * (int64_t)Dk * r;
    const float* Rg = Rf + (bh * d.NC + c) * (int64_t)r * Dv;
    for (int e = tid; e < Dk * r; e += kCThreads) Qs[(e / r) * kRmax + e % r] = Qg[e];
    for (int e = tid; e < r * Dv; e += kCThreads) Rs[e] = Rg[e];
    __syncthreads();
    for (int e = tid; e < (Dk / 8) * Dv; e += kCThreads) {
        const int gi = e / Dv, v = e % Dv;
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = qr_elem(Qs + (8 * gi + u) * kRmax, 1, Rs + v, Dv, r);
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * u], x[2 * u + 1]);
            w[u] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(out + (int64_t)gi * Dv * 16 + (int64_t)v * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

bool compress_supported(const Dims& d, int rank, int iters) {
    return rank >= 1 && rank <= kRmax && iters >= 0 && iters <= 16 && d.Dk % 8 == 0 &&
           d.Dk <= 256 && d.Dv <= 256;
}

cudaError_t launch_trunc(const Dims& d, const float* S_end, const float* omega, int rank, int iters,
                         float* S_tr, float* Qf, float* Rf, int64_t c, cudaStream_t s) {
    const size_t smem = sizeof(float) * (size_t)(2 * d.Dv * kRmax + kRmax * d.Dk);
    auto kern = trunc_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)d.Hv, (unsigned)d.B), kCThreads, smem, s>>>(d, S_end, omega, rank, iters, S_tr,
                                                                      Qf, Rf, c);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_expand_ckpt(const Dims& d, const float* S0f, const float* Qf, const float* Rf,
                               int rank, void* img, cudaStream_t s) {
    const size_t smem = sizeof(float) * (size_t)(d.Dk * kRmax + kRmax * d.Dv);
    auto kern = expand_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B), kCThreads, smem, s>>>(
        d, S0f, Qf, Rf, rank, static_cast<uint8_t*>(img));
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace gdn
