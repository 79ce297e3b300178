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
// (fp32) is the next chunk's start state.  The state is staged in shared
// memory once; the products run on the CUDA cores in fp32 (thread per row for
// S X, thread per column for S^T Q), the Gram-Schmidt in registers of one warp.
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

// Y [n][kRmax] (row-major in shared memory, n = Dk <= 256 rows, columns
// r .. kRmax - 1 zero) orthonormalised in place by one warp, the rows held in
// registers (lane l: rows l, l + 32, ...): classical Gram-Schmidt, each column
// projected twice against the earlier ones.  A column whose remaining norm is
// at most kDrop of its norm before becomes zero.
template <int NR>  // rows per lane: ceil(Dk / 32)
__device__ void orth_warp(float* Y, int n, int r, int lane) {
    float y[NR][kRmax];
#pragma unroll
    for (int m = 0; m < NR; ++m) {
        const int i = lane + 32 * m;
#pragma unroll
        for (int q = 0; q < kRmax; ++q) y[m][q] = i < n ? Y[i * kRmax + q] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kRmax; ++j) {
        if (j >= r) break;
        float own = 0.f;
#pragma unroll
        for (int m = 0; m < NR; ++m) own = fmaf(y[m][j], y[m][j], own);
        own = warp_sum(own);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            float h[kRmax];
#pragma unroll
            for (int t = 0; t < kRmax; ++t) {
                h[t] = 0.f;
                if (t < j) {
#pragma unroll
                    for (int m = 0; m < NR; ++m) h[t] = fmaf(y[m][t], y[m][j], h[t]);
                }
            }
#pragma unroll
            for (int t = 0; t < kRmax; ++t)
                if (t < j) h[t] = warp_sum(h[t]);
#pragma unroll
            for (int t = 0; t < kRmax; ++t)
                if (t < j) {
#pragma unroll
                    for (int m = 0; m < NR; ++m) y[m][j] = fmaf(-h[t], y[m][t], y[m][j]);
                }
        }
        float nn = 0.f;
#pragma unroll
        for (int m = 0; m < NR; ++m) nn = fmaf(y[m][j], y[m][j], nn);
        nn = warp_sum(nn);
        const float norm = sqrtf(nn);
        const float sc = (own > 0.f && norm > kDrop * sqrtf(own)) ? 1.f / norm : 0.f;
#pragma unroll
        for (int m = 0; m < NR; ++m) y[m][j] *= sc;
    }
#pragma unroll
    for (int m = 0; m < NR; ++m) {
        const int i = lane + 32 * m;
        if (i < n) {
#pragma unroll
            for (int q = 0; q < kRmax; ++q) Y[i * kRmax + q] = y[m][q];
        }
    }
}

// X [Dv][kRmax] and Y [Dk][kRmax] row-major in shared memory; Ss the state with
// row stride Dv + 1.  rows_times: Y = S X, thread i forms row i.
__device__ __forceinline__ void rows_times(const float* Ss, const float* X, float* Y, int Dk, int Dv,
                                           int tid) {
    for (int i = tid; i < Dk; i += kCThreads) {
        float acc[kRmax];
#pragma unroll
        for (int q = 0; q < kRmax; ++q) acc[q] = 0.f;
        const float* srow = Ss + i * (Dv + 1);
#pragma unroll 4
        for (int v = 0; v < Dv; ++v) {
            const float sv = srow[v];
            const float4* xv = reinterpret_cast<const float4*>(X + v * kRmax);
#pragma unroll
            for (int u = 0; u < kRmax / 4; ++u) {
                const float4 x4 = xv[u];
                acc[4 * u] = fmaf(sv, x4.x, acc[4 * u]);
                acc[4 * u + 1] = fmaf(sv, x4.y, acc[4 * u + 1]);
                acc[4 * u + 2] = fmaf(sv, x4.z, acc[4 * u + 2]);
                acc[4 * u + 3] = fmaf(sv, x4.w, acc[4 * u + 3]);
            }
        }
        float4* yr = reinterpret_cast<float4*>(Y + i * kRmax);
#pragma unroll
        for (int u = 0; u < kRmax / 4; ++u)
            yr[u] = make_float4(acc[4 * u], acc[4 * u + 1], acc[4 * u + 2], acc[4 * u + 3]);
    }
}

// acc[q] = sum_i S[i][v] Q[i][q] for the column v (S^T Q), i ascending
__device__ __forceinline__ void col_times(const float* Ss, const float* Q, int Dk, int Dv, int v,
                                          float (&acc)[kRmax]) {
#pragma unroll
    for (int q = 0; q < kRmax; ++q) acc[q] = 0.f;
#pragma unroll 4
    for (int i = 0; i < Dk; ++i) {
        const float sv = Ss[i * (Dv + 1) + v];
        const float4* qr = reinterpret_cast<const float4*>(Q + i * kRmax);
#pragma unroll
        for (int u = 0; u < kRmax / 4; ++u) {
            const float4 q4 = qr[u];
            acc[4 * u] = fmaf(sv, q4.x, acc[4 * u]);
            acc[4 * u + 1] = fmaf(sv, q4.y, acc[4 * u + 1]);
            acc[4 * u + 2] = fmaf(sv, q4.z, acc[4 * u + 2]);
            acc[4 * u + 3] = fmaf(sv, q4.w, acc[4 * u + 3]);
        }
    }
}

// one element of Q R: the fmaf chain over q = 0 .. r - 1 ascending, from zero
__device__ __forceinline__ float qr_elem(const float* qrow, const float* rcol, int rstride, int r) {
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kRmax; ++q)
        if (q < r) acc = fmaf(qrow[q], rcol[q * rstride], acc);
    return acc;
}

// One CTA per (value head, batch).  S_end [B][Hv][Dk][Dv] chunk-end states in,
// S_tr the truncated states out; Qf [B][Hv][NC][Dk][r], Rf [B][Hv][NC][r][Dv]
// receive slot c.  The state is staged in shared memory (rows padded to Dv + 1
// floats: conflict-free by row and by column).
template <int NR>
__global__ void __launch_bounds__(kCThreads, 1) trunc_kernel(Dims d, const float* __restrict__ S_end,
                                                             const float* __restrict__ omega, int r,
                                                             int iters, float* __restrict__ S_tr,
                                                             float* __restrict__ Qf,
                                                             float* __restrict__ Rf, int64_t c) {
    extern __shared__ __align__(16) float csm[];
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    float* Om = csm;                 // [Dv][kRmax]
    float* Zr = Om + Dv * kRmax;     // [Dv][kRmax]
    float* Yr = Zr + Dv * kRmax;     // [Dk][kRmax], Q in place
    float* Ss = Yr + Dk * kRmax;     // [Dk][Dv + 1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t bh = (int64_t)blockIdx.y * d.Hv + blockIdx.x;
    const float* S = S_end + bh * Dk * Dv;
    for (int e = tid; e < Dk * Dv / 4; e += kCThreads) {
        const float4 x = reinterpret_cast<const float4*>(S)[e];
        const int i = (4 * e) / Dv, v = (4 * e) % Dv;
        float* dst = Ss + i * (Dv + 1) + v;
        dst[0] = x.x;
        dst[1] = x.y;
        dst[2] = x.z;
        dst[3] = x.w;
    }
    for (int e = tid; e < Dv * kRmax; e += kCThreads) {
        const int v = e / kRmax, q = e % kRmax;
        Om[e] = q < r ? omega[(int64_t)v * r + q] : 0.f;
    }
    __syncthreads();
    rows_times(Ss, Om, Yr, Dk, Dv, tid);
    __syncthreads();
    if (warp == 0) orth_warp<NR>(Yr, Dk, r, lane);
    __syncthreads();
    for (int it = 0; it < iters; ++it) {
        for (int v = tid; v < Dv; v += kCThreads) {
            float acc[kRmax];
            col_times(Ss, Yr, Dk, Dv, v, acc);
            float4* zr = reinterpret_cast<float4*>(Zr + v * kRmax);
#pragma unroll
            for (int u = 0; u < kRmax / 4; ++u)
                zr[u] = make_float4(acc[4 * u], acc[4 * u + 1], acc[4 * u + 2], acc[4 * u + 3]);
        }
        __syncthreads();
        rows_times(Ss, Zr, Yr, Dk, Dv, tid);
        __syncthreads();
        if (warp == 0) orth_warp<NR>(Yr, Dk, r, lane);
        __syncthreads();
    }
    // R = Q^T S and the truncated state Q R, column by column
    float* Rg = Rf + (bh * d.NC + c) * (int64_t)r * Dv;
    float* St = S_tr + bh * Dk * Dv;
    for (int v = tid; v < Dv; v += kCThreads) {
        float acc[kRmax];
        col_times(Ss, Yr, Dk, Dv, v, acc);
#pragma unroll
        for (int q = 0; q < kRmax; ++q)
            if (q < r) Rg[(int64_t)q * Dv + v] = acc[q];
        for (int i = 0; i < Dk; ++i) St[(int64_t)i * Dv + v] = qr_elem(Yr + i * kRmax, acc, 1, r);
    }
    float* Qg = Qf + (bh * d.NC + c) * (int64_t)Dk * r;
    for (int e = tid; e < Dk * r; e += kCThreads) Qg[e] = Yr[(e / r) * kRmax + e % r];
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
        for (int u = 0; u < 8; ++u) x[u] = qr_elem(Qs + (8 * gi + u) * kRmax, Rs + v, Dv, r);
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


size_t trunc_smem(const Dims& d) {
    return sizeof(float) * (size_t)(2 * d.Dv * kRmax + kRmax * d.Dk + d.Dk * (d.Dv + 1));
}

template <int NR>
cudaError_t launch_trunc_t(const Dims& d, const float* S_end, const float* omega, int rank, int iters,
                           float* S_tr, float* Qf, float* Rf, int64_t c, cudaStream_t s) {
    const size_t smem = trunc_smem(d);
    auto kern = trunc_kernel<NR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)d.Hv, (unsigned)d.B), kCThreads, smem, s>>>(d, S_end, omega, rank, iters, S_tr,
                                                                      Qf, Rf, c);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_trunc(const Dims& d, const float* S_end, const float* omega, int rank, int iters,
                         float* S_tr, float* Qf, float* Rf, int64_t c, cudaStream_t s) {
    switch ((d.Dk + 31) / 32) {
        case 1: return launch_trunc_t<1>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 2: return launch_trunc_t<2>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 3: return launch_trunc_t<3>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 4: return launch_trunc_t<4>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 5: return launch_trunc_t<5>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 6: return launch_trunc_t<6>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 7: return launch_trunc_t<7>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
        case 8: return launch_trunc_t<8>(d, S_end, omega, rank, iters, S_tr, Qf, Rf, c, s);
    }
    return cudaErrorInvalidValue;
}

bool compress_supported(const Dims& d, int rank, int iters) {
    return rank >= 1 && rank <= kRmax && iters >= 0 && iters <= 16 && d.Dk % 8 == 0 &&
           d.Dk <= 256 && d.Dv % 4 == 0 && d.Dv <= 256 && trunc_smem(d) <= 227u * 1024u;
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
