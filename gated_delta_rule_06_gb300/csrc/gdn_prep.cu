// gdn_prep.cu -- gate / normalisation prep for the chunked path.
//
// Gates (mlx-lm PR "Add gated_delta_update VJP", "What this PR adds" and
// "Covered corner cases"): per (b, t, h)
//     l = log g = -exp(A_log[h]) * softplus(min(a + dt_bias[h], 20)),  beta = sigmoid(b)
// masked and padded steps become identity steps (l = 0, beta = 0), and
// Gamma = cumulative sum of l inside each 64-step chunk, accumulated and
// stored in fp64 so that Gamma_i - Gamma_j keeps the accuracy of the steps
// between i and j however large |Gamma| grows.
// Norms (torch-to-nnef page, op contract): r = 1 / sqrt(|x|^2 + 1e-6) for
// every query / key row; padded rows get r = 0.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kGateHeads = 8;  // heads per CTA of the gate kernel: one warp each, many CTAs

template <typename TI>
__device__ __forceinline__ void prep_gates_body(const Dims& d, const TI* __restrict__ a,
                                                const TI* __restrict__ b,
                                                const float* __restrict__ A_log,
                                                const float* __restrict__ dt_bias,
                                                const uint8_t* __restrict__ mask,
                                                double* __restrict__ gam,
                                                float* __restrict__ beta, int c, int bb, int hz) {
    __shared__ float lg[kChunk][kGateHeads + 1];
    const int h0 = hz * kGateHeads;
    const int nh = (int)(d.Hv - h0 < kGateHeads ? d.Hv - h0 : kGateHeads);
    const int64_t t0 = (int64_t)c * kChunk;
    for (int idx = threadIdx.x; idx < kChunk * nh; idx += blockDim.x) {
        const int i = idx / nh, hh = idx % nh, h = h0 + hh;
        const int64_t t = t0 + i;
        float l = 0.f, be = 0.f;
        if (t < d.T && (mask == nullptr || mask[bb * d.T + t] != 0)) {
            const int64_t ix = ((int64_t)bb * d.T + t) * d.Hv + h;
            if (d.gates == 1) {  // given log_decay and beta
                l = ldf(a + ix);
                be = ldf(b + ix);
            } else {
                const float x = ldf(a + ix) + dt_bias[h];
                const float xc = fminf(x, kSoftplusClamp);
                l = -expf(A_log[h]) * log1pf(expf(xc));
                be = 1.f / (1.f + expf(-ldf(b + ix)));
            }
        }
        lg[i][hh] = l;
        beta[((int64_t)bb * d.Hv + h) * d.Tp + t] = be;
    }
    __syncthreads();
    // in-chunk inclusive prefix sum, one warp per head, 2 steps per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int hh = warp; hh < nh; hh += blockDim.x >> 5) {
        const double x0 = lg[2 * lane][hh], x1 = lg[2 * lane + 1][hh];
        double s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        const double excl = s - (x0 + x1);
        double* g = gam + ((int64_t)bb * d.Hv + h0 + hh) * d.Tp + t0;
        g[2 * lane] = excl + x0;
        g[2 * lane + 1] = excl + x0 + x1;
    }
}

template <typename TI>
__global__ void __launch_bounds__(256) prep_norms_kernel(Dims d, const TI* __restrict__ q,
                                                         const TI* __restrict__ k,
                                                         float* __restrict__ rq,
                                                         float* __restrict__ rk) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;  // over (b, t, j)
    const int64_t nrows = d.B * d.Tp * d.Hk;
    if (row >= nrows) return;
    const int64_t j = row % d.Hk;
    const int64_t t = (row / d.Hk) % d.Tp;
    const int64_t bb = row / (d.Hk * d.Tp);
    float r_q = 0.f, r_k = 0.f;
    if (t < d.T) {
        const int64_t base = ((bb * d.T + t) * d.Hk + j) * d.Dk;
        float sq = 0.f, sk = 0.f;
        for (int64_t i = lane; i < d.Dk; i += 32) {
            const float xq = ldf(q + base + i), xk = ldf(k + base + i);
            sq = fmaf(xq, xq, sq);
            sk = fmaf(xk, xk, sk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
        }
        r_q = 1.f / sqrtf(sq + kNormEps);
        r_k = 1.f / sqrtf(sk + kNormEps);
    }
    if (lane == 0) {
        rq[(bb * d.Hk + j) * d.Tp + t] = r_q;
        rk[(bb * d.Hk + j) * d.Tp + t] = r_k;
    }
}

// Tensor-core path: the same norms, and the raw bf16 rows copied into the
// per-chunk panel images (piece g of row t of chunk c at byte g * 1024 +
// (t % 64) * 16 of image (b, j, c); rows past T are zero).  One CTA per (chunk,
// key head, batch): the chunk's q and k rows load with row-contiguous 16-byte
// reads into shared memory in the images' panel order, each 64-row panel padded
// by 16 bytes so that the staging writes and the reads below are conflict-free;
// the norms come from shared memory; each image leaves with contiguous stores.
constexpr int kPanelPad = kChunk * 16 + 16;  // bytes per staged 64-row panel

__device__ __forceinline__ void prep_norms_img_body(const Dims& d, const __nv_bfloat16* __restrict__ q,
                                                    const __nv_bfloat16* __restrict__ k,
                                                    float* __restrict__ rq, float* __restrict__ rk,
                                                    uint8_t* __restrict__ qimg,
                                                    uint8_t* __restrict__ kimg, int c, int j, int bb) {
    extern __shared__ __align__(16) uint8_t stage[];  // 2 * (Dk / 8) panels
    const int tid = threadIdx.x;
    const int ng = (int)(d.Dk / 8);  // 16-byte pieces per row
    uint8_t* sq = stage;
    uint8_t* sk = stage + ng * kPanelPad;
    const int64_t t0 = (int64_t)c * kChunk;
    // a thread's row pieces go in rounds of 4 of q and 4 of k, each round's loads
    // issued before its stores so that they are in flight together
    constexpr int kPer = 4;
    for (int e0 = tid; e0 < kChunk * ng; e0 += kPer * 256) {
        uint4 uq[kPer], uk[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {  // row r = e / ng, piece g = e % ng
            const int e = e0 + u * 256;
            uq[u] = uk[u] = make_uint4(0u, 0u, 0u, 0u);
            if (e < kChunk * ng) {
                const int r = e / ng, g = e - (e / ng) * ng;
                const int64_t t = t0 + r;
                if (t < d.T) {
                    const int64_t base = (((int64_t)bb * d.T + t) * d.Hk + j) * d.Dk + 8 * g;
                    uq[u] = *reinterpret_cast<const uint4*>(q + base);
                    uk[u] = *reinterpret_cast<const uint4*>(k + base);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = e0 + u * 256;
            if (e < kChunk * ng) {
                const int r = e / ng, g = e - (e / ng) * ng;
                *reinterpret_cast<uint4*>(sq + g * kPanelPad + r * 16) = uq[u];
                *reinterpret_cast<uint4*>(sk + g * kPanelPad + r * 16) = uk[u];
            }
        }
    }
    __syncthreads();
    if (tid < 2 * kChunk) {  // thread r: row r of q; thread 64 + r: row r of k
        const int r = tid & (kChunk - 1);
        const uint8_t* src = tid < kChunk ? sq : sk;
        float sum = 0.f;
        for (int g = 0; g < ng; ++g) {
            const uint4 u = *reinterpret_cast<const uint4*>(src + g * kPanelPad + r * 16);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h2[i]);
                sum = fmaf(f.x, f.x, sum);
                sum = fmaf(f.y, f.y, sum);
            }
        }
        const int64_t t = t0 + r;
        (tid < kChunk ? rq : rk)[((int64_t)bb * d.Hk + j) * d.Tp + t] = t < d.T ? 1.f / sqrtf(sum + kNormEps) : 0.f;
    }
    const int64_t ioff = (((int64_t)bb * d.Hk + j) * d.NC + c) * kChunk * d.Dk * 2;
    for (int e = tid; e < kChunk * ng; e += blockDim.x) {  // piece g = e / 64, row r = e % 64
        const int g = e >> 6, r = e & (kChunk - 1);
        *reinterpret_cast<uint4*>(qimg + ioff + (int64_t)e * 16) =
            *reinterpret_cast<const uint4*>(sq + g * kPanelPad + r * 16);
        *reinterpret_cast<uint4*>(kimg + ioff + (int64_t)e * 16) =
            *reinterpret_cast<const uint4*>(sk + g * kPanelPad + r * 16);
    }
}

template <typename TI>
__global__ void __launch_bounds__(256) prep_gates_kernel(Dims d, Ptrs p) {
    prep_gates_body<TI>(d, (const TI*)p.a, (const TI*)p.b, p.A_log, p.dt_bias, p.mask, p.gam,
                        p.beta, blockIdx.x, blockIdx.y, blockIdx.z);
}

// The tensor-core path's prep in one launch: one CTA per (chunk, key head j,
// batch) takes the q / k norms and images of its chunk and the gate blocks
// (chunk, batch, value heads 8 hz .. 8 hz + 7) for hz = j, j + Hk, ...  Every
// CTA of the launch reserves the images' staging, so the gates ride along in
// the image CTAs instead of taking CTAs (and staging) of their own.
__global__ void __launch_bounds__(256) prep_tc_kernel(Dims d, Ptrs p) {
    const int64_t r = blockIdx.x;  // (chunk, key head, batch)
    const int c = (int)(r % d.NC), j = (int)((r / d.NC) % d.Hk), bb = (int)(r / (d.NC * d.Hk));
    const int nhz = (int)((d.Hv + kGateHeads - 1) / kGateHeads);
    for (int hz = j; hz < nhz; hz += (int)d.Hk) {
        prep_gates_body<__nv_bfloat16>(d, (const __nv_bfloat16*)p.a, (const __nv_bfloat16*)p.b,
                                       p.A_log, p.dt_bias, p.mask, p.gam, p.beta, c, bb, hz);
        __syncthreads();  // the gate body's shared sums are reused
    }
    prep_norms_img_body(d, (const __nv_bfloat16*)p.q, (const __nv_bfloat16*)p.k, p.rq, p.rk,
                        static_cast<uint8_t*>(p.qimg), static_cast<uint8_t*>(p.kimg), c, j, bb);
}

template <typename TI>
cudaError_t launch_prep_t(const Dims& d, const Ptrs& p, cudaStream_t s) {
    if (tc_path(d)) {
        const int smem = (int)(2 * (d.Dk / 8) * kPanelPad);
        cudaError_t e = cudaFuncSetAttribute(prep_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        prep_tc_kernel<<<(unsigned)(d.NC * d.Hk * d.B), 256, smem, s>>>(d, p);
        count_launches(1);
        return cudaPeekAtLastError();
    }
    dim3 g1((unsigned)d.NC, (unsigned)d.B, (unsigned)((d.Hv + kGateHeads - 1) / kGateHeads));
    prep_gates_kernel<TI><<<g1, 256, 0, s>>>(d, p);
    const int64_t rows = d.B * d.Tp * d.Hk;
    prep_norms_kernel<TI><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(d, (const TI*)p.q,
                                                                     (const TI*)p.k, p.rq, p.rk);
    count_launches(2);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_prep_norms(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const unsigned nblk = (unsigned)((d.B * d.Tp * d.Hk + 7) / 8);
    if (d.dtype == 1)
        prep_norms_kernel<__nv_bfloat16><<<nblk, 256, 0, s>>>(d, (const __nv_bfloat16*)p.q,
                                                             (const __nv_bfloat16*)p.k, p.rq, p.rk);
    else
        prep_norms_kernel<float><<<nblk, 256, 0, s>>>(d, (const float*)p.q, (const float*)p.k,
                                                     p.rq, p.rk);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_prep(const Dims& d, const Ptrs& p, cudaStream_t s) {
    return d.dtype == 1 ? launch_prep_t<__nv_bfloat16>(d, p, s) : launch_prep_t<float>(d, p, s);
}

}  // namespace gdn
