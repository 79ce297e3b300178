// gdn_decode.cu -- single-step (T = 1) forward: the recurrent step of the
// gated delta rule fused with the q / k L2 norms and the gates (mlx-lm PR
// "Add gated_delta_update VJP", "Extension 2 - Inference kernel fusion",
// describes the same fusion for a Metal T = 1 kernel).
//
// Per (b, h), with S the fp32 state (Dk x Dv), read from HBM exactly once:
//     p = S^T kh,  r = S^T qh                       (one pass over S)
//     delta = beta (v - g p)
//     o = g r + delta <kh, qh>                      (= S'^T qh)
//     S' = g S + kh delta^T                         (written once)
// A masked step is the identity (g = 1, beta = 0).  The kernel is bound by
// HBM traffic (2 Dk Dv 4 bytes per head); it uses 16-byte vector loads and
// stores, warp shuffles and one shared-memory exchange, no tensor cores.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 512;
constexpr int kDecodeRows = 16;  // max state rows per thread (held in registers)

template <typename TI>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(Dims d, Ptrs p) {
    extern __shared__ float sm[];
    const int h = blockIdx.x, bb = blockIdx.y;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int ncg = Dv / 4;                   // float4 column groups
    const int R = kDecodeThreads / ncg;       // row groups
    float* qh = sm;                           // [Dk]
    float* kh = qh + Dk;                      // [Dk]
    float* pr = kh + Dk;                      // [R][Dv] partial S^T k
    float* rr = pr + R * Dv;                  // [R][Dv] partial S^T q
    float* red = rr + R * Dv;                 // [64] scalars

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const TI* q = (const TI*)p.q + ((int64_t)bb * d.Hk + j) * Dk;
    const TI* k = (const TI*)p.k + ((int64_t)bb * d.Hk + j) * Dk;
    // L2 norms of q and k (warp 0 and warp 1), gates (warp 2)
    if (warp < 2) {
        const TI* x = warp == 0 ? q : k;
        float s = 0.f;
        for (int i = lane; i < Dk; i += 32) {
            const float v = ldf(x + i);
            s = fmaf(v, v, s);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) red[warp] = 1.f / sqrtf(s + kNormEps);
    } else if (warp == 2 && lane == 0) {
        const bool on = p.mask == nullptr || p.mask[bb] != 0;
        float g = 1.f, be = 0.f;
        if (on) {
            const int64_t ix = (int64_t)bb * d.Hv + h;
            const float x = ldf((const TI*)p.a + ix) + p.dt_bias[h];
            g = expf(-expf(p.A_log[h]) * log1pf(expf(fminf(x, kSoftplusClamp))));
            be = 1.f / (1.f + expf(-ldf((const TI*)p.b + ix)));
        }
        red[2] = g;
        red[3] = be;
    }
    __syncthreads();
    const float qs = red[0] * rsqrtf((float)Dk), ks = red[1];
    for (int i = tid; i < Dk; i += blockDim.x) {
        qh[i] = ldf(q + i) * qs;
        kh[i] = ldf(k + i) * ks;
    }
    __syncthreads();
    const float g = red[2], be = red[3];
    const int cg = tid % ncg, rg = tid / ncg;
    const bool active = rg < R;
    const int64_t sbase = ((int64_t)bb * d.Hv + h) * Dk * Dv;
    const float4* S4 = reinterpret_cast<const float4*>(p.state0 ? p.state0 + sbase : nullptr);
    float4 Sreg[kDecodeRows];
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), rp = pp;
    if (active) {
#pragma unroll
        for (int m = 0; m < kDecodeRows; ++m) {
            const int x = rg + m * R;
            if (x < Dk) {
                const float4 s = p.state0 ? S4[(int64_t)x * ncg + cg] : make_float4(0.f, 0.f, 0.f, 0.f);
                Sreg[m] = s;
                const float kx = kh[x], qx = qh[x];
                pp.x = fmaf(s.x, kx, pp.x); pp.y = fmaf(s.y, kx, pp.y);
                pp.z = fmaf(s.z, kx, pp.z); pp.w = fmaf(s.w, kx, pp.w);
                rp.x = fmaf(s.x, qx, rp.x); rp.y = fmaf(s.y, qx, rp.y);
                rp.z = fmaf(s.z, qx, rp.z); rp.w = fmaf(s.w, qx, rp.w);
            }
        }
        reinterpret_cast<float4*>(pr + rg * Dv)[cg] = pp;
        reinterpret_cast<float4*>(rr + rg * Dv)[cg] = rp;
    }
    // <kh, qh> in warp 0
    if (warp == 0) {
        float s = 0.f;
        for (int i = lane; i < Dk; i += 32) s = fmaf(kh[i], qh[i], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) red[4] = s;
    }
    __syncthreads();
    // column sums over the row groups in fixed order -> delta, o
    for (int c = tid; c < Dv; c += blockDim.x) {
        float ps = 0.f, rs = 0.f;
        for (int r = 0; r < R; ++r) {
            ps += pr[r * Dv + c];
            rs += rr[r * Dv + c];
        }
        const int64_t vo = ((int64_t)bb * d.Hv + h) * Dv + c;
        const float dlt = be * (ldf((const TI*)p.v + vo) - g * ps);
        stf((TI*)p.o + vo, g * rs + dlt * red[4]);
        rr[c] = dlt;  // row 0 of rr is free once every thread has summed it
    }
    __syncthreads();
    if (active) {
        const float4 dv4 = reinterpret_cast<const float4*>(rr)[cg];
        float4* O4 = reinterpret_cast<float4*>(p.state_T + sbase);
#pragma unroll
        for (int m = 0; m < kDecodeRows; ++m) {
            const int x = rg + m * R;
            if (x < Dk) {
                const float kx = kh[x];
                float4 s = Sreg[m];
                s.x = fmaf(g, s.x, kx * dv4.x); s.y = fmaf(g, s.y, kx * dv4.y);
                s.z = fmaf(g, s.z, kx * dv4.z); s.w = fmaf(g, s.w, kx * dv4.w);
                O4[(int64_t)x * ncg + cg] = s;
            }
        }
    }
}

}  // namespace

bool decode_supported(int64_t Dk, int64_t Dv) {
    if (Dv % 4 != 0) return false;
    const int64_t ncg = Dv / 4;
    if (ncg > kDecodeThreads) return false;
    const int64_t R = kDecodeThreads / ncg;
    return (Dk + R - 1) / R <= kDecodeRows;
}

cudaError_t launch_decode(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const int ncg = (int)(d.Dv / 4);
    const int R = kDecodeThreads / ncg;
    const size_t smem = sizeof(float) * (2 * d.Dk + 2 * (size_t)R * d.Dv + 64);
    dim3 grid((unsigned)d.Hv, (unsigned)d.B);
    if (d.dtype == 1) {
        auto kern = decode_kernel<__nv_bfloat16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kDecodeThreads, smem, s>>>(d, p);
    } else {
        auto kern = decode_kernel<float>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kDecodeThreads, smem, s>>>(d, p);
    }
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace gdn
