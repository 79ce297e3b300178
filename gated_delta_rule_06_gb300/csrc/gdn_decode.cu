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
// HBM traffic (2 Dk Dv 4 bytes per head).  One CTA per (b, h): a single bulk
// copy brings the head's state into shared memory while the norms and gates
// are computed, the step runs out of shared memory (16-byte accesses, warp
// shuffles), and a single bulk store writes the new state back.  Shared
// memory, not registers, holds the state, so several CTAs share an SM and
// keep enough bytes in flight.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

GDN_ERROR_WORD(decode)

namespace {

constexpr int kDecThreads = 256;

struct DecPlan {
    int ncg, R;           // float4 column groups, row groups
    size_t S, qh, kh, xv, pr, rr, red, total;
};
__host__ __device__ inline DecPlan dec_plan(int Dk, int Dv) {
    DecPlan pl{};
    pl.ncg = Dv / 4;
    pl.R = kDecThreads / pl.ncg;
    size_t o = 0;
    pl.S = o;   o += (size_t)Dk * Dv * 4;
    pl.qh = o;  o += (size_t)Dk * 4;
    pl.kh = o;  o += (size_t)Dk * 4;
    pl.xv = o;  o += (size_t)Dv * 4;  // v after the short convolution (fused form)
    pl.pr = o;  o += (size_t)pl.R * Dv * 4;  // partial S^T kh per row group
    pl.rr = o;  o += (size_t)pl.R * Dv * 4;  // partial S^T qh per row group
    pl.red = o; o += 64 * 4;
    pl.total = o;
    return pl;
}

// Fused form: the short convolution in front of the recurrence (see
// gdn_conv.cu) runs first for the channels this head reads.  The mixed
// projection `hidden` [B, C] (C = 2 Hk Dk + Hv Dv) holds q | k | v, each
// head-major; each channel's K carried samples and its new sample give
// SiLU(sum_i w_i x_{1+i}) and the shifted window is the new carried state,
// written to a separate buffer (the G value heads of a key head read the same
// q / k channels) by one CTA per channel.  A masked row keeps its carried state.
// four consecutive elements as floats, one vector access (16-byte aligned for
// fp32, 8-byte for bf16)
__device__ __forceinline__ void ld4v(const float* p, float* v) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void ld4v(const __nv_bfloat16* p, float* v) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void st4v(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st4v(__nv_bfloat16* p, const float* v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

struct ConvArgs {
    const void* hidden;      // [B, C]
    const void* conv_state;  // [B, C, K]
    const void* weight;      // [C, K]
    void* final_state;       // [B, C, K]
    int64_t C;
    int K;
};

template <typename TI, bool kConv>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(Dims d, Ptrs p, ConvArgs ca) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ uint64_t bar;
    const int h = blockIdx.x, bb = blockIdx.y;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const DecPlan pl = dec_plan(Dk, Dv);
    const int ncg = pl.ncg, R = pl.R;
    float* S = reinterpret_cast<float*>(dsm + pl.S);
    float* qh = reinterpret_cast<float*>(dsm + pl.qh);
    float* kh = reinterpret_cast<float*>(dsm + pl.kh);
    float* xv = reinterpret_cast<float*>(dsm + pl.xv);
    float* pr = reinterpret_cast<float*>(dsm + pl.pr);
    float* rr = reinterpret_cast<float*>(dsm + pl.rr);
    float* red = reinterpret_cast<float*>(dsm + pl.red);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t sbase = ((int64_t)bb * d.Hv + h) * Dk * Dv;
    const uint32_t sbytes = (uint32_t)Dk * (uint32_t)Dv * 4u;

    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (p.state0) {
        if (tid == 0) {  // the whole state of the head, in flight during the prelude
            tc::mbar_arrive_expect_tx(&bar, sbytes);
            tc::bulk_g2s(S, p.state0 + sbase, sbytes, &bar);
        }
    } else {
        for (int i = tid; i < Dk * Dv / 4; i += kDecThreads)
            reinterpret_cast<float4*>(S)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const bool on = p.mask == nullptr || p.mask[bb] != 0;
    const TI* q = (const TI*)p.q + ((int64_t)bb * d.Hk + j) * Dk;
    const TI* k = (const TI*)p.k + ((int64_t)bb * d.Hk + j) * Dk;
    if constexpr (kConv) {
        // q, k (key head j) and v (value head h) channels through the convolution,
        // raw outputs into qh, kh, xv
        const int nch = 2 * Dk + Dv;
        const int64_t HkDk = d.Hk * (int64_t)Dk;
        auto chan = [&](int idx) -> int64_t {
            return idx < Dk ? j * (int64_t)Dk + idx
                 : idx < 2 * Dk ? HkDk + j * (int64_t)Dk + (idx - Dk)
                                : 2 * HkDk + (int64_t)h * Dv + (idx - 2 * Dk);
        };
        float* outs[3] = {qh, kh, xv};
        int first = 0;
        if (ca.K == 4) {
            // the common kernel length: two channels per thread with all their
            // loads in flight before either is used, one vector access per row
            for (int base = 0; base < nch; base += 2 * kDecThreads) {
                float wv[2][4], sv[2][4], xn[2];
                int64_t chs[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int idx = base + tid + u * kDecThreads;
                    chs[u] = idx < nch ? chan(idx) : -1;
                    if (chs[u] >= 0) {
                        ld4v((const TI*)ca.weight + chs[u] * 4, wv[u]);
                        ld4v((const TI*)ca.conv_state + ((int64_t)bb * ca.C + chs[u]) * 4, sv[u]);
                        xn[u] = ldf((const TI*)ca.hidden + (int64_t)bb * ca.C + chs[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int idx = base + tid + u * kDecThreads;
                    if (chs[u] < 0) continue;
                    const float nv[4] = {sv[u][1], sv[u][2], sv[u][3], xn[u]};
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc = fmaf(wv[u][i], nv[i], acc);
                    const int sel = idx < Dk ? 0 : idx < 2 * Dk ? 1 : 2;
                    outs[sel][idx - sel * Dk] = acc / (1.f + expf(-acc));
                    if (idx >= 2 * Dk || h % (int)d.G == 0)  // one writer per channel
                        st4v((TI*)ca.final_state + ((int64_t)bb * ca.C + chs[u]) * 4,
                             on ? nv : sv[u]);
                }
            }
            first = nch;  // done
        }
        for (int idx = first + tid; idx < nch; idx += kDecThreads) {
            const int64_t ch = idx < Dk ? j * (int64_t)Dk + idx
                             : idx < 2 * Dk ? HkDk + j * (int64_t)Dk + (idx - Dk)
                                            : 2 * HkDk + (int64_t)h * Dv + (idx - 2 * Dk);
            const TI* st = (const TI*)ca.conv_state + ((int64_t)bb * ca.C + ch) * ca.K;
            const TI* w = (const TI*)ca.weight + ch * ca.K;
            const float xn = ldf((const TI*)ca.hidden + (int64_t)bb * ca.C + ch);
            TI* fs = (TI*)ca.final_state + ((int64_t)bb * ca.C + ch) * ca.K;
            const bool writer = idx >= 2 * Dk || h % (int)d.G == 0;  // one per channel
            // every load of the channel in flight at once (predicated up to the
            // longest kernel), then the taps
            float wv[kConvMaxK], sv[kConvMaxK];
#pragma unroll
            for (int i = 0; i < kConvMaxK; ++i) {
                wv[i] = i < ca.K ? ldf(w + i) : 0.f;
                sv[i] = i < ca.K ? ldf(st + i) : 0.f;
            }
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kConvMaxK; ++i)
                if (i < ca.K) acc = fmaf(wv[i], i + 1 < ca.K ? sv[i < kConvMaxK - 1 ? i + 1 : i] : xn, acc);
            const float y = acc / (1.f + expf(-acc));
            (idx < Dk ? qh : idx < 2 * Dk ? kh : xv)[idx < Dk ? idx : idx < 2 * Dk ? idx - Dk : idx - 2 * Dk] = y;
            if (writer) {
#pragma unroll
                for (int i = 0; i < kConvMaxK; ++i)
                    if (i < ca.K)
                        stf(fs + i, on ? (i + 1 < ca.K ? sv[i < kConvMaxK - 1 ? i + 1 : i] : xn) : sv[i]);
            }
        }
        __syncthreads();
    }
    // L2 norms of q and k (warps 0 and 1), gates (warp 2)
    if (warp < 2) {
        float s = 0.f;
        for (int i = lane; i < Dk; i += 32) {
            const float v = kConv ? (warp == 0 ? qh : kh)[i] : ldf((warp == 0 ? q : k) + i);
            s = fmaf(v, v, s);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) red[warp] = 1.f / sqrtf(s + kNormEps);
    } else if (warp == 2 && lane == 0) {
        float g = 1.f, be = 0.f;
        if (on) {
            const int64_t ix = (int64_t)bb * d.Hv + h;
            if (d.gates == 1) {  // given log_decay and beta
                g = expf(ldf((const TI*)p.a + ix));
                be = ldf((const TI*)p.b + ix);
            } else {
                const float x = ldf((const TI*)p.a + ix) + p.dt_bias[h];
                g = expf(-expf(p.A_log[h]) * log1pf(expf(fminf(x, kSoftplusClamp))));
                be = 1.f / (1.f + expf(-ldf((const TI*)p.b + ix)));
            }
        }
        red[2] = g;
        red[3] = be;
    }
    __syncthreads();
    const float qs = red[0] * rsqrtf((float)Dk), ks = red[1];
    for (int i = tid; i < Dk; i += kDecThreads) {
        qh[i] = (kConv ? qh[i] : ldf(q + i)) * qs;
        kh[i] = (kConv ? kh[i] : ldf(k + i)) * ks;
    }
    __syncthreads();
    const float g = red[2], be = red[3];
    bool ok = true;
    if (p.state0) ok = tc::mbar_wait(&bar, 0, &g_err_decode);
    const int cg = tid % ncg, rg = tid / ncg;
    const bool active = rg < R;
    float4* S4 = reinterpret_cast<float4*>(S);
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), rp = pp;
    if (active) {
        for (int x = rg; x < Dk; x += R) {
            const float4 s = S4[x * ncg + cg];
            const float kx = kh[x], qx = qh[x];
            pp.x = fmaf(s.x, kx, pp.x); pp.y = fmaf(s.y, kx, pp.y);
            pp.z = fmaf(s.z, kx, pp.z); pp.w = fmaf(s.w, kx, pp.w);
            rp.x = fmaf(s.x, qx, rp.x); rp.y = fmaf(s.y, qx, rp.y);
            rp.z = fmaf(s.z, qx, rp.z); rp.w = fmaf(s.w, qx, rp.w);
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
    for (int c = tid; c < Dv; c += kDecThreads) {
        float ps = 0.f, rs = 0.f;
        for (int r = 0; r < R; ++r) {
            ps += pr[r * Dv + c];
            rs += rr[r * Dv + c];
        }
        const int64_t vo = ((int64_t)bb * d.Hv + h) * Dv + c;
        const float vc = kConv ? xv[c] : ldf((const TI*)p.v + vo);
        const float dlt = be * (vc - g * ps);
        stf((TI*)p.o + vo, g * rs + dlt * red[4]);
        rr[c] = dlt;  // row 0 of rr: only this thread reads column c
    }
    __syncthreads();
    if (active) {
        const float4 dv4 = reinterpret_cast<const float4*>(rr)[cg];
        for (int x = rg; x < Dk; x += R) {
            const float kx = kh[x];
            float4 s = S4[x * ncg + cg];
            s.x = fmaf(g, s.x, kx * dv4.x); s.y = fmaf(g, s.y, kx * dv4.y);
            s.z = fmaf(g, s.z, kx * dv4.z); s.w = fmaf(g, s.w, kx * dv4.w);
            S4[x * ncg + cg] = s;
        }
    }
    tc::fence_async_smem();  // the new state, written by plain stores -> the bulk store
    __syncthreads();
    if (tid == 0 && ok) {
        tc::bulk_s2g(p.state_T + sbase, S, sbytes);
        tc::bulk_commit();
        tc::bulk_wait_all();
    }
}

}  // namespace

bool decode_supported(int64_t Dk, int64_t Dv) {
    if (Dv % 4 != 0 || Dv / 4 > kDecThreads || kDecThreads % (Dv / 4) != 0) return false;
    return dec_plan((int)Dk, (int)Dv).total + 1024 <= 227u * 1024u;
}

template <typename TI, bool kConv>
cudaError_t launch_decode_t(const Dims& d, const Ptrs& p, const ConvArgs& ca, cudaStream_t s) {
    const size_t smem = dec_plan((int)d.Dk, (int)d.Dv).total;
    auto kern = decode_kernel<TI, kConv>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)d.Hv, (unsigned)d.B), kDecThreads, smem, s>>>(d, p, ca);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_decode(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const ConvArgs none{};
    return d.dtype == 1 ? launch_decode_t<__nv_bfloat16, false>(d, p, none, s)
                        : launch_decode_t<float, false>(d, p, none, s);
}

cudaError_t launch_decode_conv(const Dims& d, const Ptrs& p, const void* hidden,
                               const void* conv_state, const void* weight, void* final_state,
                               int K, cudaStream_t s) {
    const ConvArgs ca{hidden, conv_state, weight, final_state,
                      2 * d.Hk * d.Dk + d.Hv * d.Dv, K};
    return d.dtype == 1 ? launch_decode_t<__nv_bfloat16, true>(d, p, ca, s)
                        : launch_decode_t<float, true>(d, p, ca, s);
}

}  // namespace gdn
