// gdn_bwd_tc.cu -- per-chunk gradient kernel of the VJP on the tensor cores
// (tcgen05, bf16 operands, fp32 accumulators in TMEM) for bf16 inputs.
//
// Same equations as the CUDA-core version in gdn_bwd.cu (reverse-mode
// derivative of the chunked WY/UT form; mlx-lm PR "Add gated_delta_update
// VJP", "What this PR adds" and "Scope and follow-ups").  One CTA per
// (chunk, value head, batch); every product has the chunk's 64 time rows as
// its M dimension (M = 64 MMAs, accumulator row r in TMEM lane
// 32 (r / 16) + r % 16):
//   phase 0:  Pbar = Obar Delta^T,  Dbar V^T,  Y = T^T Dbar
//   phase 1:  per 32-wide block of Dk:  Obar S^T,  Wbar = -Dbar S^T,  Delta Sbar'^T
//   (Delta, a cancelling difference stored in fp32, enters as two bf16 terms)
//   phase 1b: K K^T, Q K^T, Wbar K^T, Z = T^T Wbar
//   phase 2:  Abar = -(T^T Tbar T^T) and the gate / log-decay cotangents on CUDA
//             cores in fp32 (fp64 for the cancelling row-minus-column sums)
//   phase 3:  (Pbar o M) K  and  (Pbar o M)^T Q + (Gb + Gb^T) K
// q and k are staged as the exact bf16 inputs; the normalisations r_q, r_k
// (and 1/sqrt(Dk)) are applied in fp32 in the epilogues or folded into the
// other operand, so the normalised rows are never rounded.
// Operands are staged from global memory into the canonical no-swizzle
// shared-memory layout (see gdn_tc.cuh); results leave TMEM through 32x32b
// loads, eight warps splitting the columns.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

GDN_ERROR_WORD(bwdtc)

namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int kBlkK = 32;  // Dk block of the state products

struct Smem {
    // byte offsets inside dynamic shared memory
    uint32_t K, Q, W, R1, O, D, Dlo, NB, V, S, Sp, Tt, PMk, PMq, Hk, Pf, Tbf, Gkk, Gqk, Tf, Xf, vec,
        total;
};

__host__ __device__ inline Smem smem_plan(int Dk, int Dv) {
    Smem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    const uint32_t tk = C * Dk * 2, tv = C * Dv * 2;
    s.K = take(tk);
    s.Q = take(tk);
    s.W = take(tk);
    // region R1: Dv-wide operands of phases 0-1, then fp32 scratch of phase 2 and
    // the phase-3 operands
    const uint32_t r1_ops = 6 * tv;
    const uint32_t r1_late = 4 * C * C * 4 + 3 * C * C * 2;
    s.R1 = take(r1_ops > r1_late ? r1_ops : r1_late);
    s.O = s.R1;
    s.D = s.O + tv;
    s.Dlo = s.D + tv;
    s.NB = s.Dlo + tv;
    s.V = s.NB + tv;
    s.S = s.V + tv;              // kBlkK x Dv
    s.Sp = s.S + tv / 2;
    s.Gkk = s.R1;
    s.Gqk = s.Gkk + C * C * 4;
    s.Tf = s.Gqk + C * C * 4;
    s.Xf = s.Tf + C * C * 4;
    s.PMk = s.Xf + C * C * 4;
    s.PMq = s.PMk + C * C * 2;
    s.Hk = s.PMq + C * C * 2;
    s.Tt = take(C * C * 2);
    s.Pf = take(C * C * 4);
    s.Tbf = take(C * C * 4);
    s.vec = take(24 * C * 4 + 4 * C * 8 + 256);
    s.total = o;
    return s;
}

__device__ __forceinline__ void st_bf16x8(uint8_t* dst, const float (&v)[8]) {
    uint4 u;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4], v[5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[6], v[7]);
    u.x = *reinterpret_cast<uint32_t*>(&h0);
    u.y = *reinterpret_cast<uint32_t*>(&h1);
    u.z = *reinterpret_cast<uint32_t*>(&h2);
    u.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(dst) = u;
}

__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void ld8(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// 64-row bf16 tile (x = column) fetched with 16-byte cp.async; rows >= nvalid zero
__device__ __forceinline__ void cpa_tile(uint8_t* tile, const __nv_bfloat16* src, int64_t ld,
                                         int ncols, int nvalid) {
    const int cpr = ncols / 8;
    const uint32_t base = tc::smem_u32(tile);
    const uint32_t ys = (uint32_t)ncols * 16u;
    for (int e = threadIdx.x; e < C * cpr; e += blockDim.x) {
        const int row = e / cpr, cc = e % cpr;
        const bool in = row < nvalid;
        tc::cp_async16(base + cc * 128u + (row >> 3) * ys + (row & 7) * 16u,
                       src + (in ? row : 0) * ld + cc * 8, in ? 16u : 0u);
    }
}

// Stage 64 rows x ncols of an fp32 matrix as bf16 tiles (x = column).  With lo
// != nullptr the value is split into hi + lo (lo = v - bf16(v)).  Loads are
// issued four 8-element chunks deep per thread before any is stored.
__device__ __forceinline__ void stage_f32(uint8_t* hi, uint8_t* lo, const float* src, int64_t ld,
                                          int ncols, float sign) {
    constexpr int U = 4;
    const int cpr = ncols / 8;
    const int total = C * cpr;
    const uint32_t ys = (uint32_t)ncols * 16u;
    for (int base = threadIdx.x; base < total; base += U * blockDim.x) {
        float v[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + u * blockDim.x;
            if (e < total) ld8(src + (e / cpr) * ld + (e % cpr) * 8, v[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + u * blockDim.x;
            if (e < total) {
                const int row = e / cpr, cc = e % cpr;
                const uint32_t o = cc * 128u + (row >> 3) * ys + (row & 7) * 16u;
                float l[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[u][i] *= sign;
                    l[i] = v[u][i] - __bfloat162float(__float2bfloat16_rn(v[u][i]));
                }
                st_bf16x8(hi + o, v[u]);
                if (lo) st_bf16x8(lo + o, l);
            }
        }
    }
}

// read one bf16 element of a canonical tile (x = column)
__device__ __forceinline__ float tile_at(const uint8_t* tile, int ncols, int x, int y) {
    const uint32_t off = (x >> 3) * 128u + (y >> 3) * (uint32_t)ncols * 16u + (y & 7) * 16u + (x & 7) * 2u;
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + off));
}
__device__ __forceinline__ void tile_put(uint8_t* tile, int ncols, int x, int y, float v) {
    const uint32_t off = (x >> 3) * 128u + (y >> 3) * (uint32_t)ncols * 16u + (y & 7) * 16u + (x & 7) * 2u;
    *reinterpret_cast<__nv_bfloat16*>(tile + off) = __float2bfloat16_rn(v);
}

__device__ __forceinline__ tc::Tile kmaj(uint8_t* smem, uint32_t off, int ncols) {
    tc::Tile t;
    t.base = tc::smem_u32(smem + off);
    t.xs = 128;
    t.ys = (uint32_t)ncols * 16u;
    t.k_major = true;
    return t;
}
__device__ __forceinline__ tc::Tile mnmaj(uint8_t* smem, uint32_t off, int ncols) {
    tc::Tile t = kmaj(smem, off, ncols);
    t.k_major = false;
    return t;
}

// Walk an M = 64 accumulator of `ncols` columns at TMEM column col0: eight warps,
// warp w reads rows 16 (w % 4) .. +15 and half (w / 4) of the columns.
template <typename F>
__device__ __forceinline__ void acc_rows(uint32_t tbase, uint32_t col0, int ncols, F&& f) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int sp = w & 3, g = w >> 2;
    const int half = ncols / 2;
    for (int c = g * half; c < (g + 1) * half; c += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_addr(tbase, 32 * sp, col0 + c), v);
        tc::tmem_wait_ld();
        if (l < 16) f(16 * sp + l, c, v);
    }
}

__device__ __forceinline__ void sync_after_mma(uint64_t* bar, uint32_t& phase, bool& ok) {
    ok = tc::mbar_wait(bar, phase, &g_err_bwdtc) && ok;
    phase ^= 1u;
    tc::tc_fence_after();
}

__global__ void __launch_bounds__(kThreads, 1) bwd_chunk_tc_kernel(Dims d, Ptrs p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base_sh;
    const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Smem L = smem_plan(Dk, Dv);
    float* vec = reinterpret_cast<float*>(sm + L.vec);
    float* gm = vec;            // exp(Gamma)
    float* ev = gm + C;         // exp(Gamma_63 - Gamma)
    float* bt = ev + C;         // beta
    float* rqv = bt + C;        // r_q / sqrt(Dk)
    float* rkv = rqv + C;       // r_k
    float* gq = rkv + C;        // [2][64] row-dot partials: gambar * gam
    float* ee = gq + 2 * C;     // [2][64] ebar * e
    float* bb0 = ee + 2 * C;    // [2][64] betabar (Y . V)
    float* zk = bb0 + 2 * C;    // [2][64] Z . K
    float* betab = zk + 2 * C;  // [64]
    float* red = betab + C;     // [256]
    double* Gm = reinterpret_cast<double*>(red + 256);  // [64]
    double* red2 = Gm + C;                              // [64]

    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t gbase = ((int64_t)bb * d.Hv + h) * d.Tp + t0;
    const int64_t rbase = ((int64_t)bb * d.Hk + j) * d.Tp + t0;
    const int64_t cbase = (((int64_t)bb * d.Hv + h) * d.NC + c) * Dk * Dv;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(p.d_o);
    const float* Delta = p.Delta;
    __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(p.dv);

    if (warp == 0) {
        tc::tmem_alloc(&tmem_base_sh, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    for (int i = tid; i < C; i += blockDim.x) {
        const double G = p.gam[gbase + i];
        Gm[i] = G;
        gm[i] = expf((float)G);
        ev[i] = expf((float)(p.gam[gbase + C - 1] - G));
        bt[i] = p.beta[gbase + i];
        rqv[i] = p.rq[rbase + i] * rsqrtf((float)Dk);
        rkv[i] = p.rk[rbase + i];
    }
    for (int i = tid; i < 8 * C; i += blockDim.x) gq[i] = 0.f;  // gq, ee, bb0, zk
    __syncthreads();

    // ---- stage the phase-0/1 operands
    const int64_t ldq = d.Hk * Dk, ldv = d.Hv * Dv;
    // q and k enter as the exact bf16 inputs; their normalisations are applied
    // in fp32 to the other operand or in the epilogues
    cpa_tile(sm + L.K, k + ((int64_t)bb * d.T + t0) * ldq + (int64_t)j * Dk, ldq, Dk, nvalid);
    cpa_tile(sm + L.Q, q + ((int64_t)bb * d.T + t0) * ldq + (int64_t)j * Dk, ldq, Dk, nvalid);
    cpa_tile(sm + L.O, dO + ((int64_t)bb * d.T + t0) * ldv + (int64_t)h * Dv, ldv, Dv, nvalid);
    cpa_tile(sm + L.V, v + ((int64_t)bb * d.T + t0) * ldv + (int64_t)h * Dv, ldv, Dv, nvalid);
    tc::cp_async_commit();
    stage_f32(sm + L.D, sm + L.Dlo, Delta + gbase * Dv, Dv, Dv, 1.f);
    stage_f32(sm + L.NB, nullptr, p.Dbar + gbase * Dv, Dv, Dv, -1.f);
    stage_f32(sm + L.Tt, nullptr, p.Tinv + (((int64_t)bb * d.Hv + h) * d.NC + c) * C * C, C, C, 1.f);
    tc::cp_async_wait_all();
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    uint32_t phase = 0;
    bool ok = true;

    const tc::Tile tK = kmaj(sm, L.K, Dk), tQ = kmaj(sm, L.Q, Dk), tW = kmaj(sm, L.W, Dk);
    const tc::Tile tKmn = mnmaj(sm, L.K, Dk), tQmn = mnmaj(sm, L.Q, Dk), tWmn = mnmaj(sm, L.W, Dk);
    const tc::Tile tO = kmaj(sm, L.O, Dv), tD = kmaj(sm, L.D, Dv), tNB = kmaj(sm, L.NB, Dv);
    const tc::Tile tDlo = kmaj(sm, L.Dlo, Dv);
    const tc::Tile tV = kmaj(sm, L.V, Dv), tNBmn = mnmaj(sm, L.NB, Dv);
    const tc::Tile tTmn = mnmaj(sm, L.Tt, C);

    // ---- phase 0: Pbar = Obar Delta^T | -Dbar V^T | -T^T Dbar
    if (tid == 0) {
        tc::mma_tile(tb + 0, tO, tD, C, C, Dv, false);
        tc::mma_tile(tb + 0, tO, tDlo, C, C, Dv, true);
        tc::mma_tile(tb + 64, tNB, tV, C, C, Dv, false);
        tc::mma_tile(tb + 128, tTmn, tNBmn, C, Dv, C, false);
        tc::mma_commit(&bar);
    }
    sync_after_mma(&bar, phase, ok);
    float* Pf = reinterpret_cast<float*>(sm + L.Pf);
    float* Tbf = reinterpret_cast<float*>(sm + L.Tbf);
    if (ok) {
        acc_rows(tb, 0, C, [&](int r, int c0, const float (&x)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Pf[r * C + c0 + i] = (c0 + i <= r) ? x[i] : 0.f;
        });
        acc_rows(tb, 64, C, [&](int r, int c0, const float (&x)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Tbf[r * C + c0 + i] = -bt[c0 + i] * x[i];
        });
        acc_rows(tb, 128, Dv, [&](int r, int c0, const float (&x)[16]) {
            const int g = warp >> 2;
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) s = fmaf(-x[i], tile_at(sm + L.V, Dv, c0 + i, r), s);
            bb0[g * C + r] += s;
            if (r < nvalid) {
                __nv_bfloat16* dst = dv + ((int64_t)bb * d.T + t0 + r) * ldv + (int64_t)h * Dv + c0;
#pragma unroll
                for (int i = 0; i < 16; i += 2)
                    *reinterpret_cast<__nv_bfloat162*>(dst + i) =
                        __floats2bfloat162_rn(-bt[r] * x[i], -bt[r] * x[i + 1]);
            }
        });
    }

    // ---- phase 1: state products per kBlkK-wide block of Dk.  The fp32 S and
    // Sbar' rows of the next block are loaded into registers while the current
    // block's MMAs run.
    float gcb = 0.f;
    constexpr int kPer = (kBlkK * 256 / 8 + kThreads - 1) / kThreads;  // chunks per thread (Dv <= 256)
    float pre_s[kPer][8], pre_p[kPer][8];
    const int cpr_s = Dv / 8;
    auto load_blk = [&](int dk0, int nk) {
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = tid + u * kThreads;
            if (e < nk * cpr_s) {
                const int64_t off = cbase + (int64_t)(dk0 + e / cpr_s) * Dv + (e % cpr_s) * 8;
                ld8(p.ckpt + off, pre_s[u]);
                ld8(p.dSck + off, pre_p[u]);
            }
        }
    };
    load_blk(0, Dk < kBlkK ? Dk : kBlkK);
    for (int dk0 = 0; dk0 < Dk; dk0 += kBlkK) {
        const int nk = Dk - dk0 < kBlkK ? Dk - dk0 : kBlkK;
        tc::tc_fence_before();
        __syncthreads();  // previous block's TMEM reads and MMAs are done
        {
            const uint32_t ys = (uint32_t)Dv * 16u;
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int e = tid + u * kThreads;
                if (e < nk * cpr_s) {
                    const int row = e / cpr_s, cc = e % cpr_s;
#pragma unroll
                    for (int i = 0; i < 8; ++i) gcb = fmaf(pre_s[u][i], pre_p[u][i], gcb);
                    const uint32_t o = cc * 128u + (row >> 3) * ys + (row & 7) * 16u;
                    st_bf16x8(sm + L.S + o, pre_s[u]);
                    st_bf16x8(sm + L.Sp + o, pre_p[u]);
                }
            }
        }
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
        const tc::Tile tS = kmaj(sm, L.S, Dv), tSp = kmaj(sm, L.Sp, Dv);
        if (tid == 0) {
            tc::mma_tile(tb + 0, tO, tS, C, nk, Dv, false);
            tc::mma_tile(tb + 64, tNB, tS, C, nk, Dv, false);
            tc::mma_tile(tb + 128, tD, tSp, C, nk, Dv, false);
            tc::mma_tile(tb + 128, tDlo, tSp, C, nk, Dv, true);
            tc::mma_commit(&bar);
        }
        if (dk0 + kBlkK < Dk) load_blk(dk0 + kBlkK, Dk - dk0 - kBlkK < kBlkK ? Dk - dk0 - kBlkK : kBlkK);
        sync_after_mma(&bar, phase, ok);
        if (ok) {
            const int g = warp >> 2;
            acc_rows(tb, 0, nk, [&](int r, int c0, const float (&x)[16]) {
                float* dst = p.dqh + (gbase + r) * Dk + dk0 + c0;
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float y = gm[r] * x[i];
                    dst[i] = y;
                    s = fmaf(y, tile_at(sm + L.Q, Dk, dk0 + c0 + i, r), s);
                }
                gq[g * C + r] += s;
            });
            acc_rows(tb, 64, nk, [&](int r, int c0, const float (&x)[16]) {
#pragma unroll
                for (int i = 0; i < 16; ++i) tile_put(sm + L.W, Dk, dk0 + c0 + i, r, x[i]);
            });
            acc_rows(tb, 128, nk, [&](int r, int c0, const float (&x)[16]) {
                float* dst = p.dkh + (gbase + r) * Dk + dk0 + c0;
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float y = ev[r] * x[i];
                    dst[i] = y;
                    s = fmaf(y, tile_at(sm + L.K, Dk, dk0 + c0 + i, r), s);
                }
                ee[g * C + r] += s;
            });
        }
    }
    // <Sbar', S> over the whole state: fixed-order block reduction
    red[tid] = gcb;
    tc::fence_async_smem();  // Wbar tile written by generic stores -> MMA operand
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- phase 1b: K K^T | Q K^T | Wbar K^T | Z = T^T Wbar
    if (tid == 0) {
        tc::mma_tile(tb + 0, tK, tK, C, C, Dk, false);
        tc::mma_tile(tb + 64, tQ, tK, C, C, Dk, false);
        tc::mma_tile(tb + 128, tW, tK, C, C, Dk, false);
        tc::mma_tile(tb + 192, tTmn, tWmn, C, Dk, C, false);
        tc::mma_commit(&bar);
    }
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    const float gCb = red[0];
    sync_after_mma(&bar, phase, ok);
    float* Gkk = reinterpret_cast<float*>(sm + L.Gkk);
    float* Gqk = reinterpret_cast<float*>(sm + L.Gqk);
    float* Tf = reinterpret_cast<float*>(sm + L.Tf);
    float* Xf = reinterpret_cast<float*>(sm + L.Xf);
    if (ok) {
        acc_rows(tb, 0, C, [&](int r, int c0, const float (&x)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Gkk[r * C + c0 + i] = rkv[r] * rkv[c0 + i] * x[i];
        });
        acc_rows(tb, 64, C, [&](int r, int c0, const float (&x)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Gqk[r * C + c0 + i] = rqv[r] * rkv[c0 + i] * x[i];
        });
        acc_rows(tb, 128, C, [&](int r, int c0, const float (&x)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                Tbf[r * C + c0 + i] += bt[c0 + i] * gm[c0 + i] * rkv[c0 + i] * x[i];
        });
        acc_rows(tb, 192, Dk, [&](int r, int c0, const float (&x)[16]) {
            const int g = warp >> 2;
            float* dst = p.dkh + (gbase + r) * Dk + c0;
            const float sc = bt[r] * gm[r];
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                dst[i] += sc * x[i];
                s = fmaf(x[i], tile_at(sm + L.K, Dk, c0 + i, r), s);
            }
            zk[g * C + r] += s;
        });
    }
    const float* Tg = p.Tinv + (((int64_t)bb * d.Hv + h) * d.NC + c) * C * C;
    for (int i = tid; i < C * C / 4; i += blockDim.x)
        reinterpret_cast<float4*>(Tf)[i] = reinterpret_cast<const float4*>(Tg)[i];
    __syncthreads();
    if (tid < C) {
        const int i = tid;
        betab[i] = bb0[i] + bb0[C + i];
        const float z = rkv[i] * (zk[i] + zk[C + i]);  // <Z_i, k_hat_i>
        betab[i] += gm[i] * z;
        gq[i] = rqv[i] * (gq[i] + gq[C + i]) + bt[i] * z * gm[i];  // gambar * gam
        ee[i] = rkv[i] * (ee[i] + ee[C + i]);                      // ebar * e
    }

    // ---- phase 2: Abar = -(T^T Tbar T^T), gate / log-decay cotangents
    cta_gemm<4, 4>(C, C, C, Tbf, C, 1, Tf, 1, C, Xf, C, 1.f, 0.f, nullptr);
    __syncthreads();
    cta_gemm<4, 4>(C, C, C, Tf, 1, C, Xf, C, 1, Tbf, C, -1.f, 0.f, nullptr);
    __syncthreads();
    if (tid < C) {
        const int i = tid;
        float sb = 0.f;
        for (int jj = 0; jj < C; ++jj) {
            const int idx = i * C + jj;
            const float m = jj <= i ? expf((float)(Gm[i] - Gm[jj])) : 0.f;
            const float ab = jj < i ? Tbf[idx] : 0.f;
            const float mb = ab * bt[i] * Gkk[idx] + Pf[idx] * Gqk[idx];
            sb = fmaf(ab * m, Gkk[idx], sb);
            Xf[idx] = mb * m;
            Tbf[idx] = ab * bt[i] * m;
            const float pm = Pf[idx] * m;
            Pf[idx] = pm;
            tile_put(sm + L.PMk, C, jj, i, pm * rkv[jj]);
            tile_put(sm + L.PMq, C, jj, i, pm * rqv[i]);
        }
        betab[i] += sb;
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int i = idx / C, jj = idx % C;
        tile_put(sm + L.Hk, C, jj, i, (Tbf[idx] + Tbf[jj * C + i]) * rkv[jj]);
    }
    if (tid < C) {
        const int i = tid;
        double rsum = 0.0, csum = 0.0;
        for (int jj = 0; jj < C; ++jj) {
            rsum += (double)Xf[i * C + jj];
            csum += (double)Xf[jj * C + i];
        }
        red2[i] = rsum - csum + (double)gq[i] - (double)ee[i];
    }
    tc::fence_async_smem();  // PM / H tiles -> MMA operands
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- phase 3: dQ += (Pbar o M) K;  dK += (Pbar o M)^T Q + (Gb + Gb^T) K
    const tc::Tile tPMk = kmaj(sm, L.PMk, C), tPMqmn = mnmaj(sm, L.PMq, C), tHk = kmaj(sm, L.Hk, C);
    if (tid == 0) {
        tc::mma_tile(tb + 0, tPMk, tKmn, C, Dk, C, false);
        tc::mma_tile(tb + Dk, tPMqmn, tQmn, C, Dk, C, false);
        tc::mma_tile(tb + Dk, tHk, tKmn, C, Dk, C, true);
        tc::mma_commit(&bar);
    }
    if (tid == 0) {
        double se = 0.0;
        for (int i = 0; i < C; ++i) se += (double)ee[i];
        red2[C - 1] += (double)gCb * gm[C - 1] + se;
        double run = 0.0;
        for (int i = C - 1; i >= 0; --i) {
            run += red2[i];
            red2[i] = run;
        }
    }
    __syncthreads();
    if (tid < C) {
        p.dl[gbase + tid] = (float)red2[tid];
        p.dbeta[gbase + tid] = betab[tid];
    }
    sync_after_mma(&bar, phase, ok);
    if (ok) {
        acc_rows(tb, 0, Dk, [&](int r, int c0, const float (&x)[16]) {
            float* dst = p.dqh + (gbase + r) * Dk + c0;
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[i] += x[i];
        });
        acc_rows(tb, Dk, Dk, [&](int r, int c0, const float (&x)[16]) {
            float* dst = p.dkh + (gbase + r) * Dk + c0;
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[i] += x[i];
        });
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 512);
    (void)lane;
}

}  // namespace

bool bwd_chunk_tc_supported(const Dims& d) {
    if (d.dtype != 1) return false;
    if (d.Dk % 32 || d.Dv % 32 || d.Dk > 256 || d.Dv > 256) return false;
    return smem_plan((int)d.Dk, (int)d.Dv).total + 2048 <= 227u * 1024u;
}

cudaError_t launch_bwd_chunk_tc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const Smem L = smem_plan((int)d.Dk, (int)d.Dv);
    const size_t smem = L.total + 1024;  // slack for the 1024-byte alignment of the base
    auto kern = bwd_chunk_tc_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads, smem, s>>>(d, p);
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace gdn
