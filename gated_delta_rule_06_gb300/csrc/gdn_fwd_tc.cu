// gdn_fwd_tc.cu -- chunk-local WY/UT products of the forward on the tensor
// cores (tcgen05, bf16 operands, fp32 accumulators in TMEM) for bf16 inputs.
//
// Per (chunk, value head, batch), with raw q, k (panel images written by prep), v (mlx-lm PR "Add
// gated_delta_update VJP", "Scope and follow-ups": chunk-parallel form through a
// lower-triangular solve; torch-to-nnef "custom_extractors/gdn": the chunked
// rule equals the recurrent one):
//   K K^T, Q K^T                 (M = 64 MMAs; norms and 1/sqrt(Dk) applied in fp32)
//   A_ij = beta_i M_ij <k_i, k_j>  (j < i),   P_ij = M_ij <q_i, k_j>  (j <= i)
//   T = (I + A)^-1               blocked forward substitution in fp32 (16 x 16 blocks)
//   W = T diag(beta gam r_k) K,   U = T diag(beta) V
// T enters the W / U products as two bf16 terms (hi + lo) so that U keeps fp32
// accuracy (the forward state update subtracts W S from U).  Outputs: T, P and
// W as bf16 panel images (the operand layout of the scans and the gradient
// kernel), U row-major in fp32.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"
#include "gdn_tri.cuh"

namespace gdn {

GDN_ERROR_WORD(fwdtc)

namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int kTmemCols = 256;  // half the TMEM: two CTAs per SM

__device__ __forceinline__ uint32_t canon(int x, int y, int ncols) {
    return (uint32_t)(x >> 3) * 128u + (uint32_t)(y >> 3) * (uint32_t)ncols * 16u +
           (uint32_t)(y & 7) * 16u + (uint32_t)(x & 7) * 2u;
}

__device__ __forceinline__ void st_bf16x8(uint8_t* dst, const float* v) {
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

__device__ __forceinline__ void cpa_tile(uint8_t* tile, const __nv_bfloat16* src, int64_t ld,
                                         int ncols, int nvalid) {
    const int cpr = ncols / 8;
    const uint32_t base = tc::smem_u32(tile);
    for (int e = threadIdx.x; e < C * cpr; e += blockDim.x) {
        int row, cc;
        chunk_rc(e, cpr, row, cc);
        const bool in = row < nvalid;
        tc::cp_async16(base + canon(cc * 8, row, ncols), src + (in ? row : 0) * ld + cc * 8,
                       in ? 16u : 0u);
    }
}

__device__ __forceinline__ tc::Tile tile_of(uint8_t* p, int ncols, bool k_major) {
    tc::Tile t;
    t.base = tc::smem_u32(p);
    t.xs = 128;
    t.ys = (uint32_t)ncols * 16u;
    t.k_major = k_major;
    return t;
}

// M = 64 accumulator walk with every lane busy: 32-column pieces taken in turn
// by the two warp groups g = w / 4; in a piece at column c, lane l < 16 of warp
// w reads row 16 (w % 4) + l at columns c .. c + 15 and lane l + 16 the same row
// at columns c + 16 .. c + 31 (the 16x32bx2 TMEM shape); f(row, first column,
// 8 values) takes each lane's 16 columns as two runs of 8
template <typename F>
__device__ __forceinline__ void acc_rows_all(uint32_t tbase, uint32_t col0, int ncols, F&& f) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int sp = w & 3, g = w >> 2, hl = l >> 4;
    for (int c = 32 * g; c < ncols; c += 64) {
        float v[16];
        tc::tmem_ld16x2<16>(tc::tmem_addr(tbase, 32 * sp, col0 + c), v);
        tc::tmem_wait_ld();
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = v[i];
        f(16 * sp + (l & 15), c + 16 * hl, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = v[8 + i];
        f(16 * sp + (l & 15), c + 16 * hl + 8, x);
    }
}

using tri::LDT;
using tri::tri_inverse64;

struct F1Smem {
    uint32_t K, Q, V, A, T, X, Tw, Twl, Tu, Tul, vec, total;
};

// Sized for two CTAs per SM: T takes the space of the q tile (dead after the
// Grams) when it fits, and the four bf16 T-operand tiles that of A and X (dead
// after the solve).
__host__ __device__ inline F1Smem f1_plan(int Dk, int Dv) {
    F1Smem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    const uint32_t fm = C * LDT * 4;  // one padded fp32 64 x 64 matrix
    s.K = take(C * Dk * 2);
    s.Q = take(C * Dk * 2);
    s.V = take(C * Dv * 2);
    s.A = take(2 * fm);               // A, then X right after it
    s.X = s.A + fm;
    s.T = (uint32_t)(C * Dk * 2) >= fm ? s.Q : take(fm);
    s.Tw = s.A;
    s.Twl = s.A + C * C * 2;
    s.Tu = s.A + 2 * C * C * 2;
    s.Tul = s.A + 3 * C * C * 2;
    s.vec = take(14 * C * 4 + C * 8);
    s.total = o;
    return s;
}

// u_tma: U leaves by TMA stores of swizzled 64 x 32 boxes staged in the A / X
// space (dead once the W / U products are done) instead of per-thread stores
__global__ void __launch_bounds__(kThreads, 2) fwd_chunk_tc_kernel(Dims d, Ptrs p, const __grid_constant__ Tmaps tm,
                                                                 int u_tma) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar, barKQ;
    __shared__ uint32_t tmem_sh;
    const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int tid = threadIdx.x, warp = tid >> 5;
    const F1Smem L = f1_plan(Dk, Dv);
    float* vec = reinterpret_cast<float*>(sm + L.vec);
    float* bt = vec;            // beta
    float* gm = bt + C;         // exp(Gamma)
    float* rqv = gm + C;        // r_q / sqrt(Dk)
    float* rkv = rqv + C;       // r_k
    // Gamma as an unevaluated sum hi + lo of two floats: for steps whose Gamma are
    // within a factor of two (the only case where exp(Gamma_i - Gamma_j) is not
    // negligible) hi_i - hi_j is exact, so differences keep fp64 accuracy
    float* Ghi = rkv + C;
    float* Glo = Ghi + C;
    // Off the diagonal 16 x 16 blocks, M_ij = exp(Gamma_i - Gamma_j) is the
    // product of two factors through the last step b = 16 J + 15 of the column
    // block J of j: uf[J][i] = exp(Gamma_i - Gamma_b) (i > b) and wf[J][j] =
    // exp(Gamma_b - Gamma_j) (j <= b).  Gamma does not increase, so both lie in
    // (0, 1]: neither overflows, and one underflows only where M_ij does.
    float* uf = Glo + C;      // [3][64]
    float* wf = uf + 3 * C;   // [3][64]
    float* A = reinterpret_cast<float*>(sm + L.A);
    float* Tm = reinterpret_cast<float*>(sm + L.T);
    float* X = reinterpret_cast<float*>(sm + L.X);

    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const int64_t gbase = bh * d.Tp + t0;
    const int64_t rbase = ((int64_t)bb * d.Hk + j) * d.Tp + t0;
    const int64_t ldv = d.Hv * Dv;
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);

    // the v tile is first read by the U product: its copies stay in flight under
    // the Grams, the A / P pass and the solve
    cpa_tile(sm + L.V, v + ((int64_t)bb * d.T + t0) * ldv + (int64_t)h * Dv, ldv, Dv, nvalid);
    tc::cp_async_commit();
    if (warp == 0) {
        tc::tmem_alloc(&tmem_sh, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 2);  // each MMA round: one commit (or arrival) per issuer
        tc::mbar_init(&barKQ, 1);
        tc::fence_mbar_init();
        // raw k and q rows of this chunk: panel images written by prep
        const uint32_t tk = (uint32_t)(C * Dk * 2);
        const int64_t kqi = ((int64_t)bb * d.Hk + j) * d.NC + c;
        tc::mbar_arrive_expect_tx(&barKQ, 2 * tk);
        tc::bulk_g2s(sm + L.K, static_cast<const uint8_t*>(p.kimg) + kqi * tk, tk, &barKQ);
        tc::bulk_g2s(sm + L.Q, static_cast<const uint8_t*>(p.qimg) + kqi * tk, tk, &barKQ);
    }
    if (tid < C) {
        const double G = p.gam[gbase + tid];
        const float gh = (float)G;
        Ghi[tid] = gh;
        Glo[tid] = (float)(G - (double)gh);
        gm[tid] = expf((float)G);
        bt[tid] = p.beta[gbase + tid];
        rqv[tid] = p.rq[rbase + tid] * rsqrtf((float)Dk);
        rkv[tid] = p.rk[rbase + tid];
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tb = tmem_sh;
    uint32_t phase = 0;
    bool ok = tc::mbar_wait(&barKQ, 0, &g_err_fwdtc);
    const tc::Tile tK = tc::panel_tile(sm + L.K, C, true), tQ = tc::panel_tile(sm + L.Q, C, true);
    const tc::Tile tKmn = tc::panel_tile(sm + L.K, C, false), tVmn = tile_of(sm + L.V, Dv, false);

    // ---- Grams of the raw rows.  Threads 0 and 32 (two warps) issue one product
    // chain each: one thread issues a tcgen05.mma about every 80 cycles whatever its
    // size, so the two chains run side by side.
    if (tid == 0) {
        tc::mma_tile(tb + 0, tK, tK, C, C, Dk, false);
        tc::mma_commit(&bar);
    } else if (tid == 32) {
        tc::mma_tile(tb + 64, tQ, tK, C, C, Dk, false);
        tc::mma_commit(&bar);
    }
    if (tid < 3 * C) {  // decay factors, while the Grams run
        const int J = tid / C, i = tid % C, b = 16 * J + 15;
        const float dg = (Ghi[i] - Ghi[b]) + (Glo[i] - Glo[b]);
        uf[tid] = i > b ? expf(dg) : 0.f;
        wf[tid] = i <= b ? expf(-dg) : 0.f;
    }
    __syncthreads();
    ok = tc::mbar_wait(&bar, phase, &g_err_fwdtc) && ok;
    phase ^= 1u;
    tc::tc_fence_after();
    uint8_t* Pimg = static_cast<uint8_t*>(p.P) + (bh * d.NC + c) * C * C * 2;
    if (ok) {
        // A and P in one pass over both Grams, all 32 lanes (16x32bx2 loads): warp
        // group g takes columns 32 g .. 32 g + 31 of row r, lane half hl the 16 of
        // them from 32 g + 16 hl, in two runs of 8 from c0.  The 16-column block J
        // of a run is uniform over each half-warp, so is the choice between the
        // factored and the direct decay.
        const int l = tid & 31, sp = warp & 3, g = warp >> 2, hl = l >> 4;
        const int r = 16 * sp + (l & 15);
        const float ra = bt[r] * rkv[r], rp = rqv[r], ghr = Ghi[r], glr = Glo[r];
        float va[16], vp[16];
        tc::tmem_ld16x2<16>(tc::tmem_addr(tb, 32 * sp, 32 * g), va);
        tc::tmem_ld16x2<16>(tc::tmem_addr(tb, 32 * sp, 64 + 32 * g), vp);
        tc::tmem_wait_ld();
#pragma unroll
        for (int run = 0; run < 2; ++run) {
            float xa[8], xp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                xa[i] = va[8 * run + i];
                xp[i] = vp[8 * run + i];
            }
            const int c0 = 32 * g + 16 * hl + 8 * run, J = c0 >> 4;
            float m[8];
            if (J < sp) {
                const float u = uf[J * C + r];
#pragma unroll
                for (int i = 0; i < 8; ++i) m[i] = u * wf[J * C + c0 + i];
            } else if (J == sp) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int jj = c0 + i;
                    m[i] = jj <= r ? expf((ghr - Ghi[jj]) + (glr - Glo[jj])) : 0.f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) m[i] = 0.f;
            }
            float a8[8], p8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int jj = c0 + i;
                const float mk = m[i] * rkv[jj];
                a8[i] = jj < r ? ra * mk * xa[i] : 0.f;
                p8[i] = rp * mk * xp[i];
            }
            float4* arow = reinterpret_cast<float4*>(A + r * LDT + c0);
            arow[0] = make_float4(a8[0], a8[1], a8[2], a8[3]);
            arow[1] = make_float4(a8[4], a8[5], a8[6], a8[7]);
            st_bf16x8(Pimg + tc::panel_off(c0, r, C), p8);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- T = (I + A)^-1 (fp32)
    tri_inverse64(A, Tm, X);
    // T as a bf16 panel image: 16-byte chunk e holds row e % 64, columns 8 (e / 64) ..
    uint8_t* Timg = reinterpret_cast<uint8_t*>(p.Tinv) + (bh * d.NC + c) * C * C * 2;
    for (int e = tid; e < C * (C / 8); e += blockDim.x) {
        const int i = e % C, j0 = (e / C) * 8;
        float4 t0 = make_float4(0.f, 0.f, 0.f, 0.f), t1 = t0;
        if ((j0 >> 4) <= (i >> 4)) {
            t0 = *reinterpret_cast<const float4*>(Tm + i * LDT + j0);
            t1 = *reinterpret_cast<const float4*>(Tm + i * LDT + j0 + 4);
        }
        const float t8[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        st_bf16x8(Timg + 16 * e, t8);
    }
    // A operands T diag(beta gam r_k) and T diag(beta), each as hi + lo bf16 (x = j, y = i)
    for (int e = tid; e < C * (C / 8); e += blockDim.x) {
        int i, jg;
        chunk_rc(e, C / 8, i, jg);  // eight consecutive rows per 8-lane group
        const int j0 = 8 * jg;
        float4 t0 = make_float4(0.f, 0.f, 0.f, 0.f), t1 = t0;
        if ((j0 >> 4) <= (i >> 4)) {
            t0 = *reinterpret_cast<const float4*>(Tm + i * LDT + j0);
            t1 = *reinterpret_cast<const float4*>(Tm + i * LDT + j0 + 4);
        }
        const float tr[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        float w8[8], wl[8], u8[8], ul[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int jj = j0 + s;
            const float t = tr[s];
            w8[s] = t * bt[jj] * gm[jj] * rkv[jj];
            u8[s] = t * bt[jj];
            wl[s] = w8[s] - __bfloat162float(__float2bfloat16_rn(w8[s]));
            ul[s] = u8[s] - __bfloat162float(__float2bfloat16_rn(u8[s]));
        }
        const uint32_t o = canon(j0, i, C);
        st_bf16x8(sm + L.Tw + o, w8);
        st_bf16x8(sm + L.Twl + o, wl);
        st_bf16x8(sm + L.Tu + o, u8);
        st_bf16x8(sm + L.Tul + o, ul);
    }
    tc::cp_async_wait_all();  // this thread's pieces of the v tile
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- W = T diag(beta gam r_k) K,  U = T diag(beta) V: one round of MMAs
    // when both fit in the 256 TMEM columns, else W first, then U
    const tc::Tile tTw = tile_of(sm + L.Tw, C, true), tTwl = tile_of(sm + L.Twl, C, true);
    const tc::Tile tTu = tile_of(sm + L.Tu, C, true), tTul = tile_of(sm + L.Tul, C, true);
    const bool one_round = Dk + Dv <= kTmemCols;
    if (tid == 0) {
        tc::mma_tile(tb + 0, tTw, tKmn, C, Dk, C, false);
        tc::mma_tile(tb + 0, tTwl, tKmn, C, Dk, C, true);
        tc::mma_commit(&bar);
    } else if (tid == 32) {
        if (one_round) {
            tc::mma_tile(tb + Dk, tTu, tVmn, C, Dv, C, false);
            tc::mma_tile(tb + Dk, tTul, tVmn, C, Dv, C, true);
            tc::mma_commit(&bar);
        } else {
            tc::mbar_arrive(&bar);
        }
    }
    ok = tc::mbar_wait(&bar, phase, &g_err_fwdtc) && ok;
    phase ^= 1u;
    tc::tc_fence_after();
    uint8_t* Wimg = static_cast<uint8_t*>(p.W) + gbase * Dk * 2;
    if (ok) {
        acc_rows_all(tb, 0, Dk, [&](int r, int c0, const float (&x)[8]) {
            st_bf16x8(Wimg + tc::panel_off(c0, r, C), x);
        });
    }
    uint32_t ucol = (uint32_t)Dk;
    if (!one_round) {
        tc::tc_fence_before();
        __syncthreads();  // W read out of TMEM
        tc::tc_fence_after();
        if (tid == 0) {
            tc::mma_tile(tb + 0, tTu, tVmn, C, Dv, C, false);
            tc::mma_tile(tb + 0, tTul, tVmn, C, Dv, C, true);
            tc::mma_commit(&bar);
        } else if (tid == 32) {
            tc::mbar_arrive(&bar);
        }
        ok = tc::mbar_wait(&bar, phase, &g_err_fwdtc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        ucol = 0;
    }
    if (ok && !u_tma) {
        float* U = p.U + gbase * Dv;
        acc_rows_all(tb, ucol, Dv, [&](int r, int c0, const float (&x)[8]) {
            float4* dst = reinterpret_cast<float4*>(U + (int64_t)r * Dv + c0);
            dst[0] = make_float4(x[0], x[1], x[2], x[3]);
            dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        });
    } else if (ok) {
        // box b (columns 32 b .. 32 b + 31) 8 KB after the box before it, from the
        // first 1024-byte aligned shared address in the A / X space (the swizzle
        // follows the address bits): row r's 16-byte piece j at r * 128 +
        // ((j ^ (r % 8)) * 16), the layout of the 128-byte swizzle
        uint8_t* stage = sm + L.A + ((1024u - (tc::smem_u32(sm + L.A) & 1023u)) & 1023u);
        acc_rows_all(tb, ucol, Dv, [&](int r, int c0, const float (&x)[8]) {
            uint8_t* box = stage + (c0 >> 5) * (C * 128) + r * 128;
            const int j = (c0 & 31) >> 2;
            *reinterpret_cast<float4*>(box + (((j) ^ (r & 7)) << 4)) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(box + (((j + 1) ^ (r & 7)) << 4)) = make_float4(x[4], x[5], x[6], x[7]);
        });
        tc::fence_async_smem();  // generic-proxy writes -> the TMA store reads them
    }
    tc::tc_fence_before();
    __syncthreads();
    if (ok && u_tma && tid == 0) {
        const uint8_t* stage = sm + L.A + ((1024u - (tc::smem_u32(sm + L.A) & 1023u)) & 1023u);
        for (int bx = 0; bx < Dv / 32; ++bx)
            tc::tma_store_2d(&tm.Us, stage + bx * (C * 128), 32 * bx, (int)gbase);
        tc::bulk_commit();
        tc::bulk_wait_all();  // the stores have read the staging space and are done
    }
    if (warp == 0) tc::tmem_dealloc(tb, kTmemCols);
}

}  // namespace

bool fwd_chunk_tc_supported(const Dims& d) {
    if (d.dtype != 1) return false;
    if (d.Dk % 32 || d.Dv % 32 || d.Dk > 256 || d.Dv > 256) return false;
    return f1_plan((int)d.Dk, (int)d.Dv).total + 2048 <= 227u * 1024u;
}

cudaError_t launch_fwd_chunk_tc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = f1_plan((int)d.Dk, (int)d.Dv).total + 1024;
    auto kern = fwd_chunk_tc_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B);
    // the U staging needs 64 Dv fp32 (plus up to 1 KB of alignment) in the A / X
    // space (two padded 64 x 64 fp32 matrices) and a 32-column box grid
    const int u_tma = p.tmaps != nullptr && d.Dv % 32 == 0 &&
                      (uint32_t)(C * d.Dv * 4) + 1024u <= 2u * (uint32_t)(C * LDT * 4);
    Tmaps tmz{};
    kern<<<grid, kThreads, smem, s>>>(d, p, u_tma ? *p.tmaps : tmz, u_tma);
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace gdn
