// gdn_scan_ta.cu -- the forward and backward chunk scans for 128-row value
// tiles (M = 128 tcgen05 MMAs) with the state operand held in tensor memory.
//
// Same recurrence as gdn_scan_tc.cu (mlx-lm PR "Add gated_delta_update VJP",
// "What this PR adds" and "Design notes": chunk 64, sequential over chunks):
//   Delta^T = U^T - S^T W^T,   O^T = S^T Qs^T + Delta^T P^T,
//   S^T <- gam_63 S^T + (Delta^T diag(e r_k)) K
// with Qs = diag(gam r_q / sqrt(Dk)) Q.  The products with N = 64 (one chunk of
// steps) would be bound by shared-memory bandwidth if their 128-row A operand
// were read from shared memory, so S^T (as bf16 pairs) and Delta^T (hi + lo, and
// diag(e r_k)-scaled hi + lo) are written by the epilogue threads straight into
// TMEM, each thread its own accumulator row, and the MMAs take A from there.
// B operands: the W and P images and the raw q and k images by bulk copy (q is
// scaled by gam r_q / sqrt(Dk) in place); U rows by TMA; the per-chunk gate
// and norm vectors by bulk copy two chunks ahead.  Output rows are accumulated in two TMEM
// buffers so the epilogue of chunk c runs while the products of chunk c + 1 do.
//
// TMEM columns: [0, Dk) the fp32 state S^T; [Dk, Dk + 128) A operands (S^T as
// bf16 pairs during step 2, then Delta^T hi | lo | e-scaled hi | lo, 32 each);
// [Dk + 128, +64) the Delta^T accumulator; then two 64-column output buffers.
//
// The reverse scan lives in gdn_scan_ta.cuh (shared with the fused backward
// of gdn_bwd_tc.cu); this file also holds its stand-alone launch.
#include "gdn_scan_ta.cuh"

namespace gdn {

GDN_ERROR_WORD(scanta)

namespace {

using namespace ta;

struct TaSmem {
    uint32_t W, Q, K, P, Ub, St, Dt, Dlo, Ob, raw, vec, total;
};

__host__ __device__ inline TaSmem ta_plan(int Dk) {
    TaSmem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    s.W = take(C * Dk * 2);     // panel images (64 rows)
    s.Q = take(C * Dk * 2);
    s.K = take(C * Dk * 2);
    s.P = take(C * C * 2);
    s.Ub = take(C * DVT * 4);   // U rows of the value tile [t][dv], fp32, by TMA
    s.St = take(DVT * Dk * 2);  // checkpoint image staging (panel, 128 rows)
    s.Dt = take(DVT * C * 2);   // Delta^T hi / lo image staging (canonical, x = step)
    s.Dlo = take(DVT * C * 2);
    s.Ob = take(C * DVT * 2);   // output rows [t][dv]
    s.raw = take(2 * kRawBytes);
    s.vec = take(2 * 4 * C * 4);
    s.total = o;
    return s;
}

struct TaCols {
    uint32_t aop, dacc, o0;
};
__host__ __device__ inline TaCols ta_cols(int Dk) {
    TaCols t;
    t.aop = (uint32_t)Dk;
    t.dacc = (uint32_t)Dk + 128;
    t.o0 = (uint32_t)Dk + 192;
    return t;
}

// gam r_q / sqrt(Dk) of its step; each thread keeps one step
__device__ __forceinline__ void scale_q(uint8_t* Q, const uint8_t* raw, int Dk) {
    const int t = threadIdx.x & (C - 1);
    const double* G = reinterpret_cast<const double*>(raw);
    const float* rq = reinterpret_cast<const float*>(raw + C * 8);
    const float s = expf((float)G[t]) * rq[t] * rsqrtf((float)Dk);
    for (int e = threadIdx.x; e < C * Dk / 8; e += kThreads) {
        uint4 u = reinterpret_cast<const uint4*>(Q)[e];
        uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            w[i] = tc::pack_bf16(f.x * s, f.y * s);
        }
        reinterpret_cast<uint4*>(Q)[e] = u;
    }
}

// KC: per-key-channel gates.  W, P and U as above (from the per-channel chunk
// kernel); the B operands Qs and K are the per-value-head images Q_r = qh o
// exp(Gamma) and K_d = kh o exp(Gamma_63 - Gamma) (qimg, kimg indexed by
// (b, value head)) with no per-step factor, and S^T decays column by column by
// the chunk's exp(Gamma_63, i) (p.ecd).
template <bool KC>
__global__ void __launch_bounds__(kThreads + 64, 1)
    fwd_scan_ta_kernel(Dims d, Ptrs p, const __grid_constant__ Tmaps tm, ScanSeg sg) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar, barW, barQ, barK, barP, barU, barR[2], barD[2];
    __shared__ uint32_t tmem_sh;
    const int tile = blockIdx.x, h = blockIdx.y;
    const int bb = (int)(blockIdx.z % d.B), sgi = sg.first + (int)(blockIdx.z / d.B);  // batch, segment
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int n0 = tile * DVT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps 0-7: epilogues (accumulator row r, column half g); warp 8: loads and MMA
    // issue; warp 9: MMA issue of the second chain of steps 2 and 4 (one thread issues
    // a tcgen05.mma about every 80 cycles, so two issuing warps overlap the chains)
    const bool epi = tid < kThreads;
    const bool prod = warp == kThreads / 32 && lane == 0;
    const bool prod2 = warp == kThreads / 32 + 1 && lane == 0;
    const int r = 32 * (warp & 3) + lane;
    const int g = (tid >> 7) & 1;
    const uint32_t lb = 32u * (uint32_t)(warp & 3);
    const TaSmem L = ta_plan(Dk);
    const TaCols TC = ta_cols(Dk);
    const int64_t bh = (int64_t)bb * d.Hv + h;
    // chunks cb .. ce - 1 of segment sgi; barrier phases and double buffers count
    // from cb (lp: the parity of a chunk within the segment)
    const int64_t cb = (int64_t)sgi * sg.len;
    const int64_t ce = cb + sg.len < d.NC ? cb + sg.len : d.NC;
    auto lp = [&](int64_t c) { return (uint32_t)((c - cb) & 1); };
    const bool maps = sg.mode != 0;       // segment maps: no checkpoints, Delta or outputs
    const bool uz = maps && n0 >= Dv;     // linear part of a map: U = 0, identity start
    const uint32_t wbytes = (uint32_t)(C * Dk * 2), pbytes = (uint32_t)(C * C * 2);
    const uint8_t* Wimg = static_cast<const uint8_t*>(p.W);
    const uint8_t* Pimg = static_cast<const uint8_t*>(p.P);
    uint8_t* ckimg = reinterpret_cast<uint8_t*>(p.ckpt);
    uint8_t* dlimg = reinterpret_cast<uint8_t*>(p.Delta);
    __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(sm + L.Ob);
    const float* Ub = reinterpret_cast<const float*>(sm + L.Ub);

    // loads (producer)
    auto load_w = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barW, wbytes);
        tc::bulk_g2s(sm + L.W, Wimg + (bh * d.NC + c) * wbytes, wbytes, &barW);
    };
    auto load_p = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barP, pbytes);
        tc::bulk_g2s(sm + L.P, Pimg + (bh * d.NC + c) * pbytes, pbytes, &barP);
    };
    // (b, key head): q / k images of its chunks; (b, value head) with KC
    const int64_t kq = KC ? bh : (int64_t)bb * d.Hk + j;
    auto load_q = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barQ, wbytes);
        tc::bulk_g2s(sm + L.Q, static_cast<const uint8_t*>(p.qimg) + (kq * d.NC + c) * wbytes, wbytes, &barQ);
    };
    auto load_k = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barK, wbytes);
        tc::bulk_g2s(sm + L.K, static_cast<const uint8_t*>(p.kimg) + (kq * d.NC + c) * wbytes, wbytes, &barK);
    };
    auto load_raw = [&](int64_t c) {
        const int s = (int)lp(c);
        uint8_t* dst = sm + L.raw + s * kRawBytes;
        if constexpr (KC) {
            tc::mbar_arrive_expect_tx(&barR[s], (uint32_t)(Dk * 4));
            tc::bulk_g2s(dst, p.ecd + (bh * d.NC + c) * Dk, (uint32_t)(Dk * 4), &barR[s]);
            return;
        }
        tc::mbar_arrive_expect_tx(&barR[s], kRawBytes);
        tc::bulk_g2s(dst, p.gam + bh * d.Tp + c * C, C * 8, &barR[s]);
        tc::bulk_g2s(dst + C * 8, p.rq + ((int64_t)bb * d.Hk + j) * d.Tp + c * C, C * 4, &barR[s]);
        tc::bulk_g2s(dst + C * 12, p.rk + ((int64_t)bb * d.Hk + j) * d.Tp + c * C, C * 4, &barR[s]);
    };
    auto load_u = [&](int64_t c) {  // U rows of chunk c, value columns n0 .. n0 + 127
        tc::mbar_arrive_expect_tx(&barU, (uint32_t)(C * DVT * 4));
        tc::tma_load_2d(sm + L.Ub, &tm.U, n0, (int)(bh * d.Tp + c * C), &barU);
    };
    // stores (lane 0 of the store warp; the caller commits)
    auto store_o = [&](int64_t c) { tc::tma_store_3d(&tm.o, Ob, h * Dv + n0, (int)(c * C), bb); };
    auto store_ck = [&](int64_t c) {
        uint8_t* img = ckimg + (bh * d.NC + c) * (int64_t)Dk * Dv * 2;
        if (DVT == Dv) {
            tc::bulk_s2g(img, sm + L.St, (uint32_t)(DVT * Dk * 2));
        } else {
            for (int gi = 0; gi < Dk / 8; ++gi)
                tc::bulk_s2g(img + (size_t)gi * Dv * 16 + (size_t)n0 * 16, sm + L.St + gi * DVT * 16,
                             (uint32_t)(DVT * 16));
        }
    };
    auto store_delta = [&](int64_t c) {
        uint8_t* base = dlimg + (bh * d.NC + c) * (int64_t)C * Dv * 4 + (int64_t)n0 * 128;
        tc::bulk_s2g(base, sm + L.Dt, (uint32_t)(DVT * 128));
        tc::bulk_s2g(base + (int64_t)C * Dv * 2, sm + L.Dlo, (uint32_t)(DVT * 128));
    };
    const bool storer = warp == kStoreWarp && lane == 0;
    // output rows of chunk c (buffer c & 1) -> staging
    auto step5 = [&](uint32_t tb, int64_t c) {
        float a[2][16];
        const uint32_t col = TC.o0 + lp(c) * 64u + 32u * g;
        tc::tmem_ld16(tc::tmem_addr(tb, lb, col), a[0]);
        tc::tmem_ld16(tc::tmem_addr(tb, lb, col + 16), a[1]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 16; ++i) Ob[(32 * g + 16 * u + i) * DVT + r] = __float2bfloat16_rn(a[u][i]);
    };

    if (warp == 0) {
        tc::tmem_alloc(&tmem_sh, 512);
        tc::tmem_relinquish();
    }
    if (prod) {
        tc::mbar_init(&bar, 2);  // one commit from each issuer per MMA round
        tc::mbar_init(&barW, 1);
        tc::mbar_init(&barQ, 1);
        tc::mbar_init(&barK, 1);
        tc::mbar_init(&barP, 1);
        tc::mbar_init(&barU, 1);
        tc::mbar_init(&barR[0], 1);
        tc::mbar_init(&barR[1], 1);
        for (int i = 0; i < 2; ++i) tc::mbar_init(&barD[i], kThreads / 32);
        tc::fence_mbar_init();
    }
    __syncthreads();  // barriers initialised
    if (prod) {
        load_w(cb);
        load_q(cb);
        load_k(cb);
        load_p(cb);
        if (!uz) load_u(cb);
        load_raw(cb);
        if (ce - cb > 1) load_raw(cb + 1);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tb = tmem_sh;
    const int halfk = Dk / 2;
    // start state (rows dk, row stride Dv): state0 for the first segment, the
    // chained start states for the others; zero / the identity for the maps
    const float* sin = nullptr;
    if (!maps && sgi == 0 && p.state0) sin = p.state0 + bh * Dk * Dv + n0;
    if (!maps && sgi > 0 && sg.start) sin = sg.start + ((int64_t)(sgi - 1) * d.B * d.Hv + bh) * Dk * Dv + n0;
    if (!maps && sg.sin) sin = sg.sin + bh * Dk * Dv + n0;
    bool ok = true;
    if (epi) {
        for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {  // initial state -> TMEM
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = uz ? (cc + i == n0 - Dv + r ? 1.f : 0.f) : sin ? sin[(int64_t)(cc + i) * Dv + r] : 0.f;
            tc::tmem_st16(tc::tmem_addr(tb, lb, cc), v);
        }
        tc::tmem_wait_st();
        ok = tc::mbar_wait(&barR[0], 0, &g_err_scanta);
        ok = tc::mbar_wait(&barQ, 0, &g_err_scanta) && ok;
        vectors_from_raw<KC>(sm + L.raw, reinterpret_cast<float*>(sm + L.vec), Dk);
        if (!KC) scale_q(sm + L.Q, sm + L.raw, Dk);
        tc::fence_async_smem();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    const tc::Tile tW = tc::panel_tile(sm + L.W, C, true);     // B = W^T: x = dk = K
    const tc::Tile tQ = tc::panel_tile(sm + L.Q, C, true);     // B = Qs^T
    const tc::Tile tP = tc::panel_tile(sm + L.P, C, true);     // B = P^T: x = s = K
    const tc::Tile tKmn = tc::panel_tile(sm + L.K, C, false);  // B = K: x = dk = N
    uint32_t phase = 0;

    for (int64_t c = cb; c < ce; ++c) {
        const float* vb = reinterpret_cast<const float*>(sm + L.vec) + lp(c) * 4 * C;
        const float* kev = vb + 3 * C;
        const float gC = vb[C - 1];
        const uint32_t ocol = TC.o0 + lp(c) * 64u;
        if (storer) {  // Delta images of chunk c - 1, staged before the barrier above
            if (!maps && c > cb) store_delta(c - 1);
            tc::bulk_commit();
        }
        // step 1: S^T -> A operand (bf16 pairs in TMEM); S^T *= gam_63
        if (epi) {
            for (int cb = g * halfk; cb < (g + 1) * halfk; cb += 32) {
                float v[2][16];
                tc::tmem_ld16(tc::tmem_addr(tb, lb, cb), v[0]);
                tc::tmem_ld16(tc::tmem_addr(tb, lb, cb + 16), v[1]);
                tc::tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w[i] = tc::pack_bf16(v[0][2 * i], v[0][2 * i + 1]);
                    w[8 + i] = tc::pack_bf16(v[1][2 * i], v[1][2 * i + 1]);
                }
                tc::tmem_st16u(tc::tmem_addr(tb, lb, TC.aop + cb / 2), w);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v[0][i] *= KC ? vb[cb + i] : gC;
                    v[1][i] *= KC ? vb[cb + 16 + i] : gC;
                }
                tc::tmem_st16(tc::tmem_addr(tb, lb, cb), v[0]);
                tc::tmem_st16(tc::tmem_addr(tb, lb, cb + 16), v[1]);
            }
            tc::tmem_wait_st();
        }
        if (storer) tc::bulk_wait_read_but1();  // checkpoint / output staging read out
        tc::tc_fence_before();
        __syncthreads();  // (B)
        tc::tc_fence_after();
        uint32_t hiw[16], low[16];
        if (prod) {
            // step 2: Delta^T acc = S^T W^T here and O^T = S^T Qs^T by the second
            // issuer, two independent accumulation chains
            ok = tc::mbar_wait(&barW, lp(c), &g_err_scanta) && ok;
            const uint32_t id = tc::idesc_bf16(DVT, C, false, false);
            uint64_t dw = tW.desc(0);
            const uint64_t iw = tW.desc_step();
            for (int k = 0; k < Dk; k += 16) {
                tc::mma_bf16_ta(tb + TC.dacc, tb + TC.aop + k / 2, dw, id, k > 0);
                dw += iw;
            }
            tc::mma_commit(&bar);
            ok = tc::mbar_wait(&bar, phase, &g_err_scanta) && ok;  // both chains
            phase ^= 1u;
            if (c + 1 < ce) {
                load_w(c + 1);
                load_q(c + 1);
            }
        } else if (prod2) {
            // (the epilogue waits for q and scales it before (B); KC has no scaling)
            if (KC) ok = tc::mbar_wait(&barQ, lp(c), &g_err_scanta) && ok;
            const uint32_t id = tc::idesc_bf16(DVT, C, false, false);
            uint64_t dq = tQ.desc(0);
            const uint64_t iq = tQ.desc_step();
            for (int k = 0; k < Dk; k += 16) {
                tc::mma_bf16_ta(tb + ocol, tb + TC.aop + k / 2, dq, id, k > 0);
                dq += iq;
            }
            tc::mma_commit(&bar);
            phase ^= 1u;
        } else if (epi) {
            // meanwhile: the checkpoint image (S^T bf16, from the A operand) and
            // the output rows of chunk c - 1
            for (int cb = g * (Dk / 4); cb < (g + 1) * (Dk / 4); cb += 16) {
                uint32_t w[16];
                tc::tmem_ld16u(tc::tmem_addr(tb, lb, TC.aop + cb), w);
                tc::tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4*>(sm + L.St + tc::panel_off(2 * cb + 8 * q4, r, DVT)) =
                        make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
            }
            if (!maps && c > cb) step5(tb, c - 1);
            tc::fence_async_smem();
            ok = tc::mbar_wait(&bar, phase, &g_err_scanta) && ok;
            phase ^= 1u;
            tc::tc_fence_after();
            // step 3: Delta^T = U^T - acc -> A operands hi, lo and (diag(e r_k)) hi, lo,
            // in two passes of 16 steps (32 g + 16 u2 .. + 15), each handed to the
            // MMA issuer on its own barrier
            if (!uz) ok = tc::mbar_wait(&barU, lp(c), &g_err_scanta) && ok;
            float a[2][16];
            tc::tmem_ld16(tc::tmem_addr(tb, lb, TC.dacc + 32 * g), a[0]);
            tc::tmem_ld16(tc::tmem_addr(tb, lb, TC.dacc + 32 * g + 16), a[1]);
            tc::tmem_wait_ld();
            uint32_t dew[16], delw[16];
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
#pragma unroll
                for (int i = 8 * u2; i < 8 * u2 + 8; ++i) {
                    float dl[2], lo[2], de[2], dlo[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int ti = 2 * i + u;  // step 32 g + ti
                        dl[u] = (uz ? 0.f : Ub[(32 * g + ti) * DVT + r]) - a[ti >> 4][ti & 15];
                        lo[u] = dl[u] - __bfloat162float(__float2bfloat16_rn(dl[u]));
                        de[u] = KC ? dl[u] : dl[u] * kev[32 * g + ti];
                        dlo[u] = de[u] - __bfloat162float(__float2bfloat16_rn(de[u]));
                    }
                    hiw[i] = tc::pack_bf16(dl[0], dl[1]);
                    low[i] = tc::pack_bf16(lo[0], lo[1]);
                    dew[i] = tc::pack_bf16(de[0], de[1]);
                    delw[i] = tc::pack_bf16(dlo[0], dlo[1]);
                }
                const uint32_t cc = 16 * g + 8 * u2;
                tc::tmem_st8u(tc::tmem_addr(tb, lb, TC.aop + cc), hiw + 8 * u2);
                tc::tmem_st8u(tc::tmem_addr(tb, lb, TC.aop + 32 + cc), low + 8 * u2);
                tc::tmem_st8u(tc::tmem_addr(tb, lb, TC.aop + 64 + cc), dew + 8 * u2);
                tc::tmem_st8u(tc::tmem_addr(tb, lb, TC.aop + 96 + cc), delw + 8 * u2);
                tc::tmem_wait_st();
                tc::warp_arrive_after_st(&barD[u2]);
            }
            if (storer) tc::bulk_wait_read_all();  // Delta staging of c - 1 read out
            tc::named_sync(1, kThreads);
        }
        if (prod || prod2) {
            // step 4: O^T += Delta^T P^T (hi, lo) here and S^T += (Delta^T diag(e r_k)) K
            // (hi, lo) by the second issuer; the steps of pass u2 (16-step slices u2 and
            // 2 + u2) once it is handed over
            if (prod) ok = tc::mbar_wait(&barP, lp(c), &g_err_scanta) && ok;
            else ok = tc::mbar_wait(&barK, lp(c), &g_err_scanta) && ok;
            const uint32_t idp = tc::idesc_bf16(DVT, C, false, false);
            const uint32_t idk = tc::idesc_bf16(DVT, Dk, false, true);
            const uint64_t dp0 = tP.desc(0), ip = tP.desc_step();
            const uint64_t dk0 = tKmn.desc(0), ik = tKmn.desc_step();
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
                ok = tc::mbar_wait(&barD[u2], lp(c), &g_err_scanta) && ok;
                tc::tc_fence_after();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ks = 2 * (i & 1) + u2;  // 16-step slice
                    const uint32_t hl = (uint32_t)(i >> 1) * 32u;
                    if (prod)
                        tc::mma_bf16_ta(tb + ocol, tb + TC.aop + hl + 8 * ks, dp0 + (uint64_t)ks * ip, idp, 1u);
                    else
                        tc::mma_bf16_ta(tb, tb + TC.aop + 64 + hl + 8 * ks, dk0 + (uint64_t)ks * ik, idk, 1u);
                }
            }
            tc::mma_commit(&bar);
        }
        if (prod2) {
            phase ^= 1u;
        } else if (prod) {
            if (!uz && c + 1 < ce) load_u(c + 1);  // step 3 of chunk c has read U
            ok = tc::mbar_wait(&bar, phase, &g_err_scanta) && ok;
            phase ^= 1u;
            if (c + 1 < ce) {
                load_k(c + 1);
                load_p(c + 1);
            }
            if (c + 2 < ce) load_raw(c + 2);
        } else if (epi) {
            if (storer) {
                if (!maps) {
                    store_ck(c);
                    if (c > cb) store_o(c - 1);
                }
                tc::bulk_commit();
            }
            // meanwhile: Delta image staging, U / vectors / scaled q of chunk c + 1
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint32_t off = canon(32 * g + 8 * q4, r, C);
                *reinterpret_cast<uint4*>(sm + L.Dt + off) =
                    make_uint4(hiw[4 * q4], hiw[4 * q4 + 1], hiw[4 * q4 + 2], hiw[4 * q4 + 3]);
                *reinterpret_cast<uint4*>(sm + L.Dlo + off) =
                    make_uint4(low[4 * q4], low[4 * q4 + 1], low[4 * q4 + 2], low[4 * q4 + 3]);
            }
            if (c + 1 < ce) {
                const int64_t l1 = c + 1 - cb;
                const uint8_t* raw = sm + L.raw + (l1 & 1) * kRawBytes;
                ok = tc::mbar_wait(&barR[l1 & 1], (uint32_t)((l1 >> 1) & 1), &g_err_scanta) && ok;
                vectors_from_raw<KC>(raw, reinterpret_cast<float*>(sm + L.vec) + (l1 & 1) * 4 * C, Dk);
                if (!KC) {
                    ok = tc::mbar_wait(&barQ, (uint32_t)(l1 & 1), &g_err_scanta) && ok;
                    scale_q(sm + L.Q, raw, Dk);
                }
            }
            tc::fence_async_smem();
            ok = tc::mbar_wait(&bar, phase, &g_err_scanta) && ok;
            phase ^= 1u;
            tc::tc_fence_after();
        }
        // before the last chunk's output rows are staged: all stores have read out
        if (storer && c + 1 == ce) tc::bulk_wait_read_all();
        tc::tc_fence_before();
        __syncthreads();  // (A) of chunk c + 1
        tc::tc_fence_after();
    }
    // the last chunk's output rows and Delta images
    if (epi && !maps) step5(tb, ce - 1);
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (storer && !maps) {
        store_delta(ce - 1);
        store_o(ce - 1);
        tc::bulk_commit();
    }
    // end state: the final state (last segment) or the segment map's columns
    float* sout = nullptr;
    int64_t ostr = Dv;
    if (maps) {
        ostr = seg_wd(Dk, Dv);
        sout = sg.maps + ((int64_t)sgi * d.B * d.Hv + bh) * Dk * ostr + n0;
    } else if (sg.sout) {
        sout = sg.sout + bh * Dk * Dv + n0;
    } else if (sgi == sg.nseg - 1) {
        sout = p.state_T + bh * Dk * Dv + n0;
    }
    if (epi && sout) {
        for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {
            float v[16];
            tc::tmem_ld16(tc::tmem_addr(tb, lb, cc), v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) sout[(int64_t)(cc + i) * ostr + r] = v[i];
        }
    }
    if (storer) tc::bulk_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

template <bool KC>
__global__ void __launch_bounds__(kThreads + 64, 1)
    bwd_scan_ta_kernel(Dims d, Ptrs p, const __grid_constant__ Tmaps tm, ScanSeg sg) {
    bwd_scan_ta_body<KC>(d, p, tm, blockIdx.x, blockIdx.y, (int)(blockIdx.z % d.B), sg,
                     sg.first + (int)(blockIdx.z / d.B), &g_err_scanta, nullptr, true);
}

}  // namespace

bool scan_ta_supported(const Dims& d) {
    return d.dtype == 1 && d.Dv % DVT == 0 && d.Dk % 64 == 0 && d.Dk >= 64 && d.Dk <= 192 &&
           ta_plan((int)d.Dk).total + 2048 <= 227u * 1024u && tb_plan((int)d.Dk).total + 2048 <= 227u * 1024u;
}

cudaError_t launch_fwd_scan_ta(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = ta_plan((int)d.Dk).total + 1024;
    auto kern = fwd_scan_ta_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, ScanSeg{1, (int)d.NC, 0, nullptr, nullptr});
    count_launches(1);
    return cudaPeekAtLastError();
}

int64_t seg_map_width(const Dims& d) { return seg_wd(d.Dk, d.Dv); }

cudaError_t launch_fwd_scan_ta_seg(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s) {
    const size_t smem = ta_plan((int)d.Dk).total + 1024;
    auto kern = fwd_scan_ta_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t nx = sg.mode == 0 ? d.Dv / DVT : seg_wd(d.Dk, d.Dv) / DVT;
    const int64_t nz = (sg.mode == 0 ? sg.nseg : sg.nseg - 1) * d.B;
    dim3 grid((unsigned)nx, (unsigned)d.Hv, (unsigned)nz);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, sg);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_fwd_scan_ta_one(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s) {
    if (sg.mode != 0) return cudaErrorInvalidValue;
    const size_t smem = ta_plan((int)d.Dk).total + 1024;
    auto kern = fwd_scan_ta_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, sg);
    count_launches(1);
    return cudaPeekAtLastError();
}

namespace {
constexpr int kChainCols = 8;  // value columns of the state per chain CTA
constexpr int kChainThreads = 256;
constexpr int kChainRowGroups = kChainThreads / kChainCols;

// S_{s+1} = A_s S_s + B_s for s = 0 .. nseg - 2 from S_0 = state0 (zero when
// null), fp32 on the CUDA cores, each entry summed over k in ascending order.
// One CTA per (8 value columns, value head, batch) keeps its columns of the
// state in shared memory and stages each A_s there with asynchronous 16-byte
// copies (all in flight at once); thread (row group rg, column n) forms rows rg + 32 j,
// j < R = Dk / 32, as R independent sums.
template <int R>
__global__ void __launch_bounds__(kChainThreads)
    seg_chain_kernel(Dims d, const float* __restrict__ state0, ScanSeg sg) {
    constexpr int Dk = 32 * R;
    // rows of A padded by 4 floats: the 4 rows a warp reads fall in distinct banks
    constexpr int AS = Dk + 4;
    extern __shared__ __align__(16) float cs[];  // A [Dk][AS], then S [2][Dk][8]
    float* As = cs;
    float* cur = cs + Dk * AS;
    float* nxt = cur + Dk * kChainCols;
    const int n0 = blockIdx.x * kChainCols, h = blockIdx.y, bb = blockIdx.z;
    const int Dv = (int)d.Dv;
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const int64_t Wd = seg_wd(Dk, Dv);
    const int n = threadIdx.x % kChainCols, rg = threadIdx.x / kChainCols;
    for (int i = threadIdx.x; i < Dk * kChainCols; i += kChainThreads)
        cur[i] = state0 ? state0[(bh * Dk + i / kChainCols) * Dv + n0 + i % kChainCols] : 0.f;
    for (int sgi = 0; sgi + 1 < sg.nseg; ++sgi) {
        const float* M = sg.maps + ((int64_t)sgi * d.B * d.Hv + bh) * Dk * Wd;  // rows: [B_s | A_s]
        __syncthreads();  // the previous step's reads of As are done
        for (int e = threadIdx.x; e < Dk * Dk / 4; e += kChainThreads) {  // async copies, all in flight
            const int i = e / (Dk / 4), k4 = e % (Dk / 4);
            tc::cp_async16(tc::smem_u32(As + i * AS + 4 * k4), M + (int64_t)i * Wd + Dv + 4 * k4, 16);
        }
        tc::cp_async_commit();
        float acc[R];
#pragma unroll
        for (int j = 0; j < R; ++j) acc[j] = M[(int64_t)(rg + kChainRowGroups * j) * Wd + n0 + n];
        tc::cp_async_wait_all();
        __syncthreads();  // As staged
#pragma unroll 4
        for (int k = 0; k < Dk; k += 4) {
            const float s0 = cur[(k + 0) * kChainCols + n], s1 = cur[(k + 1) * kChainCols + n];
            const float s2 = cur[(k + 2) * kChainCols + n], s3 = cur[(k + 3) * kChainCols + n];
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const float4 a = *reinterpret_cast<const float4*>(As + (rg + kChainRowGroups * j) * AS + k);
                acc[j] = fmaf(a.x, s0, acc[j]);
                acc[j] = fmaf(a.y, s1, acc[j]);
                acc[j] = fmaf(a.z, s2, acc[j]);
                acc[j] = fmaf(a.w, s3, acc[j]);
            }
        }
        float* out = sg.start + ((int64_t)sgi * d.B * d.Hv + bh) * Dk * Dv + n0;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int i = rg + kChainRowGroups * j;
            nxt[i * kChainCols + n] = acc[j];
            out[(int64_t)i * Dv + n] = acc[j];
        }
        float* t = cur;
        cur = nxt;
        nxt = t;
    }
}

template <int R>
cudaError_t launch_chain_r(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s) {
    constexpr int Dk = 32 * R;
    const size_t smem = ((size_t)Dk * (Dk + 4) + 2 * (size_t)Dk * kChainCols) * sizeof(float);
    auto kern = seg_chain_kernel<R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / kChainCols), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kChainThreads, smem, s>>>(d, p.state0, sg);
    count_launches(1);
    return cudaPeekAtLastError();
}
}  // namespace

cudaError_t launch_seg_chain(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s) {
    switch (d.Dk) {  // the tensor-core scan's key widths
        case 64: return launch_chain_r<2>(d, p, sg, s);
        case 128: return launch_chain_r<4>(d, p, sg, s);
        case 192: return launch_chain_r<6>(d, p, sg, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn

namespace gdn {
cudaError_t launch_bwd_scan_ta(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = tb_plan((int)d.Dk).total + 1024;
    auto kern = bwd_scan_ta_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, ScanSeg{1, (int)d.NC, 0, nullptr, nullptr});
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_bwd_scan_ta_seg(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s) {
    const size_t smem = tb_plan((int)d.Dk).total + 1024;
    auto kern = bwd_scan_ta_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t nx = sg.mode == 0 ? d.Dv / DVT : seg_wd(d.Dk, d.Dv) / DVT;
    const int64_t nz = (sg.mode == 0 ? sg.nseg : sg.nseg - 1) * d.B;
    dim3 grid((unsigned)nx, (unsigned)d.Hv, (unsigned)nz);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, sg);
    count_launches(1);
    return cudaPeekAtLastError();
}

// per-key-channel gates: the forward and reverse scans over all chunks (grid as
// launch_fwd_scan_ta / launch_bwd_scan_ta)
cudaError_t launch_fwd_scan_kc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = ta_plan((int)d.Dk).total + 1024;
    auto kern = fwd_scan_ta_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, ScanSeg{1, (int)d.NC, 0, nullptr, nullptr});
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_bwd_scan_kc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = tb_plan((int)d.Dk).total + 1024;
    auto kern = bwd_scan_ta_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, ScanSeg{1, (int)d.NC, 0, nullptr, nullptr});
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_bwd_scan_ta_one(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s) {
    if (sg.mode != 0) return cudaErrorInvalidValue;
    const size_t smem = tb_plan((int)d.Dk).total + 1024;
    auto kern = bwd_scan_ta_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps, sg);
    count_launches(1);
    return cudaPeekAtLastError();
}
}  // namespace gdn
