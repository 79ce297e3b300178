// gdn_scan_tc.cu -- the two sequential chunk scans on the tensor cores
// (tcgen05, bf16 operands, fp32 state held in TMEM) for bf16 inputs.
//
// The state S (Dk x Dv) is kept transposed in TMEM: accumulator rows are the
// Dv columns of S (one CTA per (Dv tile, value head, batch)), TMEM columns
// are Dk.  Per chunk (equations in gdn_fwd.cu / gdn_bwd.cu; mlx-lm PR "Add
// gated_delta_update VJP", "What this PR adds" and "Design notes": chunk 64,
// reverse sweep over per-chunk state for the backward):
//
// forward   S^T            -> bf16 operand (also the saved checkpoint image); S^T *= gam_63
//           Delta^T acc     = S^T W^T          QS acc = S^T Q^T
//           Delta^T         = U^T - Delta^T acc          (epilogue)
//           PDelta acc      = Delta^T P^T
//           S^T            += (Delta^T diag(e r_k)) K     (accumulates in TMEM)
//           Delta enters both products as two bf16 terms (hi + lo): it is a
//           difference of nearly equal quantities and one bf16 term is too
//           coarse for the gate gradients; the two terms are also what is
//           saved for the backward.  q and k stay the exact bf16 inputs, their
//           scalings are applied in fp32 on the other operand or in the epilogue
//           O^T             = diag(gam r_q / sqrt(Dk)) QS + PDelta
// backward  Sbar^T         -> bf16 operand (also the saved chunk-end cotangent image); *= gam_63
//           A1 = Obar^T P,  A2 = Sbar^T K^T,  Sbar^T += (Obar^T diag(gam r_q / sqrt(Dk))) Q
//           Dbar^T          = A1 + A2 diag(e r_k)        (epilogue)
//           Sbar^T         += (-Dbar^T) W               (-Dbar^T is saved as an image)
//
// Data movement: the W and P images of the next chunk arrive by bulk copies
// (one thread, completion on an mbarrier) as soon as the MMAs that read the
// current ones have completed; q, k and dO tiles by 16-byte cp.async.  The
// operand tiles the epilogues build are written back to global memory by bulk
// stores straight from shared memory (checkpoints, Delta, Dbar, the output o),
// so no thread stalls on them.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

GDN_ERROR_WORD(scantc)

namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
// TMEM column map (Dk <= 256)
constexpr uint32_t kColState = 0, kColA = 256, kColB = 320, kColC = 384;
// warp whose lanes issue (and wait for) the bulk stores
constexpr int kStoreWarp = 1;

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

// 64-row tile, x = column in [0, ncols), canonical layout; rows >= nvalid zero-filled
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

// Accumulator row held by this thread's TMEM lane (M = 128: lane; M = 64:
// rows 16 (w % 4) + lane for lane < 16, else -1) and its warp's lane base.
template <int M>
__device__ __forceinline__ int acc_row() {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (M == 128) return 32 * (w & 3) + l;
    return l < 16 ? 16 * (w & 3) + l : -1;
}
__device__ __forceinline__ uint32_t lane0() { return 32u * ((threadIdx.x >> 5) & 3u); }
__device__ __forceinline__ int col_group() { return threadIdx.x >> 7; }  // 0 or 1

struct ScanSmem {
    uint32_t St, Q, K, W, P, O, Os, Oslo, Dt, Dlo, De, Delo, Ob, vec, total;
};

__host__ __device__ inline ScanSmem scan_plan(int Dk, int DVT, bool fwd) {
    ScanSmem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    s.St = take(DVT * Dk * 2);  // S^T / Sbar^T operand, panel layout (rows = DVT)
    s.Q = take(C * Dk * 2);
    s.K = take(C * Dk * 2);
    s.W = take(C * Dk * 2);     // panel image
    s.P = take(C * C * 2);      // panel image
    if (fwd) {
        s.Dt = take(DVT * C * 2);    // Delta^T, high bf16 part
        s.Dlo = take(DVT * C * 2);   // Delta^T, low bf16 part (Delta - high)
        s.De = take(DVT * C * 2);    // (Delta^T diag(e r_k)), high part
        s.Delo = take(DVT * C * 2);  // low part
        s.Ob = take(C * DVT * 2);    // output rows staged for the bulk stores
    } else {
        s.O = take(C * DVT * 2);
        s.Os = take(C * DVT * 2);    // Obar^T diag(gam r_q / sqrt(Dk)), high part
        s.Oslo = take(C * DVT * 2);  // low part
        s.Dt = take(DVT * C * 2);    // -Dbar^T
    }
    s.vec = take(2 * 4 * C * 4);
    s.total = o;
    return s;
}

// per-chunk vectors: gam, e, gam r_q / sqrt(Dk), e r_k
__device__ __forceinline__ void chunk_vectors(const Dims& d, const Ptrs& p, int bb, int h, int j,
                                              int64_t c, float* v) {
    const int i = threadIdx.x;
    if (i < C) {
        const int64_t gb = ((int64_t)bb * d.Hv + h) * d.Tp + c * C;
        const int64_t rb = ((int64_t)bb * d.Hk + j) * d.Tp + c * C;
        const double G = p.gam[gb + i];
        const float gm = expf((float)G);
        const float e = expf((float)(p.gam[gb + C - 1] - G));
        v[i] = gm;
        v[C + i] = e;
        v[2 * C + i] = gm * p.rq[rb + i] * rsqrtf((float)d.Dk);
        v[3 * C + i] = e * p.rk[rb + i];
    }
}

// Step 1 of both scans: the state (TMEM columns kColState .. + Dk) -> bf16
// operand St (panel layout, row = this thread's accumulator row), then the
// state is scaled by gC in place.  Up to four 16-column loads per wait.
template <int DVT>
__device__ __forceinline__ void state_to_operand(uint32_t tb, uint8_t* St, int Dk, float gC) {
    const int r = acc_row<DVT>();
    const int g = col_group();
    const int halfk = Dk / 2;
    const int end = (g + 1) * halfk;
    for (int cb = g * halfk; cb < end; cb += 64) {
        float v[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (cb + 16 * u < end) tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColState + cb + 16 * u), v[u]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (cb + 16 * u < end) {
                const int cc = cb + 16 * u;
                if (r >= 0) {
                    st_bf16x8(St + tc::panel_off(cc, r, DVT), v[u]);
                    st_bf16x8(St + tc::panel_off(cc + 8, r, DVT), v[u] + 8);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[u][i] *= gC;
                tc::tmem_st16(tc::tmem_addr(tb, lane0(), kColState + cc), v[u]);
            }
        }
    }
    tc::tmem_wait_st();
}

// Bulk store of the St operand into the chunk's image (Dv rows x Dk, panel):
// one copy when the CTA holds all Dv rows, else one per 8-column panel.
// Executed by every lane of one warp; each lane commits its own group.
template <int DVT>
__device__ __forceinline__ void store_state_image(uint8_t* img, const uint8_t* St, int Dk, int Dv,
                                                  int n0) {
    const int lane = threadIdx.x & 31;
    if (DVT == Dv) {
        if (lane == 0) tc::bulk_s2g(img, St, (uint32_t)(DVT * Dk * 2));
    } else {
        for (int gi = lane; gi < Dk / 8; gi += 32)
            tc::bulk_s2g(img + (size_t)gi * Dv * 16 + (size_t)n0 * 16, St + gi * DVT * 16,
                         (uint32_t)(DVT * 16));
    }
    tc::bulk_commit();
}

// ---------------------------------------------------------------------------
// forward scan
// ---------------------------------------------------------------------------
template <int DVT>
__global__ void __launch_bounds__(kThreads, 1) fwd_scan_tc_kernel(Dims d, Ptrs p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar, barW, barP;
    __shared__ uint32_t tmem_sh;
    const int tile = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int n0 = tile * DVT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ScanSmem L = scan_plan(Dk, DVT, true);
    float* vecs = reinterpret_cast<float*>(sm + L.vec);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
    const uint8_t* Wimg = static_cast<const uint8_t*>(p.W);
    const uint8_t* Pimg = static_cast<const uint8_t*>(p.P);
    uint8_t* ckimg = reinterpret_cast<uint8_t*>(p.ckpt);
    uint8_t* dlimg = reinterpret_cast<uint8_t*>(p.Delta);
    const float* U = p.U;
    uint8_t* o = static_cast<uint8_t*>(p.o);
    __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(sm + L.Ob);
    const int64_t ldq = d.Hk * Dk, ldo = d.Hv * Dv;
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const uint32_t wbytes = (uint32_t)(C * Dk * 2), pbytes = (uint32_t)(C * C * 2);

    auto nvalid = [&](int64_t c) { return (int)(d.T - c * C < C ? d.T - c * C : C); };
    auto load_w = [&](int64_t c) {  // one thread
        tc::mbar_arrive_expect_tx(&barW, wbytes);
        tc::bulk_g2s(sm + L.W, Wimg + (bh * d.NC + c) * wbytes, wbytes, &barW);
    };
    auto load_p = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barP, pbytes);
        tc::bulk_g2s(sm + L.P, Pimg + (bh * d.NC + c) * pbytes, pbytes, &barP);
    };
    auto fetch_q = [&](int64_t c) {
        cpa_tile(sm + L.Q, q + ((int64_t)bb * d.T + c * C) * ldq + (int64_t)j * Dk, ldq, Dk, nvalid(c));
    };
    auto fetch_k = [&](int64_t c) {
        cpa_tile(sm + L.K, k + ((int64_t)bb * d.T + c * C) * ldq + (int64_t)j * Dk, ldq, Dk, nvalid(c));
    };
    // output rows of chunk c (staged in Ob) -> o, one bulk copy per valid row
    auto store_o = [&](int64_t c) {
        const int nv = nvalid(c);
        for (int t = lane; t < nv; t += 32)
            tc::bulk_s2g(o + (((int64_t)bb * d.T + c * C + t) * ldo + (int64_t)h * Dv + n0) * 2,
                         Ob + t * DVT, (uint32_t)(DVT * 2));
        tc::bulk_commit();
    };
    auto store_delta = [&](int64_t c) {  // {hi, lo} images of Delta^T rows n0 .. n0 + DVT
        uint8_t* base = dlimg + (bh * d.NC + c) * (int64_t)C * Dv * 4 + (int64_t)n0 * 128;
        if (lane == 0) tc::bulk_s2g(base, sm + L.Dt, (uint32_t)(DVT * 128));
        if (lane == 1) tc::bulk_s2g(base + (int64_t)C * Dv * 2, sm + L.Dlo, (uint32_t)(DVT * 128));
        tc::bulk_commit();
    };

    if (warp == 0) {
        tc::tmem_alloc(&tmem_sh, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_init(&barW, 1);
        tc::mbar_init(&barP, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();  // barriers initialised
    if (tid == 0) {
        load_w(0);
        load_p(0);
    }
    fetch_q(0);
    fetch_k(0);
    tc::cp_async_commit();
    chunk_vectors(d, p, bb, h, j, 0, vecs);
    const int r = acc_row<DVT>();
    const int g = col_group();
    // this thread's U^T values of the current chunk (rows t of its column half)
    float ureg[C / 2];
    if (r >= 0) {
        const float* up = U + (bh * d.Tp + g * (C / 2)) * Dv + n0 + r;
#pragma unroll
        for (int i = 0; i < C / 2; ++i) ureg[i] = up[(int64_t)i * Dv];
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tb = tmem_sh;
    const int halfk = Dk / 2;
    const int64_t sbase = bh * Dk * Dv + n0;
    // initial state -> TMEM
    for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = (r >= 0 && p.state0) ? p.state0[sbase + (int64_t)(cc + i) * Dv + r] : 0.f;
        tc::tmem_st16(tc::tmem_addr(tb, lane0(), kColState + cc), v);
    }
    tc::tmem_wait_st();
    const tc::Tile tSt = tc::panel_tile(sm + L.St, DVT, true);
    const tc::Tile tQ = tile_of(sm + L.Q, Dk, true);
    const tc::Tile tW = tc::panel_tile(sm + L.W, C, true);
    const tc::Tile tKmn = tile_of(sm + L.K, Dk, false);
    const tc::Tile tP = tc::panel_tile(sm + L.P, C, true);
    const tc::Tile tDt = tile_of(sm + L.Dt, C, true), tDlo = tile_of(sm + L.Dlo, C, true);
    const tc::Tile tDe = tile_of(sm + L.De, C, true), tDelo = tile_of(sm + L.Delo, C, true);
    uint32_t phase = 0, phW = 0, phP = 0;
    bool ok = true;

    for (int64_t c = 0; c < d.NC; ++c) {
        const float* vb = vecs + (c & 1) * 4 * C;
        const float* gmv = vb;
        const float* kev = vb + 3 * C;
        const float* qsv = vb + 2 * C;
        const int64_t t0 = c * C;
        if (warp == kStoreWarp) tc::bulk_wait_read_all();  // St / Delta images of c - 1 read out
        tc::tc_fence_before();
        __syncthreads();  // (A) vectors of chunk c ready; output rows of c - 1 staged
        tc::tc_fence_after();
        if (warp == kStoreWarp && c > 0) store_o(c - 1);
        // step 1: S^T -> bf16 operand (= checkpoint image); S^T *= gam_63
        state_to_operand<DVT>(tb, sm + L.St, Dk, gmv[C - 1]);
        tc::cp_async_wait_all();
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();  // (B)
        tc::tc_fence_after();
        // step 2: Delta^T acc = S^T W^T, QS = S^T Q^T
        if (tid == 0) {
            ok = tc::mbar_wait(&barW, phW, &g_err_scantc) && ok;
            phW ^= 1u;
            tc::mma_tile(tb + kColA, tSt, tW, DVT, C, Dk, false);
            tc::mma_tile(tb + kColB, tSt, tQ, DVT, C, Dk, false);
            tc::mma_commit(&bar);
        }
        if (warp == kStoreWarp)
            store_state_image<DVT>(ckimg + (bh * d.NC + c) * (int64_t)Dk * Dv * 2, sm + L.St, Dk, Dv, n0);
        ok = tc::mbar_wait(&bar, phase, &g_err_scantc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        if (tid == 0 && c + 1 < d.NC) load_w(c + 1);
        // step 3: Delta^T = U^T - acc as a two-term bf16 operand (hi + lo) and
        // (Delta^T diag(e r_k)) likewise
        if (ok) {
            for (int cc = g * (C / 2); cc < (g + 1) * (C / 2); cc += 16) {
                float v[16];
                tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColA + cc), v);
                tc::tmem_wait_ld();
                if (r >= 0) {
                    float lo[16], de[16], delo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = cc + i;
                        const float dl = ureg[cc - g * (C / 2) + i] - v[i];
                        v[i] = dl;
                        lo[i] = dl - __bfloat162float(__float2bfloat16_rn(dl));
                        de[i] = dl * kev[t];
                        delo[i] = de[i] - __bfloat162float(__float2bfloat16_rn(de[i]));
                    }
                    st_bf16x8(sm + L.Dt + canon(cc, r, C), v);
                    st_bf16x8(sm + L.Dt + canon(cc + 8, r, C), v + 8);
                    st_bf16x8(sm + L.Dlo + canon(cc, r, C), lo);
                    st_bf16x8(sm + L.Dlo + canon(cc + 8, r, C), lo + 8);
                    st_bf16x8(sm + L.De + canon(cc, r, C), de);
                    st_bf16x8(sm + L.De + canon(cc + 8, r, C), de + 8);
                    st_bf16x8(sm + L.Delo + canon(cc, r, C), delo);
                    st_bf16x8(sm + L.Delo + canon(cc + 8, r, C), delo + 8);
                }
            }
        }
        // U of the next chunk: in flight while the step-4 MMAs and the output run
        if (c + 1 < d.NC && r >= 0) {
            const float* up = U + (bh * d.Tp + t0 + C + g * (C / 2)) * Dv + n0 + r;
#pragma unroll
            for (int i = 0; i < C / 2; ++i) ureg[i] = up[(int64_t)i * Dv];
        }
        if (warp == kStoreWarp) tc::bulk_wait_read_all();  // output rows of c - 1 read out of Ob
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();  // (C)
        tc::tc_fence_after();
        // step 4: PDelta = Delta^T P^T;  S^T += (Delta^T diag(e r_k)) K
        if (tid == 0) {
            ok = tc::mbar_wait(&barP, phP, &g_err_scantc) && ok;
            phP ^= 1u;
            tc::mma_tile(tb + kColC, tDt, tP, DVT, C, C, false);
            tc::mma_tile(tb + kColC, tDlo, tP, DVT, C, C, true);
            tc::mma_tile(tb + kColState, tDe, tKmn, DVT, Dk, C, true);
            tc::mma_tile(tb + kColState, tDelo, tKmn, DVT, Dk, C, true);
            tc::mma_commit(&bar);
        }
        if (warp == kStoreWarp) store_delta(c);
        if (c + 1 < d.NC) {
            fetch_q(c + 1);
            chunk_vectors(d, p, bb, h, j, c + 1, vecs + ((c + 1) & 1) * 4 * C);
        }
        ok = tc::mbar_wait(&bar, phase, &g_err_scantc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        if (tid == 0 && c + 1 < d.NC) load_p(c + 1);
        if (c + 1 < d.NC) fetch_k(c + 1);
        tc::cp_async_commit();
        // step 5: O^T = diag(gam r_q / sqrt(Dk)) QS + PDelta -> staged output rows
        if (ok) {
            for (int cc = g * (C / 2); cc < (g + 1) * (C / 2); cc += 16) {
                float a[16], b2[16];
                tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColB + cc), a);
                tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColC + cc), b2);
                tc::tmem_wait_ld();
                if (r >= 0) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = cc + i;
                        Ob[t * DVT + r] = __float2bfloat16_rn(qsv[t] * a[i] + b2[i]);
                    }
                }
            }
        }
        tc::fence_async_smem();  // staged rows -> the bulk stores issued after (A)
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == kStoreWarp) store_o(d.NC - 1);
    for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColState + cc), v);
        tc::tmem_wait_ld();
        if (r >= 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) p.state_T[sbase + (int64_t)(cc + i) * Dv + r] = v[i];
        }
    }
    if (warp == kStoreWarp) tc::bulk_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------------------
// backward (reverse) scan
// ---------------------------------------------------------------------------
template <int DVT>
__global__ void __launch_bounds__(kThreads, 1) bwd_scan_tc_kernel(Dims d, Ptrs p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar, barW, barP;
    __shared__ uint32_t tmem_sh;
    const int tile = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int n0 = tile * DVT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ScanSmem L = scan_plan(Dk, DVT, false);
    float* vecs = reinterpret_cast<float*>(sm + L.vec);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(p.d_o);
    const uint8_t* Wimg = static_cast<const uint8_t*>(p.W);
    const uint8_t* Pimg = static_cast<const uint8_t*>(p.P);
    uint8_t* dsimg = reinterpret_cast<uint8_t*>(p.dSck);
    uint8_t* dbimg = reinterpret_cast<uint8_t*>(p.Dbar);
    const int64_t ldq = d.Hk * Dk, ldo = d.Hv * Dv;
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const uint32_t wbytes = (uint32_t)(C * Dk * 2), pbytes = (uint32_t)(C * C * 2);

    auto nvalid = [&](int64_t c) { return (int)(d.T - c * C < C ? d.T - c * C : C); };
    auto load_w = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barW, wbytes);
        tc::bulk_g2s(sm + L.W, Wimg + (bh * d.NC + c) * wbytes, wbytes, &barW);
    };
    auto load_p = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barP, pbytes);
        tc::bulk_g2s(sm + L.P, Pimg + (bh * d.NC + c) * pbytes, pbytes, &barP);
    };
    auto fetch = [&](int64_t c) {  // Obar, K, Q of chunk c
        const int64_t t0 = c * C;
        const int nv = nvalid(c);
        cpa_tile(sm + L.O, dO + ((int64_t)bb * d.T + t0) * ldo + (int64_t)h * Dv + n0, ldo, DVT, nv);
        cpa_tile(sm + L.K, k + ((int64_t)bb * d.T + t0) * ldq + (int64_t)j * Dk, ldq, Dk, nv);
        cpa_tile(sm + L.Q, q + ((int64_t)bb * d.T + t0) * ldq + (int64_t)j * Dk, ldq, Dk, nv);
    };
    // Obar^T diag(gam r_q / sqrt(Dk)) as a two-term bf16 operand, from the Obar tile
    auto build_os = [&](const float* qsv) {
        const int cpr = DVT / 8;
        for (int e = tid; e < C * cpr; e += blockDim.x) {
            int row, cc;
            chunk_rc(e, cpr, row, cc);
            const uint32_t off = canon(cc * 8, row, DVT);
            const uint4 u = *reinterpret_cast<const uint4*>(sm + L.O + off);
            const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&u);
            const float s = qsv[row];
            float v[8], lo[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(hh[i]);
                v[2 * i] = f.x * s;
                v[2 * i + 1] = f.y * s;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) lo[i] = v[i] - __bfloat162float(__float2bfloat16_rn(v[i]));
            st_bf16x8(sm + L.Os + off, v);
            st_bf16x8(sm + L.Oslo + off, lo);
        }
    };

    if (warp == 0) {
        tc::tmem_alloc(&tmem_sh, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_init(&barW, 1);
        tc::mbar_init(&barP, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();  // barriers initialised
    const int64_t cl = d.NC - 1;
    if (tid == 0) {
        load_w(cl);
        load_p(cl);
    }
    fetch(cl);
    tc::cp_async_commit();
    chunk_vectors(d, p, bb, h, j, cl, vecs + (cl & 1) * 4 * C);
    tc::cp_async_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    build_os(vecs + (cl & 1) * 4 * C + 2 * C);
    const uint32_t tb = tmem_sh;
    const int r = acc_row<DVT>();
    const int g = col_group();
    const int halfk = Dk / 2;
    const int64_t sbase = bh * Dk * Dv + n0;
    for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = (r >= 0 && p.d_state_T) ? p.d_state_T[sbase + (int64_t)(cc + i) * Dv + r] : 0.f;
        tc::tmem_st16(tc::tmem_addr(tb, lane0(), kColState + cc), v);
    }
    tc::tmem_wait_st();
    tc::fence_async_smem();  // Os / Oslo written by plain stores
    const tc::Tile tSt = tc::panel_tile(sm + L.St, DVT, true);
    const tc::Tile tOmn = tile_of(sm + L.O, DVT, false), tOsmn = tile_of(sm + L.Os, DVT, false);
    const tc::Tile tOslomn = tile_of(sm + L.Oslo, DVT, false);
    const tc::Tile tPmn = tc::panel_tile(sm + L.P, C, false);
    const tc::Tile tK = tile_of(sm + L.K, Dk, true);
    const tc::Tile tQmn = tile_of(sm + L.Q, Dk, false);
    const tc::Tile tWmn = tc::panel_tile(sm + L.W, C, false);
    const tc::Tile tNDb = tile_of(sm + L.Dt, C, true);
    uint32_t phase = 0, phW = 0, phP = 0;
    bool ok = true;

    for (int64_t c = cl; c >= 0; --c) {
        const float* vb = vecs + (c & 1) * 4 * C;
        const float* gmv = vb;
        const float* kev = vb + 3 * C;
        if (warp == kStoreWarp) tc::bulk_wait_read_all();  // images of chunk c + 1 read out
        tc::tc_fence_before();
        __syncthreads();  // (A)
        tc::tc_fence_after();
        // step 1: Sbar^T -> bf16 operand (= chunk-end cotangent image); *= gam_63
        state_to_operand<DVT>(tb, sm + L.St, Dk, gmv[C - 1]);
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();  // (B)
        tc::tc_fence_after();
        // step 2: A1 = Obar^T P, A2 = Sbar^T K^T, Sbar^T += Obar^T diag(s) Q
        if (tid == 0) {
            ok = tc::mbar_wait(&barP, phP, &g_err_scantc) && ok;
            phP ^= 1u;
            tc::mma_tile(tb + kColA, tOmn, tPmn, DVT, C, C, false);
            tc::mma_tile(tb + kColB, tSt, tK, DVT, C, Dk, false);
            tc::mma_tile(tb + kColState, tOsmn, tQmn, DVT, Dk, C, true);
            tc::mma_tile(tb + kColState, tOslomn, tQmn, DVT, Dk, C, true);
            tc::mma_commit(&bar);
        }
        if (warp == kStoreWarp)
            store_state_image<DVT>(dsimg + (bh * d.NC + c) * (int64_t)Dk * Dv * 2, sm + L.St, Dk, Dv, n0);
        ok = tc::mbar_wait(&bar, phase, &g_err_scantc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        // Obar, K, Q, P of chunk c - 1 load while the epilogue and step 4 run
        if (c > 0) {
            if (tid == 0) load_p(c - 1);
            fetch(c - 1);
            chunk_vectors(d, p, bb, h, j, c - 1, vecs + ((c - 1) & 1) * 4 * C);
        }
        tc::cp_async_commit();
        // step 3: -Dbar^T = -(A1 + A2 diag(e r_k)) as a bf16 operand
        if (ok) {
            for (int cc = g * (C / 2); cc < (g + 1) * (C / 2); cc += 16) {
                float a[16], b2[16];
                tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColA + cc), a);
                tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColB + cc), b2);
                tc::tmem_wait_ld();
                if (r >= 0) {
                    float nd[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) nd[i] = -(a[i] + kev[cc + i] * b2[i]);
                    st_bf16x8(sm + L.Dt + canon(cc, r, C), nd);
                    st_bf16x8(sm + L.Dt + canon(cc + 8, r, C), nd + 8);
                }
            }
        }
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();  // (C)
        tc::tc_fence_after();
        // step 4: Sbar^T += (-Dbar^T) W
        if (tid == 0) {
            ok = tc::mbar_wait(&barW, phW, &g_err_scantc) && ok;
            phW ^= 1u;
            tc::mma_tile(tb + kColState, tNDb, tWmn, DVT, Dk, C, true);
            tc::mma_commit(&bar);
        }
        if (warp == kStoreWarp) {
            if (lane == 0)
                tc::bulk_s2g(dbimg + (bh * d.NC + c) * (int64_t)C * Dv * 2 + (int64_t)n0 * 128,
                             sm + L.Dt, (uint32_t)(DVT * 128));
            tc::bulk_commit();
        }
        ok = tc::mbar_wait(&bar, phase, &g_err_scantc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        if (c > 0) {
            if (tid == 0) load_w(c - 1);
            tc::cp_async_wait_all();
            __syncthreads();  // Obar tile and vectors of chunk c - 1 in place
            build_os(vecs + ((c - 1) & 1) * 4 * C + 2 * C);
            tc::fence_async_smem();
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_addr(tb, lane0(), kColState + cc), v);
        tc::tmem_wait_ld();
        if (r >= 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) p.dstate0[sbase + (int64_t)(cc + i) * Dv + r] = v[i];
        }
    }
    if (warp == kStoreWarp) tc::bulk_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

template <int DVT>
cudaError_t launch_scan(const Dims& d, const Ptrs& p, cudaStream_t s, bool fwd) {
    const ScanSmem L = scan_plan((int)d.Dk, DVT, fwd);
    const size_t smem = L.total + 1024;
    dim3 grid((unsigned)(d.Dv / DVT), (unsigned)d.Hv, (unsigned)d.B);
    if (fwd) {
        auto kern = fwd_scan_tc_kernel<DVT>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, s>>>(d, p);
    } else {
        auto kern = bwd_scan_tc_kernel<DVT>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, s>>>(d, p);
    }
    count_launches(1);
    return cudaPeekAtLastError();
}

uint32_t scan_need(int Dk, int dvt) {
    const uint32_t a = scan_plan(Dk, dvt, true).total, b = scan_plan(Dk, dvt, false).total;
    return (a > b ? a : b) + 2048;
}

// Dv tile per CTA: 128 (M = 128 MMAs) when it divides Dv and fits in shared
// memory, else 64 (M = 64); 0 if neither applies
int scan_dvt(const Dims& d) {
    if (d.Dv % 128 == 0 && scan_need((int)d.Dk, 128) <= 227u * 1024u) return 128;
    if (d.Dv % 64 == 0 && scan_need((int)d.Dk, 64) <= 227u * 1024u) return 64;
    return 0;
}

}  // namespace

bool scan_tc_supported(const Dims& d) {
    if (d.dtype != 1) return false;
    if (d.Dk % 32 || d.Dk > 256) return false;
    return scan_dvt(d) != 0;
}

cudaError_t launch_fwd_scan_tc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    if (scan_ta_supported(d) && p.tmaps) return launch_fwd_scan_ta(d, p, s);
    return scan_dvt(d) == 128 ? launch_scan<128>(d, p, s, true) : launch_scan<64>(d, p, s, true);
}

cudaError_t launch_bwd_scan_tc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    if (scan_ta_supported(d) && p.tmaps) return launch_bwd_scan_ta(d, p, s);
    return scan_dvt(d) == 128 ? launch_scan<128>(d, p, s, false) : launch_scan<64>(d, p, s, false);
}

}  // namespace gdn
