// gdn_scan_ta.cuh -- the reverse chunk scan for 128-row value tiles (M = 128
// tcgen05 MMAs, the state cotangent held in tensor memory) as a device
// function, with the helpers it shares with the forward scan.  Included by
// gdn_scan_ta.cu (the forward scan and the stand-alone reverse scan) and by
// gdn_bwd_tc.cu (the reverse scan and the per-chunk gradients in one launch).
//
// Same recurrence as gdn_scan_tc.cu (mlx-lm PR "Add gated_delta_update VJP",
// "What this PR adds" and "Design notes": chunk 64, sequential over chunks).
// Backward (reverse over chunks), per chunk with Sbar^T the state cotangent:
//   A1 = Obar^T P,  A2 = Sbar^T K^T  (Sbar^T as bf16 pairs in TMEM),
//   Sbar^T <- gam_63 Sbar^T + (Obar^T diag(gam r_q / sqrt(Dk))) Q   (hi + lo),
//   -Dbar^T = -(A1 + A2 diag(e r_k)),   Sbar^T += (-Dbar^T) W.
// Obar tiles by TMA two chunks ahead (double-buffered); q, k, P and W images by
// bulk copy; the Sbar'^T image stored from registers, the -Dbar^T image
// (double-buffered, it is also the step-4 operand) by bulk stores.  TMEM: [0, Dk)
// state, [Dk, Dk + 128) Sbar^T bf16 pairs, then A1 and A2 (64 columns each).
#pragma once

#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace ta {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int DVT = 128;
constexpr int kStoreWarp = 1;
constexpr uint32_t kRawBytes = C * 8 + 2 * C * 4;  // gam (fp64) | r_q | r_k of one chunk

__device__ __forceinline__ uint32_t canon(int x, int y, int ncols) {
    return (uint32_t)(x >> 3) * 128u + (uint32_t)(y >> 3) * (uint32_t)ncols * 16u +
           (uint32_t)(y & 7) * 16u + (uint32_t)(x & 7) * 2u;
}

// gam, e, gam r_q / sqrt(Dk), e r_k of one chunk from its raw block; with
// per-key-channel gates (KC) the raw block is the chunk's decay exp(Gamma_63,i)
// of each key channel i, copied to v[0 .. Dk)
template <bool KC>
__device__ __forceinline__ void vectors_from_raw(const uint8_t* raw, float* v, int Dk) {
    const int i = threadIdx.x;
    if constexpr (KC) {
        for (int c = i; c < Dk; c += kThreads) v[c] = reinterpret_cast<const float*>(raw)[c];
    } else if (i < C) {
        const double* G = reinterpret_cast<const double*>(raw);
        const float* rq = reinterpret_cast<const float*>(raw + C * 8);
        const float* rk = reinterpret_cast<const float*>(raw + C * 12);
        const float gm = expf((float)G[i]);
        const float e = expf((float)(G[C - 1] - G[i]));
        v[i] = gm;
        v[C + i] = e;
        v[2 * C + i] = gm * rq[i] * rsqrtf((float)Dk);
        v[3 * C + i] = e * rk[i];
    }
}

// q tile (panel layout, 16-byte chunk e holds step e % 64) scaled in place by

struct TbSmem {
    uint32_t P, K, Q, W, O, Os, Oslo, ND, raw, vec, total;
};

__host__ __device__ inline TbSmem tb_plan(int Dk) {
    TbSmem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    s.P = take(C * C * 2);      // panel images / TMA panel tiles (64 rows)
    s.K = take(C * Dk * 2);
    s.Q = take(C * Dk * 2);
    s.W = take(C * Dk * 2);
    s.O = take(2 * C * DVT * 2);  // Obar tiles of two chunks, panel (x = value column)
    s.Os = take(C * DVT * 2);   // Obar diag(gam r_q / sqrt(Dk)), hi and lo, same layout
    s.Oslo = take(C * DVT * 2);
    s.ND = take(2 * DVT * C * 2);  // -Dbar^T of two chunks (canonical, x = step): operand and image
    s.raw = take(2 * kRawBytes);
    s.vec = take(2 * 4 * C * 4);
    s.total = o;
    return s;
}

// Obar tile (panel layout, chunk e holds step e % 64) -> Os, Oslo: the tile
// scaled by gam r_q / sqrt(Dk) of its step, as hi + lo bf16 (KC: the per-step
// factors are in the Q operand already, so Os = Obar and Oslo = 0)
template <bool KC>
__device__ __forceinline__ void build_os(const uint8_t* O, uint8_t* Os, uint8_t* Oslo,
                                         const uint8_t* raw, int Dk) {
    const int t = threadIdx.x & (C - 1);
    const double* G = reinterpret_cast<const double*>(raw);
    const float* rq = reinterpret_cast<const float*>(raw + C * 8);
    const float s = KC ? 1.f : expf((float)G[t]) * rq[t] * rsqrtf((float)Dk);
    for (int e = threadIdx.x; e < C * DVT / 8; e += kThreads) {
        uint4 u = reinterpret_cast<const uint4*>(O)[e];
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&u);
        uint4 hi, lo;
        uint32_t* hw = reinterpret_cast<uint32_t*>(&hi);
        uint32_t* lw = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            const float x = f.x * s, y = f.y * s;
            hw[i] = tc::pack_bf16(x, y);
            const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[i]));
            lw[i] = tc::pack_bf16(x - hf.x, y - hf.y);
        }
        reinterpret_cast<uint4*>(Os)[e] = hi;
        reinterpret_cast<uint4*>(Oslo)[e] = lo;
    }
}

// width of a segment map: the offset part (Dv columns), then the linear part (Dk
// columns, padded to whole value tiles)
__host__ __device__ inline int64_t seg_wd(int64_t Dk, int64_t Dv) { return Dv + (Dk + DVT - 1) / DVT * DVT; }

// The reverse scan of value tile `tile` of (batch bb, value head h), run by a
// CTA of kThreads + 64 threads with tb_plan(Dk).total + 1024 bytes of dynamic
// shared memory and all 512 TMEM columns.  err: the caller's error word for
// bounded waits.  progress (may be null): after the -Dbar^T and Sbar'^T images
// of a chunk are complete in global memory, progress[b Hv + h] goes up by one
// (two chunks after the chunk itself, the last two at the end), so a consumer
// may read the images of chunk c of this tile once the count reaches NC - c.
// relinquish: give up the CTA's TMEM allocation permit after the allocation
// (false when the CTA allocates again after this body).
// Segments (sg.nseg > 1; progress null): segment t counts from the top, chunks
// hi - sg.len .. hi - 1 with hi = NC - t sg.len (the bottom one may be shorter).
// Mode 0 scans segment t from d_state_T (t = 0) or from the chained start state
// sg.start[t - 1], storing its images; the bottom segment writes dstate0.  Mode 1
// (maps, t < nseg - 1) scans it from zero (offset part, the Dv value tiles) and,
// with Obar = 0, from the identity (linear part, tiles over Dk padded), storing
// only the end states, into sg.maps[t] with rows of seg_wd(Dk, Dv).
// KC: per-key-channel gates.  The Q and K operands are then the per-value-head
// images Q_r = qh o exp(Gamma) and K_d = kh o exp(Gamma_63 - Gamma) (qimg, kimg
// indexed by (b, value head)), the state cotangent decays column by column by
// the chunk's exp(Gamma_63, i) (p.ecd), and no per-step factor scales Obar or A2.
template <bool KC>
__device__ __forceinline__ void bwd_scan_ta_body(const Dims& d, const Ptrs& p, const Tmaps& tm,
                                                 int tile, int h, int bb, const ScanSeg& sg, int t,
                                                 unsigned int* err, unsigned int* progress,
                                                 bool relinquish) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar, barW, barQ, barK, barP, barO[2], barR[2];
    __shared__ uint32_t tmem_sh;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int n0 = tile * DVT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = tid < kThreads;
    const bool prod = warp == kThreads / 32 && lane == 0;
    // warp 9 issues the second MMA chain of step 2 (one thread issues a tcgen05.mma
    // about every 80 cycles, so two issuing warps overlap the chains)
    const bool prod2 = warp == kThreads / 32 + 1 && lane == 0;
    const bool storer = warp == kStoreWarp && lane == 0;
    const int r = 32 * (warp & 3) + lane;
    const int g = (tid >> 7) & 1;
    const uint32_t lb = 32u * (uint32_t)(warp & 3);
    const TbSmem L = tb_plan(Dk);
    const uint32_t aop = (uint32_t)Dk, kA1 = (uint32_t)Dk + 128, kA2 = (uint32_t)Dk + 192;
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const uint32_t kbytes = (uint32_t)(C * Dk * 2), pbytes = (uint32_t)(C * C * 2);
    const uint32_t obytes = (uint32_t)(C * DVT * 2);
    const uint8_t* Wimg = static_cast<const uint8_t*>(p.W);
    const uint8_t* Pimg = static_cast<const uint8_t*>(p.P);
    uint8_t* dsimg = reinterpret_cast<uint8_t*>(p.dSck);
    uint8_t* dbimg = reinterpret_cast<uint8_t*>(p.Dbar);
    const int64_t NC = d.NC;
    // chunks lo .. hi - 1 of segment t, walked downwards
    const int64_t hi = NC - (int64_t)t * sg.len;
    const int64_t lo = hi - sg.len > 0 ? hi - sg.len : 0;
    const bool maps = sg.mode != 0;    // segment maps: no images, no progress
    const bool oz = maps && n0 >= Dv;  // linear part of a map: Obar = 0, identity start

    // m = hi - 1 - c counts processed chunks: ring slots and mbarrier parities follow it
    auto load_w = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barW, kbytes);
        tc::bulk_g2s(sm + L.W, Wimg + (bh * NC + c) * kbytes, kbytes, &barW);
    };
    auto load_p = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barP, pbytes);
        tc::bulk_g2s(sm + L.P, Pimg + (bh * NC + c) * pbytes, pbytes, &barP);
    };
    // (b, key head): q / k images of its chunks; (b, value head) with KC
    const int64_t kq = KC ? bh : (int64_t)bb * d.Hk + j;
    auto load_kq = [&](int64_t c) {
        tc::mbar_arrive_expect_tx(&barK, kbytes);
        tc::bulk_g2s(sm + L.K, static_cast<const uint8_t*>(p.kimg) + (kq * NC + c) * kbytes, kbytes, &barK);
        tc::mbar_arrive_expect_tx(&barQ, kbytes);
        tc::bulk_g2s(sm + L.Q, static_cast<const uint8_t*>(p.qimg) + (kq * NC + c) * kbytes, kbytes, &barQ);
    };
    // Obar tile of chunk c -> buffer (hi - 1 - c) & 1
    auto obuf = [&](int64_t c) { return sm + L.O + ((hi - 1 - c) & 1) * obytes; };
    auto load_o = [&](int64_t c) {
        uint64_t* b = &barO[(hi - 1 - c) & 1];
        tc::mbar_arrive_expect_tx(b, obytes);
        tc::tma_load_5d(obuf(c), &tm.dO, 0, (int)(c * C), n0 / 8, h, bb, b);
    };
    auto load_raw = [&](int64_t c) {
        const int s = (int)((hi - 1 - c) & 1);
        uint8_t* dst = sm + L.raw + s * kRawBytes;
        if constexpr (KC) {
            tc::mbar_arrive_expect_tx(&barR[s], (uint32_t)(Dk * 4));
            tc::bulk_g2s(dst, p.ecd + (bh * NC + c) * Dk, (uint32_t)(Dk * 4), &barR[s]);
            return;
        }
        tc::mbar_arrive_expect_tx(&barR[s], kRawBytes);
        tc::bulk_g2s(dst, p.gam + bh * d.Tp + c * C, C * 8, &barR[s]);
        tc::bulk_g2s(dst + C * 8, p.rq + ((int64_t)bb * d.Hk + j) * d.Tp + c * C, C * 4, &barR[s]);
        tc::bulk_g2s(dst + C * 12, p.rk + ((int64_t)bb * d.Hk + j) * d.Tp + c * C, C * 4, &barR[s]);
    };
    // -Dbar^T tile of chunk c (and its image source) -> buffer (hi - 1 - c) & 1
    auto ndbuf = [&](int64_t c) { return sm + L.ND + ((hi - 1 - c) & 1) * (uint32_t)(DVT * C * 2); };
    auto store_dbar = [&](int64_t c) {  // storer; the caller commits
        tc::bulk_s2g(dbimg + (bh * NC + c) * (int64_t)C * Dv * 2 + (int64_t)n0 * 128, ndbuf(c),
                     (uint32_t)(DVT * 128));
    };

    if (warp == 0) {
        tc::tmem_alloc(&tmem_sh, 512);
        if (relinquish) tc::tmem_relinquish();
    }
    if (prod) {
        tc::mbar_init(&bar, 2);  // one commit (or arrival) from each issuer per MMA round
        tc::mbar_init(&barW, 1);
        tc::mbar_init(&barQ, 1);
        tc::mbar_init(&barK, 1);
        tc::mbar_init(&barP, 1);
        tc::mbar_init(&barO[0], 1);
        tc::mbar_init(&barO[1], 1);
        tc::mbar_init(&barR[0], 1);
        tc::mbar_init(&barR[1], 1);
        tc::fence_mbar_init();
    }
    __syncthreads();  // barriers initialised
    if (prod) {
        load_w(hi - 1);
        load_kq(hi - 1);
        load_p(hi - 1);
        if (!oz) {
            load_o(hi - 1);
            if (hi - lo > 1) load_o(hi - 2);
        }
        load_raw(hi - 1);
        if (hi - lo > 1) load_raw(hi - 2);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tb = tmem_sh;
    const int halfk = Dk / 2;
    // cotangent entering the segment (rows dk, row stride Dv): d_state_T for the
    // top segment, the chained one below it; zero / the identity for the maps
    const float* sin = nullptr;
    if (!maps && t == 0 && p.d_state_T) sin = p.d_state_T + bh * Dk * Dv + n0;
    if (!maps && t > 0 && sg.start) sin = sg.start + ((int64_t)(t - 1) * d.B * d.Hv + bh) * Dk * Dv + n0;
    if (!maps && sg.sin) sin = sg.sin + bh * Dk * Dv + n0;
    bool ok = true;
    if (epi) {
        for (int cc = g * halfk; cc < (g + 1) * halfk; cc += 16) {  // final cotangent -> TMEM
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = oz ? (cc + i == n0 - Dv + r ? 1.f : 0.f) : sin ? sin[(int64_t)(cc + i) * Dv + r] : 0.f;
            tc::tmem_st16(tc::tmem_addr(tb, lb, cc), v);
        }
        tc::tmem_wait_st();
        ok = tc::mbar_wait(&barR[0], 0, err);
        vectors_from_raw<KC>(sm + L.raw, reinterpret_cast<float*>(sm + L.vec), Dk);
        if (!oz) {
            ok = tc::mbar_wait(&barO[0], 0, err) && ok;
            build_os<KC>(obuf(hi - 1), sm + L.Os, sm + L.Oslo, sm + L.raw, Dk);
        }
        tc::fence_async_smem();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // A = Obar^T: x = dv = M (tile of the current chunk's buffer, below)
    const tc::Tile tOsmn = tc::panel_tile(sm + L.Os, C, false);
    const tc::Tile tOslomn = tc::panel_tile(sm + L.Oslo, C, false);
    const tc::Tile tPmn = tc::panel_tile(sm + L.P, C, false);      // B = P: x = s = N
    const tc::Tile tK = tc::panel_tile(sm + L.K, C, true);         // B = K^T: x = dk = K
    const tc::Tile tQmn = tc::panel_tile(sm + L.Q, C, false);      // B = Q: x = dk = N
    const tc::Tile tWmn = tc::panel_tile(sm + L.W, C, false);      // B = W: x = dk = N
    tc::Tile tND;                                                  // A = -Dbar^T: x = t = K
    tND.xs = 128;
    tND.ys = (uint32_t)C * 16u;
    tND.k_major = true;
    uint32_t phase = 0;

    for (int64_t c = hi - 1; c >= lo; --c) {
        const int64_t m = hi - 1 - c;
        if (progress && m >= 2 && epi) {
            // chunk c + 2 is complete in global memory: its Sbar'^T image went out
            // by generic stores in its step 2, its -Dbar^T image by the bulk store
            // committed in its step 4, and only chunk c + 1's group may still be
            // in flight
            if (storer) {
                tc::bulk_wait_but1();
                tc::fence_async_global();  // the bulk store's writes, before the release
            }
            __threadfence();
            tc::named_sync(1, kThreads);
            if (storer) {
                __threadfence();
                atomicAdd(progress + (int64_t)bb * d.Hv + h, 1u);
            }
        }
        const float* vb = reinterpret_cast<const float*>(sm + L.vec) + (m & 1) * 4 * C;
        const float* kev = vb + 3 * C;
        const float gC = vb[C - 1];
        // step 1: Sbar^T -> A operand (bf16 pairs in TMEM); Sbar^T *= gam_63
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
                tc::tmem_st16u(tc::tmem_addr(tb, lb, aop + cb / 2), w);
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
        if (storer) tc::bulk_wait_read_but1();  // -Dbar image of chunk c + 2 read out of its buffer
        tc::tc_fence_before();
        __syncthreads();  // (B)
        tc::tc_fence_after();
        const tc::Tile tOmn = tc::panel_tile(obuf(c), C, false);
        tND.base = tc::smem_u32(ndbuf(c));
        if (prod2) {
            // step 2, second issuer: A1 = Obar^T P and Sbar^T += Os Q + Oslo Q, two
            // chains interleaved.  The P and Q copies are waited for even when they
            // are not read (a map's linear part): the producer's next copy into the
            // buffer re-arms the barrier, which it may only do once this phase is
            // complete.
            ok = tc::mbar_wait(&barP, (uint32_t)(m & 1), err) && ok;
            ok = tc::mbar_wait(&barQ, (uint32_t)(m & 1), err) && ok;
            if (!oz) {
                const uint32_t id64 = tc::idesc_bf16(DVT, C, true, true);
                const uint32_t idq = tc::idesc_bf16(DVT, Dk, true, true);
                uint64_t dO = tOmn.desc(0), dP = tPmn.desc(0), dOs = tOsmn.desc(0), dQ = tQmn.desc(0),
                         dOl = tOslomn.desc(0);
                const uint64_t iO = tOmn.desc_step(), iP = tPmn.desc_step(), iOs = tOsmn.desc_step(),
                               iQ = tQmn.desc_step(), iOl = tOslomn.desc_step();
                for (int k = 0; k < C; k += 16) {
                    tc::mma_bf16(tb + kA1, dO, dP, id64, k > 0);
                    tc::mma_bf16(tb, dOs, dQ, idq, 1u);
                    tc::mma_bf16(tb, dOl, dQ, idq, 1u);
                    dO += iO; dP += iP; dOs += iOs; dQ += iQ; dOl += iOl;
                }
                tc::mma_commit(&bar);
            } else {
                tc::mbar_arrive(&bar);  // nothing to issue in this round
            }
            phase ^= 1u;
        } else if (prod) {
            // step 2: A2 = Sbar^T K^T (A1 and the state update by the second issuer)
            ok = tc::mbar_wait(&barK, (uint32_t)(m & 1), err) && ok;
            const uint32_t id2 = tc::idesc_bf16(DVT, C, false, false);
            uint64_t dK = tK.desc(0);
            const uint64_t iK = tK.desc_step();
            for (int k = 0; k < Dk; k += 16) {
                tc::mma_bf16_ta(tb + kA2, tb + aop + k / 2, dK, id2, k > 0);
                dK += iK;
            }
            tc::mma_commit(&bar);
            ok = tc::mbar_wait(&bar, phase, err) && ok;
            phase ^= 1u;
            if (c > lo) {  // P, K, Q tiles (and this chunk's Obar buffer) are free
                if (!oz && c > lo + 1) load_o(c - 2);
                load_p(c - 1);
                load_kq(c - 1);
            }
        } else if (epi) {
            // meanwhile: the Sbar'^T image, straight from the A operand to global
            // memory (each warp store covers 32 consecutive 16-byte rows of a panel)
            uint8_t* img = dsimg + (bh * NC + c) * (int64_t)Dk * Dv * 2;
            for (int cb = g * (Dk / 4); !maps && cb < (g + 1) * (Dk / 4); cb += 16) {
                uint32_t w[16];
                tc::tmem_ld16u(tc::tmem_addr(tb, lb, aop + cb), w);
                tc::tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4*>(img + tc::panel_off(2 * cb + 8 * q4, n0 + r, Dv)) =
                        make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
            }
            ok = tc::mbar_wait(&bar, phase, err) && ok;
            phase ^= 1u;
            tc::tc_fence_after();
            // step 3: -Dbar^T = -(A1 + A2 diag(e r_k)) -> operand / image tile
            float a1[2][16], a2[2][16];
            if (oz) {  // no Obar: A1 was not formed (its TMEM columns are not read)
#pragma unroll
                for (int i = 0; i < 16; ++i) a1[0][i] = a1[1][i] = 0.f;
            } else {
                tc::tmem_ld16(tc::tmem_addr(tb, lb, kA1 + 32 * g), a1[0]);
                tc::tmem_ld16(tc::tmem_addr(tb, lb, kA1 + 32 * g + 16), a1[1]);
            }
            tc::tmem_ld16(tc::tmem_addr(tb, lb, kA2 + 32 * g), a2[0]);
            tc::tmem_ld16(tc::tmem_addr(tb, lb, kA2 + 32 * g + 16), a2[1]);
            tc::tmem_wait_ld();
            uint32_t nd[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t0 = 32 * g + 2 * i;
                const float e0 = KC ? 1.f : kev[t0], e1 = KC ? 1.f : kev[t0 + 1];
                const float x = -(a1[(2 * i) >> 4][(2 * i) & 15] + e0 * a2[(2 * i) >> 4][(2 * i) & 15]);
                const float y = -(a1[(2 * i + 1) >> 4][(2 * i + 1) & 15] +
                                  e1 * a2[(2 * i + 1) >> 4][(2 * i + 1) & 15]);
                nd[i] = tc::pack_bf16(x, y);
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                *reinterpret_cast<uint4*>(ndbuf(c) + canon(32 * g + 8 * q4, r, C)) =
                    make_uint4(nd[4 * q4], nd[4 * q4 + 1], nd[4 * q4 + 2], nd[4 * q4 + 3]);
            tc::fence_async_smem();
        }
        tc::tc_fence_before();
        __syncthreads();  // (C)
        tc::tc_fence_after();
        if (prod2) {
            tc::mbar_arrive(&bar);  // step 4 has one chain: nothing to issue here
            phase ^= 1u;
        } else if (prod) {
            // step 4: Sbar^T += (-Dbar^T) W
            ok = tc::mbar_wait(&barW, (uint32_t)(m & 1), err) && ok;
            tc::mma_tile(tb, tND, tWmn, DVT, Dk, C, true);
            tc::mma_commit(&bar);
            ok = tc::mbar_wait(&bar, phase, err) && ok;
            phase ^= 1u;
            if (c > lo) load_w(c - 1);
            if (c > lo + 1) load_raw(c - 2);
        } else if (epi) {
            if (storer) {
                if (!maps) store_dbar(c);
                tc::bulk_commit();
            }
            if (c > lo) {  // vectors and the scaled Obar operands of chunk c - 1
                const uint8_t* raw = sm + L.raw + ((m + 1) & 1) * kRawBytes;
                ok = tc::mbar_wait(&barR[(m + 1) & 1], (uint32_t)(((m + 1) >> 1) & 1), err) && ok;
                vectors_from_raw<KC>(raw, reinterpret_cast<float*>(sm + L.vec) + ((m + 1) & 1) * 4 * C, Dk);
                if (!oz) {
                    ok = tc::mbar_wait(&barO[(m + 1) & 1], (uint32_t)(((m + 1) >> 1) & 1), err) && ok;
                    build_os<KC>(obuf(c - 1), sm + L.Os, sm + L.Oslo, raw, Dk);
                }
                tc::fence_async_smem();
            }
            ok = tc::mbar_wait(&bar, phase, err) && ok;
            phase ^= 1u;
            tc::tc_fence_after();
        }
        tc::tc_fence_before();
        __syncthreads();  // (A) of chunk c - 1
        tc::tc_fence_after();
    }
    // cotangent leaving the segment: dstate0 (bottom segment) or the map's columns
    float* sout = nullptr;
    int64_t ostr = Dv;
    if (maps) {
        ostr = seg_wd(Dk, Dv);
        sout = sg.maps + ((int64_t)t * d.B * d.Hv + bh) * Dk * ostr + n0;
    } else if (sg.sout) {
        sout = sg.sout + bh * Dk * Dv + n0;
    } else if (t == sg.nseg - 1) {
        sout = p.dstate0 + bh * Dk * Dv + n0;
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
    if (progress) {
        if (storer) tc::fence_async_global();
        __threadfence();
    }
    tc::tc_fence_before();
    __syncthreads();
    if (progress && storer) {  // the last (up to) two chunks
        __threadfence();
        atomicAdd(progress + (int64_t)bb * d.Hv + h, (unsigned int)(hi - lo < 2 ? hi - lo : 2));
    }
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

}  // namespace ta
}  // namespace gdn
