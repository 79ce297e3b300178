// gdn_kc_tc.cu -- chunked form of the recurrence with one decay per key channel
// (the vectorised gating the mlx-lm page lists as g.ndim == 4) for bf16 inputs.
//
// Within a chunk (steps t, s = 0 .. 63, key channel i), with l = 0 and beta = 0
// on masked and padded steps, Gamma_ti = sum_{u <= t} l_ui and E = exp(Gamma):
//   A_ts = beta_t sum_i kh_ti kh_si exp(Gamma_ti - Gamma_si)   (s < t)
//   P_ts = sum_i qh_ti kh_si exp(Gamma_ti - Gamma_si)          (s <= t)
//   T = (I + A)^-1,  W = T diag(beta) (kh o E),  U = T diag(beta) V,
//   Q_r = qh o E,  K_d = kh o exp(Gamma_63 - Gamma),  e_C = exp(Gamma_63)
// and, chunk after chunk, Delta = U - W S, O = Q_r S + P Delta,
// S <- diag(e_C) S + K_d^T Delta: the applied steps of the torch-to-nnef op
// contract with diag(g_t) in place of the scalar decay, unrolled over a chunk
// (the rows of S decay independently, so the scalar chunked form carries over
// with per-channel factors inside the key products).
//
// exp(Gamma_ti - Gamma_si) is never formed as exp(Gamma_ti) / exp(Gamma_si), which
// over- or underflows for strong decays.  Off the diagonal 16 x 16 blocks it is
// the product of exp(Gamma_ti - Gamma_bi) and exp(Gamma_bi - Gamma_si) through
// the last step b of the block of s, both in (0, 1]; on the diagonal blocks
// every term takes its own exponential.  Exponentials use the fast intrinsic
// (a few ulp; the arguments are never positive).
//
// This file: the chunk-local forward products (CUDA cores, fp32), then the
// per-chunk gradients (see the backward section below).  The scans are the KC
// variants of the tensor-core scans in gdn_scan_ta.cu / gdn_scan_ta.cuh.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"
#include "gdn_tri.cuh"

namespace gdn {

GDN_ERROR_WORD(kctc)

namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
using tri::LDT;

__device__ __forceinline__ void st_bf16x8(uint8_t* dst, const float* v) {
    uint4 u;
    u.x = tc::pack_bf16(v[0], v[1]);
    u.y = tc::pack_bf16(v[2], v[3]);
    u.z = tc::pack_bf16(v[4], v[5]);
    u.w = tc::pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = u;
}
__device__ __forceinline__ void ld_bf16x8(const void* src, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// ---- forward: chunk-local products ------------------------------------------

// Shared memory of the chunk kernel, byte offsets.  q, k and Gamma rows are fp32
// with rows of Dk + 4 floats (16-byte aligned, so four channels move as one
// float4; consecutive rows four banks apart).  Region q later holds T and the
// solve's scratch; region R the right factors kh_s exp(Gamma_b - Gamma_s) of
// the steps s < 48 channel-major ([Dk][52]: one pivot block's 8 or 16 factors
// of a channel are contiguous), then beta V.
constexpr int kRS = 52;
struct KfSmem {
    uint32_t q, k, G, R, A, P, vec, total;
};
__host__ __device__ inline KfSmem kf_plan(int Dk, int Dv) {
    const uint32_t LD = (uint32_t)Dk + 4;
    KfSmem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 127u) & ~127u;
        return r;
    };
    const uint32_t rows = C * LD * 4, mat = C * LDT * 4;
    const uint32_t rR = (uint32_t)Dk * kRS * 4, rV = C * ((uint32_t)Dv + 4) * 4;
    s.q = take(rows > 2 * mat ? rows : 2 * mat);
    s.k = take(rows);
    s.G = take(rows);
    s.R = take(rR > rV ? rR : rV);
    s.A = take(mat);
    s.P = take(mat);
    s.vec = take(4 * C * 4);
    s.total = o;
    return s;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float e) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, e);
}

// One 512-thread CTA per (chunk, value head, batch).  p.a = log_decay [B, T, Hv, Dk], p.b =
// beta [B, T, Hv] (bf16); rq, rk from prep.  Writes the panel images of Q_r, K_d
// (p.qimg, p.kimg, per value head), K_r = kh o E (p.krimg), P, T, W, the fp32
// rows of U, e_C (p.ecd) and the decayed Gram of the k rows (p.gram, for the
// beta cotangent).
constexpr int kChunkThreads = 512;
__global__ void __launch_bounds__(kChunkThreads, 1) kc_chunk_kernel(Dims d, Ptrs p) {
    extern __shared__ __align__(16) uint8_t ksm[];
    const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv, LD = Dk + 4, LV = Dv + 4;
    const int tid = threadIdx.x;
    const KfSmem L = kf_plan(Dk, Dv);
    float* qf = reinterpret_cast<float*>(ksm + L.q);
    float* kf = reinterpret_cast<float*>(ksm + L.k);
    float* Gf = reinterpret_cast<float*>(ksm + L.G);
    float* Rt = reinterpret_cast<float*>(ksm + L.R);
    float* A = reinterpret_cast<float*>(ksm + L.A);
    float* Pm = reinterpret_cast<float*>(ksm + L.P);
    float* bt = reinterpret_cast<float*>(ksm + L.vec);  // beta (0 off the applied steps)
    float* on = bt + C;                                 // 1 on applied steps
    float* rqs = on + C;                                // r_q / sqrt(Dk) (0 past T)
    float* rks = rqs + C;                               // r_k
    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const int64_t ci = bh * d.NC + c;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);
    const __nv_bfloat16* lg = static_cast<const __nv_bfloat16*>(p.a);
    const __nv_bfloat16* be = static_cast<const __nv_bfloat16*>(p.b);

    if (tid < C) {
        const bool in = tid < nvalid;
        const int64_t t = t0 + tid;
        const bool live = in && (p.mask == nullptr || p.mask[(int64_t)bb * d.T + t] != 0);
        bt[tid] = live ? __bfloat162float(be[((int64_t)bb * d.T + t) * d.Hv + h]) : 0.f;
        on[tid] = live ? 1.f : 0.f;
        const int64_t ri = ((int64_t)bb * d.Hk + j) * d.Tp + t;
        rqs[tid] = in ? p.rq[ri] * rsqrtf((float)Dk) : 0.f;
        rks[tid] = in ? p.rk[ri] : 0.f;
    }
    __syncthreads();
    // normalised q, k rows and the log-decays (zero off the applied steps)
    const int cpr = Dk / 8;
    for (int e = tid; e < C * cpr; e += kChunkThreads) {
        const int t = e / cpr, i0 = (e % cpr) * 8;
        float xq[8], xk[8], xl[8];
        if (t < nvalid) {
            const int64_t qi = (((int64_t)bb * d.T + t0 + t) * d.Hk + j) * Dk + i0;
            ld_bf16x8(q + qi, xq);
            ld_bf16x8(k + qi, xk);
            ld_bf16x8(lg + (((int64_t)bb * d.T + t0 + t) * d.Hv + h) * Dk + i0, xl);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) xq[u] = xk[u] = xl[u] = 0.f;
        }
        const float rq = rqs[t], rk = rks[t], o = on[t];
#pragma unroll
        for (int u = 0; u < 8; u += 4) {
            st4(qf + t * LD + i0 + u, xq[u] * rq, xq[u + 1] * rq, xq[u + 2] * rq, xq[u + 3] * rq);
            st4(kf + t * LD + i0 + u, xk[u] * rk, xk[u + 1] * rk, xk[u + 2] * rk, xk[u + 3] * rk);
            st4(Gf + t * LD + i0 + u, xl[u] * o, xl[u + 1] * o, xl[u + 2] * o, xl[u + 3] * o);
        }
    }
    __syncthreads();
    for (int i = tid; i < Dk; i += kChunkThreads) {  // Gamma: running sums down each key channel
        float g = 0.f;
        for (int t = 0; t < C; ++t) {
            g += Gf[t * LD + i];
            Gf[t * LD + i] = g;
        }
    }
    __syncthreads();

    // Q_r and K_d panel images (chunk e: row e % 64, channels 8 (e / 64) ..), e_C,
    // and the right factors kh_s exp(Gamma_b - Gamma_s) of the off-diagonal blocks
    uint8_t* qr_img = static_cast<uint8_t*>(p.qimg) + ci * C * Dk * 2;
    uint8_t* kd_img = static_cast<uint8_t*>(p.kimg) + ci * C * Dk * 2;
    uint8_t* kr_img = static_cast<uint8_t*>(p.krimg) + ci * C * Dk * 2;
    for (int e = tid; e < C * cpr; e += kChunkThreads) {
        const int t = e % C, i0 = (e / C) * 8;
        float a[8], b[8], kr[8];
#pragma unroll
        for (int u = 0; u < 8; u += 4) {
            const float4 g = ld4(Gf + t * LD + i0 + u), gl = ld4(Gf + (C - 1) * LD + i0 + u);
            const float4 qq = ld4(qf + t * LD + i0 + u), kk = ld4(kf + t * LD + i0 + u);
            a[u] = qq.x * __expf(g.x);
            a[u + 1] = qq.y * __expf(g.y);
            a[u + 2] = qq.z * __expf(g.z);
            a[u + 3] = qq.w * __expf(g.w);
            b[u] = kk.x * __expf(gl.x - g.x);
            b[u + 1] = kk.y * __expf(gl.y - g.y);
            b[u + 2] = kk.z * __expf(gl.z - g.z);
            b[u + 3] = kk.w * __expf(gl.w - g.w);
            kr[u] = kk.x * __expf(g.x);
            kr[u + 1] = kk.y * __expf(g.y);
            kr[u + 2] = kk.z * __expf(g.z);
            kr[u + 3] = kk.w * __expf(g.w);
        }
        st_bf16x8(qr_img + 16 * e, a);
        st_bf16x8(kd_img + 16 * e, b);
        st_bf16x8(kr_img + 16 * e, kr);
    }
    for (int i = tid; i < Dk; i += kChunkThreads) p.ecd[ci * Dk + i] = __expf(Gf[(C - 1) * LD + i]);
    for (int e = tid; e < 48 * Dk; e += kChunkThreads) {
        const int s = e / Dk, i = e % Dk, b = s | 15;
        Rt[i * kRS + s] = kf[s * LD + i] * __expf(Gf[b * LD + i] - Gf[s * LD + i]);
    }
    __syncthreads();

    // A and P off the diagonal blocks (warps 0-5: one row t and eight columns s
    // of a pivot block J per thread, four channels per step) and on the
    // diagonal blocks (warps 6-13), side by side
    if (tid < 192) {
        const int half = tid / 96, r = tid % 96;
        const int J = r < 48 ? 0 : r < 80 ? 1 : 2;
        const int t = J == 0 ? 16 + r : J == 1 ? 32 + (r - 48) : 48 + (r - 80);
        const int b = 16 * J + 15, s0 = 16 * J + 8 * half;
        float a8[8], p8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) a8[x] = p8[x] = 0.f;
        for (int i = 0; i < Dk; i += 4) {
            const float4 kt = ld4(kf + t * LD + i), qt = ld4(qf + t * LD + i);
            const float4 gt = ld4(Gf + t * LD + i), gb = ld4(Gf + b * LD + i);
            const float u[4] = {__expf(gt.x - gb.x), __expf(gt.y - gb.y), __expf(gt.z - gb.z), __expf(gt.w - gb.w)};
            const float ka[4] = {kt.x * u[0], kt.y * u[1], kt.z * u[2], kt.w * u[3]};
            const float qa[4] = {qt.x * u[0], qt.y * u[1], qt.z * u[2], qt.w * u[3]};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float4 r0 = ld4(Rt + (i + x) * kRS + s0), r1 = ld4(Rt + (i + x) * kRS + s0 + 4);
                const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                for (int y = 0; y < 8; ++y) {
                    a8[y] = fmaf(ka[x], rr[y], a8[y]);
                    p8[y] = fmaf(qa[x], rr[y], p8[y]);
                }
            }
        }
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            A[t * LDT + s0 + x] = bt[t] * a8[x];
            Pm[t * LDT + s0 + x] = p8[x];
        }
        float* gr = p.gram + (ci * C + t) * C + s0;
        reinterpret_cast<float4*>(gr)[0] = make_float4(a8[0], a8[1], a8[2], a8[3]);
        reinterpret_cast<float4*>(gr)[1] = make_float4(a8[4], a8[5], a8[6], a8[7]);
    }
    // the diagonal blocks: thread (row t, channel quarter qq) forms row t against
    // every s = 16 I .. t of its block over its quarter of the channels, each term
    // with its own exponential; the quarters' sums meet by shuffles
    else if (tid < 448) {
        const int t = (tid - 192) >> 2, qq = tid & 3, I = t >> 4, n = t - 16 * I;  // s = 16 I + 0 .. n
        const int qw = Dk / 4;
        float ad[16], pd[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) ad[x] = pd[x] = 0.f;
        for (int i = qq * qw; i < (qq + 1) * qw; i += 4) {
            const float4 kt = ld4(kf + t * LD + i), qt = ld4(qf + t * LD + i), gt = ld4(Gf + t * LD + i);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                if (x <= n) {
                    const int sr = 16 * I + x;
                    const float4 ks = ld4(kf + sr * LD + i), gs = ld4(Gf + sr * LD + i);
                    const float e0 = ks.x * __expf(gt.x - gs.x), e1 = ks.y * __expf(gt.y - gs.y);
                    const float e2 = ks.z * __expf(gt.z - gs.z), e3 = ks.w * __expf(gt.w - gs.w);
                    ad[x] = fmaf(kt.x, e0, fmaf(kt.y, e1, fmaf(kt.z, e2, fmaf(kt.w, e3, ad[x]))));
                    pd[x] = fmaf(qt.x, e0, fmaf(qt.y, e1, fmaf(qt.z, e2, fmaf(qt.w, e3, pd[x]))));
                }
            }
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            ad[x] += __shfl_xor_sync(0xffffffffu, ad[x], 1);
            ad[x] += __shfl_xor_sync(0xffffffffu, ad[x], 2);
            pd[x] += __shfl_xor_sync(0xffffffffu, pd[x], 1);
            pd[x] += __shfl_xor_sync(0xffffffffu, pd[x], 2);
        }
        if (qq == 0) {
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                if (x <= n) {
                    const int sr = 16 * I + x;
                    A[t * LDT + sr] = x < n ? bt[t] * ad[x] : 0.f;
                    Pm[t * LDT + sr] = pd[x];
                    if (x < n) p.gram[(ci * C + t) * C + sr] = ad[x];
                }
            }
        }
    }
    __syncthreads();

    // P image (zero above the diagonal), then T = (I + A)^-1 into region q
    uint8_t* Pimg = static_cast<uint8_t*>(p.P) + ci * C * C * 2;
    for (int e = tid; e < C * (C / 8); e += kChunkThreads) {
        const int t = e % C, s0 = (e / C) * 8;
        float v8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v8[u] = s0 + u <= t ? Pm[t * LDT + s0 + u] : 0.f;
        st_bf16x8(Pimg + 16 * e, v8);
    }
    float* Tm = qf;
    float* X = qf + C * LDT;
    tri::tri_inverse64(A, Tm, X);  // ends synchronised
    uint8_t* Timg = reinterpret_cast<uint8_t*>(p.Tinv) + ci * C * C * 2;
    for (int e = tid; e < C * (C / 8); e += kChunkThreads) {
        const int t = e % C, s0 = (e / C) * 8;
        float v8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v8[u] = (s0 >> 4) <= (t >> 4) ? Tm[t * LDT + s0 + u] : 0.f;
        st_bf16x8(Timg + 16 * e, v8);
    }
    // beta (kh o E) in place of kh, beta V in region R
    for (int e = tid; e < C * Dk; e += kChunkThreads) {
        const int s = e / Dk, i = e % Dk;
        kf[s * LD + i] *= bt[s] * __expf(Gf[s * LD + i]);
    }
    float* Vb = Rt;
    for (int e = tid; e < C * (Dv / 8); e += kChunkThreads) {
        const int t = e / (Dv / 8), c0 = (e % (Dv / 8)) * 8;
        float x[8];
        if (t < nvalid) {
            ld_bf16x8(v + (((int64_t)bb * d.T + t0 + t) * d.Hv + h) * Dv + c0, x);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = 0.f;
        }
        const float bs = bt[t];
        st4(Vb + t * LV + c0, bs * x[0], bs * x[1], bs * x[2], bs * x[3]);
        st4(Vb + t * LV + c0 + 4, bs * x[4], bs * x[5], bs * x[6], bs * x[7]);
    }
    __syncthreads();

    // W = T (beta kh o E) and U = T (beta V): 4 x 4 tiles, T read only on and
    // below the diagonal (a row quad never reaches past its own 16-row block)
    uint8_t* Wimg = static_cast<uint8_t*>(p.W) + ci * C * Dk * 2;
    float* U = p.U + (bh * d.Tp + t0) * Dv;
    const int ncq = (Dk + Dv) / 4;
    for (int e = tid; e < 16 * ncq; e += kChunkThreads) {
        const int tq = 4 * (e / ncq), c0 = 4 * (e % ncq);
        const bool isW = c0 < Dk;
        const float* Bm = isW ? kf + c0 : Vb + (c0 - Dk);
        const int ldb = isW ? LD : LV;
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[r][x] = 0.f;
        for (int s = 0; s <= tq + 3; ++s) {
            float tv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) tv[r] = Tm[(tq + r) * LDT + s];
            const float4 b4 = ld4(Bm + s * ldb);
            const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) acc[r][x] = fmaf(tv[r], bv[x], acc[r][x]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (isW) {
                uint2 w;
                w.x = tc::pack_bf16(acc[r][0], acc[r][1]);
                w.y = tc::pack_bf16(acc[r][2], acc[r][3]);
                *reinterpret_cast<uint2*>(Wimg + tc::panel_off((uint32_t)(c0 & ~7), (uint32_t)(tq + r), C) +
                                          (c0 & 7) * 2) = w;
            } else {
                *reinterpret_cast<float4*>(U + (int64_t)(tq + r) * Dv + (c0 - Dk)) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            }
        }
    }
}

// ---- backward: per-chunk gradients ------------------------------------------
//
// Per chunk, from the chunk-start state S (checkpoint image), the cotangent
// Sbar' of the chunk-end state and -Dbar (reverse scan, Dbar the whole
// cotangent of Delta), Delta (hi + lo images) and Obar:
//   Kbar_d = Delta Sbar'^T,  Qbar_r = Obar S^T,  Wbar = -Dbar S^T,
//   ebar_i = <Sbar'_i, S_i>,  Pbar = Obar Delta^T (s <= t),  M1 = Dbar V^T,
//   dv = diag(beta) T^T Dbar,  M2 = Wbar K_r^T (K_r = kh o E),  Tbar = (M1 + M2) diag(beta),
//   Abar = -T^T Tbar T^T (s < t),  Gbar = diag(beta) Abar,  Kbar_r = diag(beta) T^T Wbar,
//   betabar_t = sum_u T_ut (M1 + M2)_ut + sum_{s < t} Abar_ts G_ts,
// then, per key channel with e_ts = exp(Gamma_t - Gamma_s), the sums through
// the decayed products ("left": over the columns s of row t, "right": over the
// rows t of column s)
//   LG_t = sum_s Gbar_ts kh_s e_ts,  RG_s = sum_t Gbar_ts kh_t e_ts,
//   LP_t = sum_s Pbar_ts kh_s e_ts,  RP_s = sum_t Pbar_ts qh_t e_ts,
// and the cotangents of the normalised rows and of Gamma:
//   qhbar = Qbar_r o E + LP,
//   khbar = Kbar_r o E + Kbar_d o exp(Gamma_63 - Gamma) + LG + RG + RP,
//   Gammabar = Qbar_r o Q_r + Kbar_r o (kh o E) - Kbar_d o K_d + qh o LP + kh o (LG - RG - RP),
//   Gammabar_63 += sum_t Kbar_d o K_d + ebar o e_C,
//   lbar_t = sum_{u >= t} Gammabar_u  (applied steps; 0 elsewhere).
// Kernel 1 (tensor cores) forms the products whose sums run over the Dv value
// columns, and M2 and Kbar_r (Wbar staged as a bf16 operand); kernel 2 (CUDA
// cores, fp32) Abar, Gbar and the beta cotangent per chunk; kernel 3 (CUDA
// cores, fp32) the decayed-Gram sums, 32 key channels at a time.

struct KpSmem {
    uint32_t O, V, D, Dlo, ND, Tt, S, Sp, Kr, Wt, total;
};
__host__ __device__ inline KpSmem kp_plan(int Dv) {
    KpSmem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    const uint32_t tv = (uint32_t)(C * Dv * 2);
    s.O = take(tv);
    s.V = take(tv);
    s.D = take(tv);
    s.Dlo = take(tv);
    s.ND = take(tv);
    s.Tt = take(C * C * 2);
    s.S = take(tv);   // one 64-channel block of the S^T image (Dv rows)
    s.Sp = take(tv);  // and of the Sbar'^T image
    s.Kr = take(C * 64 * 2);  // the block's 64 channels of the K_r image (panel, 64 rows)
    s.Wt = take(C * 64 * 2);  // Wbar of the block as a bf16 operand (canonical, x = channel)
    s.total = o;
    return s;
}

// canonical operand tile of a 64-column image (8-row groups ncols * 16 bytes apart)
__device__ __forceinline__ tc::Tile canon_tile(uint8_t* smem, uint32_t off, int ncols, bool k_major) {
    tc::Tile t;
    t.base = tc::smem_u32(smem + off);
    t.xs = 128;
    t.ys = (uint32_t)ncols * 16u;
    t.k_major = k_major;
    return t;
}

// An M = 64 accumulator of ncols columns at TMEM column col (row r in lane
// 32 (r / 16) + r % 16), walked by eight warps: warp w takes rows 16 (w % 4) ..
// + 15 and half w / 4 of the columns; lane l < 16 gets columns c .. c + 7 of
// row 16 (w % 4) + l, lane l + 16 columns c + 8 .. c + 15 (by shuffles).
// f(row, first column, 8 values)
template <typename F>
__device__ __forceinline__ void acc_walk(uint32_t tb, uint32_t col, int ncols, F&& f) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int sp = w & 3, g = w >> 2, hl = l >> 4;
    const int half = ncols / 2;
    for (int c = g * half; c < (g + 1) * half; c += 16) {
        float v[16];
        tc::tmem_ld16(tc::tmem_addr(tb, 32 * sp, col + c), v);
        tc::tmem_wait_ld();
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float up = __shfl_sync(0xffffffffu, v[8 + i], l & 15);
            x[i] = hl ? up : v[i];
        }
        f(16 * sp + (l & 15), c + 8 * hl, x);
    }
}

__device__ __forceinline__ void st_f32x8(float* dst, const float* x) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// beta of step t0 + t (0 off the applied steps) and the applied flag
__device__ __forceinline__ void step_gate(const Dims& d, const Ptrs& p, int bb, int h, int64_t t0,
                                          int nvalid, int t, float* bt, float* on) {
    const bool live = t < nvalid && (p.mask == nullptr || p.mask[(int64_t)bb * d.T + t0 + t] != 0);
    *bt = live ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.b)[((int64_t)bb * d.T + t0 + t) * d.Hv + h])
               : 0.f;
    *on = live ? 1.f : 0.f;
}

// Kernel 1: one CTA per (chunk, value head, batch), 256 threads, all 512 TMEM
// columns.  Products: Pbar (cols 0..63), -M1 (64..127), -T^T Dbar (128..) from
// dO, v (TMA tiles), Delta, -Dbar and T images; then per 64-channel block of S,
// Sbar' and K_r: Kbar_d (0..63), Qbar_r (64..127), Wbar (128..191) and ebar;
// Wbar as a bf16 tile, then Kbar_r = T^T Wbar (192..255, times beta on the way
// out) and M2 += Wbar K_r^T (256..319); M = M1 + M2 at the end.
__global__ void __launch_bounds__(kThreads, 1)
    kc_bwd_prod_kernel(Dims d, Ptrs p, const __grid_constant__ Tmaps tm) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar, barL, barS;
    __shared__ uint32_t tmem_sh;
    __shared__ float bt[C];
    const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int tid = threadIdx.x, warp = tid >> 5;
    const KpSmem L = kp_plan(Dv);
    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const int64_t ci = bh * d.NC + c;
    const uint32_t tv = (uint32_t)(C * Dv * 2), blk = (uint32_t)(64 * Dv * 2);
    const int nblk = Dk / 64;
    const uint8_t* ckimg = reinterpret_cast<const uint8_t*>(p.ckpt) + ci * (int64_t)Dk * Dv * 2;
    const uint8_t* dsimg = reinterpret_cast<const uint8_t*>(p.dSck) + ci * (int64_t)Dk * Dv * 2;
    if (tid < C) {
        float o;
        step_gate(d, p, bb, h, t0, nvalid, tid, &bt[tid], &o);
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_sh, 512);
        tc::tmem_relinquish();
    }
    const uint8_t* krimg = static_cast<const uint8_t*>(p.krimg) + ci * (int64_t)C * Dk * 2;
    const uint32_t kblk = (uint32_t)(C * 64 * 2);
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_init(&barL, 1);
        tc::mbar_init(&barS, 1);
        tc::fence_mbar_init();
        tc::mbar_arrive_expect_tx(&barL, 5 * tv + C * C * 2);
        tc::tma_load_5d(sm + L.O, &tm.dOf, 0, c * C, 0, h, bb, &barL);
        tc::tma_load_5d(sm + L.V, &tm.v, 0, c * C, 0, h, bb, &barL);
        const uint8_t* dl = reinterpret_cast<const uint8_t*>(p.Delta) + ci * (int64_t)C * Dv * 4;
        tc::bulk_g2s(sm + L.D, dl, tv, &barL);
        tc::bulk_g2s(sm + L.Dlo, dl + tv, tv, &barL);
        tc::bulk_g2s(sm + L.ND, reinterpret_cast<const uint8_t*>(p.Dbar) + ci * (int64_t)tv, tv, &barL);
        tc::bulk_g2s(sm + L.Tt, reinterpret_cast<const uint8_t*>(p.Tinv) + ci * C * C * 2, C * C * 2, &barL);
        tc::mbar_arrive_expect_tx(&barS, 2 * blk + kblk);
        tc::bulk_g2s(sm + L.S, ckimg, blk, &barS);
        tc::bulk_g2s(sm + L.Sp, dsimg, blk, &barS);
        tc::bulk_g2s(sm + L.Kr, krimg, kblk, &barS);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tb = tmem_sh;
    bool ok = tc::mbar_wait(&barL, 0, &g_err_kctc);
    // dO, v: TMA panel tiles (K-major over the value columns); Delta, -Dbar:
    // images of the transposes (x = step); T: panel image (x = column)
    const tc::Tile tO = tc::panel_tile(sm + L.O, C, true), tV = tc::panel_tile(sm + L.V, C, true);
    const tc::Tile tDmn = canon_tile(sm, L.D, C, false), tDlomn = canon_tile(sm, L.Dlo, C, false);
    const tc::Tile tNB = canon_tile(sm, L.ND, C, true), tNBmn = canon_tile(sm, L.ND, C, false);
    const tc::Tile tTmn = tc::panel_tile(sm + L.Tt, C, false);
    const tc::Tile tS = tc::panel_tile(sm + L.S, Dv, false), tSp = tc::panel_tile(sm + L.Sp, Dv, false);
    const tc::Tile tKr = tc::panel_tile(sm + L.Kr, C, true);  // B = K_r^T: x = channel = K
    const tc::Tile tWk = canon_tile(sm, L.Wt, 64, true);       // A = Wbar: x = channel = K
    const tc::Tile tWmn = canon_tile(sm, L.Wt, 64, false);     // B = Wbar: x = channel = N
    if (tid == 0) {
        tc::mma_tile(tb + 0, tO, tDmn, C, C, Dv, false);     // Obar Delta^T (hi + lo)
        tc::mma_tile(tb + 0, tO, tDlomn, C, C, Dv, true);
        tc::mma_tile(tb + 64, tNBmn, tV, C, C, Dv, false);   // -Dbar V^T
        tc::mma_tile(tb + 128, tTmn, tNB, C, Dv, C, false);  // T^T (-Dbar)
        tc::mma_commit(&bar);
    }
    uint32_t phase = 0;
    ok = tc::mbar_wait(&bar, phase, &g_err_kctc) && ok;
    phase ^= 1u;
    tc::tc_fence_after();
    if (ok) {
        float* Pb = p.pbm + ci * C * C;
        float* M1 = p.m1 + ci * C * C;
        __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(p.dv);
        acc_walk(tb, 0, C, [&](int r, int c0, const float* x) {
            float m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = c0 + i <= r ? x[i] : 0.f;
            st_f32x8(Pb + r * C + c0, m);
        });
        acc_walk(tb, 64, C, [&](int r, int c0, const float* x) {
            float m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = -x[i];
            st_f32x8(M1 + r * C + c0, m);
        });
        acc_walk(tb, 128, Dv, [&](int r, int c0, const float* x) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = -bt[r] * x[i];
            if (r < nvalid)
                st_bf16x8(reinterpret_cast<uint8_t*>(dv + (((int64_t)bb * d.T + t0 + r) * d.Hv + h) * Dv + c0), y);
        });
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const int64_t rowbase = bh * d.Tp + t0;
    for (int b = 0; b < nblk; ++b) {
        ok = tc::mbar_wait(&barS, (uint32_t)(b & 1), &g_err_kctc) && ok;
        if (tid == 0) {
            tc::mma_tile(tb + 0, tDmn, tSp, C, 64, Dv, false);  // Delta Sbar'^T
            tc::mma_tile(tb + 0, tDlomn, tSp, C, 64, Dv, true);
            tc::mma_tile(tb + 64, tO, tS, C, 64, Dv, false);     // Obar S^T
            tc::mma_tile(tb + 128, tNBmn, tS, C, 64, Dv, false); // -Dbar S^T
            tc::mma_commit(&bar);
        }
        {  // <Sbar'_i, S_i>: four threads per channel, a quarter of the value rows each
            const int x = tid >> 2, part = tid & 3;
            const uint8_t* s0 = sm + L.S + (x >> 3) * Dv * 16 + (x & 7) * 2;
            const uint8_t* s1 = sm + L.Sp + (x >> 3) * Dv * 16 + (x & 7) * 2;
            float acc = 0.f;
            for (int v = part * (Dv / 4); v < (part + 1) * (Dv / 4); ++v)
                acc = fmaf(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(s0 + v * 16)),
                           __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(s1 + v * 16)), acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0) p.ecb[ci * Dk + 64 * b + x] = acc;
        }
        ok = tc::mbar_wait(&bar, phase, &g_err_kctc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        const int64_t cb0 = 64 * b;
        if (ok) {  // Wbar as a bf16 operand tile, then Kbar_d and Qbar_r out
            acc_walk(tb, 128, 64, [&](int r, int c0, const float* x) {
                st_bf16x8(sm + L.Wt + (c0 >> 3) * 128 + (r >> 3) * 1024 + (r & 7) * 16, x);
            });
        }
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();  // Wbar tile written
        tc::tc_fence_after();
        if (tid == 0) {
            tc::mma_tile(tb + 192, tTmn, tWmn, C, 64, C, false);  // T^T Wbar
            tc::mma_tile(tb + 256, tWk, tKr, C, C, 64, b > 0);    // M2 += Wbar K_r^T
            tc::mma_commit(&bar);
        }
        if (ok) {
            acc_walk(tb, 0, 64, [&](int r, int c0, const float* x) { st_f32x8(p.kdb + (rowbase + r) * Dk + cb0 + c0, x); });
            acc_walk(tb, 64, 64, [&](int r, int c0, const float* x) { st_f32x8(p.qrb + (rowbase + r) * Dk + cb0 + c0, x); });
        }
        ok = tc::mbar_wait(&bar, phase, &g_err_kctc) && ok;
        phase ^= 1u;
        tc::tc_fence_after();
        if (ok) {
            acc_walk(tb, 192, 64, [&](int r, int c0, const float* x) {
                float y[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = bt[r] * x[i];
                st_f32x8(p.wb + (rowbase + r) * Dk + cb0 + c0, y);
            });
        }
        tc::tc_fence_before();
        __syncthreads();  // accumulators read; S, Sbar', K_r and Wbar tiles read
        tc::tc_fence_after();
        if (tid == 0 && b + 1 < nblk) {
            tc::mbar_arrive_expect_tx(&barS, 2 * blk + kblk);
            tc::bulk_g2s(sm + L.S, ckimg + (int64_t)(b + 1) * blk, blk, &barS);
            tc::bulk_g2s(sm + L.Sp, dsimg + (int64_t)(b + 1) * blk, blk, &barS);
            tc::bulk_g2s(sm + L.Kr, krimg + (int64_t)(b + 1) * kblk, kblk, &barS);
        }
    }
    if (ok) {  // M = M1 + M2 (M1 written by this CTA before the block loop)
        float* M1 = p.m1 + ci * C * C;
        acc_walk(tb, 256, C, [&](int r, int c0, const float* x) {
            float m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = M1[r * C + c0 + i] + x[i];
            st_f32x8(M1 + r * C + c0, m);
        });
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

constexpr int CB = 32;       // key channels per block of kernels 2 and 3
constexpr int LB = CB + 1;   // row stride of their per-block arrays (odd: conflict-free columns)
constexpr int kBlkMat = C * LDT * 4, kBlkArr = C * LB * 4;

// rows of the pivot factors exp(Gamma_t - Gamma_b), b = 16 J + 15, t > b: J-major
__device__ __forceinline__ int frow(int J, int t) { return J == 0 ? t - 16 : J == 1 ? 48 + t - 32 : 80 + t - 48; }

// normalised k (and, WITH_Q, q) rows and Gamma of key channels cb0 .. cb0 + 31
// (256 threads: thread = (row, 8 channels)); Gamma by a two-level running sum,
// warp w over rows 8 w .. 8 w + 7 of channel `lane`, then the offsets of the
// pieces above (part: [8][CB] scratch).  Ends synchronised.
template <bool WITH_Q>
__device__ __forceinline__ void load_block(const Dims& d, const Ptrs& p, int bb, int h, int j, int64_t t0,
                                           int nvalid, int cb0, const float* on, const float* rqs,
                                           const float* rks, float* qb, float* kb, float* Gm, float* part) {
    const int tid = threadIdx.x, t = tid >> 2, i0 = (tid & 3) * 8;
    const int Dk = (int)d.Dk;
    float xq[8], xk[8], xl[8];
    if (t < nvalid) {
        const int64_t qi = (((int64_t)bb * d.T + t0 + t) * d.Hk + j) * Dk + cb0 + i0;
        if (WITH_Q) ld_bf16x8(static_cast<const __nv_bfloat16*>(p.q) + qi, xq);
        ld_bf16x8(static_cast<const __nv_bfloat16*>(p.k) + qi, xk);
        ld_bf16x8(static_cast<const __nv_bfloat16*>(p.a) + (((int64_t)bb * d.T + t0 + t) * d.Hv + h) * Dk + cb0 + i0,
                  xl);
    } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) xq[u] = xk[u] = xl[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        if (WITH_Q) qb[t * LB + i0 + u] = xq[u] * rqs[t];
        kb[t * LB + i0 + u] = xk[u] * rks[t];
        Gm[t * LB + i0 + u] = on[t] != 0.f ? xl[u] : 0.f;
    }
    __syncthreads();
    const int w = tid >> 5, i = tid & 31;
    float sacc = 0.f;
    for (int r = 8 * w; r < 8 * w + 8; ++r) {
        sacc += Gm[r * LB + i];
        Gm[r * LB + i] = sacc;
    }
    part[w * CB + i] = sacc;
    __syncthreads();
    float off = 0.f;
    for (int w2 = 0; w2 < w; ++w2) off += part[w2 * CB + i];
    for (int r = 8 * w; r < 8 * w + 8; ++r) Gm[r * LB + i] += off;
    __syncthreads();
}

// per-step vectors of a chunk: beta, applied flag, r_q / sqrt(Dk), r_k
__device__ __forceinline__ void chunk_vectors(const Dims& d, const Ptrs& p, int bb, int h, int j, int64_t t0,
                                              int nvalid, float* bt, float* on, float* rqs, float* rks) {
    const int tid = threadIdx.x;
    if (tid < C) {
        step_gate(d, p, bb, h, t0, nvalid, tid, &bt[tid], &on[tid]);
        const int64_t ri = ((int64_t)bb * d.Hk + j) * d.Tp + t0 + tid;
        rqs[tid] = tid < nvalid ? p.rq[ri] * rsqrtf((float)d.Dk) : 0.f;
        rks[tid] = tid < nvalid ? p.rk[ri] : 0.f;
    }
}

// Kernel 2: one CTA per (chunk, value head, batch), 256 threads, CUDA cores:
// betabar (p.db) and Gbar (into p.m1, over M) from T, M = M1 + M2 and G.
__global__ void __launch_bounds__(kThreads, 3) kc_bwd_gate_kernel(Dims d, Ptrs p) {
    extern __shared__ __align__(16) uint8_t lsm[];
    const int c = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
    const int tid = threadIdx.x;
    float* Tm = reinterpret_cast<float*>(lsm);
    float* Mm = Tm + C * LDT;
    float* Xm = Mm + C * LDT;
    float* bt = Xm + C * LDT;
    float* on = bt + C;
    float* bbar = on + C;
    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const int64_t ci = bh * d.NC + c;

    if (tid < C) step_gate(d, p, bb, h, t0, nvalid, tid, &bt[tid], &on[tid]);
    {  // T (from its bf16 panel image) and M
        const uint8_t* Timg = reinterpret_cast<const uint8_t*>(p.Tinv) + ci * C * C * 2;
        for (int e = tid; e < C * (C / 8); e += kThreads) {
            float x[8];
            ld_bf16x8(Timg + 16 * e, x);
            const int t = e % C, s0 = (e / C) * 8;
#pragma unroll
            for (int u = 0; u < 8; ++u) Tm[t * LDT + s0 + u] = x[u];
        }
        const float* mg = p.m1 + ci * C * C;
        for (int e = tid; e < C * C / 4; e += kThreads) {
            const int t = e / (C / 4), s0 = (e % (C / 4)) * 4;
            *reinterpret_cast<float4*>(Mm + t * LDT + s0) = reinterpret_cast<const float4*>(mg)[e];
        }
    }
    __syncthreads();

    // betabar (T o M column sums), Tbar = M diag(beta), X = Tbar T^T, Abar = -T^T X
    if (tid < C) {
        float sacc = 0.f;
        for (int u = tid; u < C; ++u) sacc = fmaf(Tm[u * LDT + tid], Mm[u * LDT + tid], sacc);
        bbar[tid] = sacc;
    }
    __syncthreads();
    for (int e = tid; e < C * C; e += kThreads) {
        const int t = e / C, s = e % C;
        Mm[t * LDT + s] *= bt[s];
    }
    __syncthreads();
    {
        const int tq = 4 * (tid >> 4), uq = 4 * (tid & 15);
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[r][x] = 0.f;
        for (int s = 0; s <= uq + 3; ++s) {
            float a[4], b[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) a[r] = Mm[(tq + r) * LDT + s];
#pragma unroll
            for (int x = 0; x < 4; ++x) b[x] = Tm[(uq + x) * LDT + s];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) acc[r][x] = fmaf(a[r], b[x], acc[r][x]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) Xm[(tq + r) * LDT + uq + x] = acc[r][x];
    }
    __syncthreads();
    {
        const int tq = 4 * (tid >> 4), sq = 4 * (tid & 15);
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[r][x] = 0.f;
        for (int u = tq; u < C; ++u) {
            float a[4], b[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) a[r] = Tm[u * LDT + tq + r];
#pragma unroll
            for (int x = 0; x < 4; ++x) b[x] = Xm[u * LDT + sq + x];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) acc[r][x] = fmaf(a[r], b[x], acc[r][x]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) Mm[(tq + r) * LDT + sq + x] = sq + x < tq + r ? -acc[r][x] : 0.f;
    }
    __syncthreads();
    {  // the forward's decayed Gram G (into X)
        const float* gg = p.gram + ci * C * C;
        for (int e = tid; e < C * C; e += kThreads) {
            const int t = e / C, s = e % C;
            Xm[t * LDT + s] = s < t ? gg[e] : 0.f;
        }
    }
    __syncthreads();
    if (tid < C) {  // betabar += sum_s Abar G
        float sacc = bbar[tid];
        for (int s = 0; s < tid; ++s) sacc = fmaf(Mm[tid * LDT + s], Xm[tid * LDT + s], sacc);
        if (tid < nvalid)
            static_cast<__nv_bfloat16*>(p.db)[((int64_t)bb * d.T + t0 + tid) * d.Hv + h] =
                __float2bfloat16_rn(on[tid] != 0.f ? sacc : 0.f);
    }
    {  // Gbar = diag(beta) Abar over M1's place
        float* gb = p.m1 + ci * C * C;
        for (int e = tid; e < C * C; e += kThreads) {
            const int t = e / C, s = e % C;
            gb[e] = bt[t] * Mm[t * LDT + s];
        }
    }
}

// Kernel 3: one CTA per (chunk, 32-channel block, value head, batch), 256
// threads, CUDA cores, two CTAs per SM.  Thread (warp w, lane i) takes channel
// i of the row quads w and w + 8: the four rows share every load of a column
// value, and the rows of Gbar / Pbar come as 16-byte loads.
__global__ void __launch_bounds__(kThreads, 2) kc_bwd_chan_kernel(Dims d, Ptrs p) {
    extern __shared__ __align__(16) uint8_t lsm[];
    const int nblk = (int)d.Dk / CB;
    const int c = blockIdx.x / nblk, cb0 = (blockIdx.x % nblk) * CB;
    const int h = blockIdx.y, bb = blockIdx.z;
    const int j = h / (int)d.G;
    const int Dk = (int)d.Dk;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* Pb = reinterpret_cast<float*>(lsm);
    float* Gg = Pb + C * LDT;
    float* qb = Gg + C * LDT;
    float* kb = qb + C * LB;
    float* Gm = kb + C * LB;
    float* Gb = Gm + C * LB;
    float* Fm = Gb + C * LB;   // [96][LB]
    float* Rm = Fm + 96 * LB;  // [48][LB]
    float* part = Rm + 48 * LB;  // [8][CB]
    float* bt = part + 8 * CB;
    float* on = bt + C;
    float* rqs = on + C;
    float* rks = rqs + C;
    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t bh = (int64_t)bb * d.Hv + h;
    const int64_t ci = bh * d.NC + c;
    const int64_t rowbase = bh * d.Tp + t0;

    chunk_vectors(d, p, bb, h, j, t0, nvalid, bt, on, rqs, rks);
    {
        const float* pg = p.pbm + ci * C * C;
        const float* gg = p.m1 + ci * C * C;
        for (int e = tid; e < C * C / 4; e += kThreads) {
            const int t = e / (C / 4), s0 = (e % (C / 4)) * 4;
            *reinterpret_cast<float4*>(Pb + t * LDT + s0) = reinterpret_cast<const float4*>(pg)[e];
            *reinterpret_cast<float4*>(Gg + t * LDT + s0) = reinterpret_cast<const float4*>(gg)[e];
        }
    }
    __syncthreads();
    load_block<true>(d, p, bb, h, j, t0, nvalid, cb0, on, rqs, rks, qb, kb, Gm, part);
    for (int e = tid; e < 96 * CB; e += kThreads) {
        const int row = e / CB, i = e % CB;
        const int J = row < 48 ? 0 : row < 80 ? 1 : 2;
        const int t = J == 0 ? 16 + row : J == 1 ? 32 + (row - 48) : 48 + (row - 80);
        Fm[row * LB + i] = __expf(Gm[t * LB + i] - Gm[(16 * J + 15) * LB + i]);
    }
    for (int e = tid; e < 48 * CB; e += kThreads) {
        const int s = e / CB, i = e % CB, b = s | 15;
        Rm[s * LB + i] = kb[s * LB + i] * __expf(Gm[b * LB + i] - Gm[s * LB + i]);
    }
    __syncthreads();

    const int i = lane;
    float colK = 0.f;
    for (int it = 0; it < 2; ++it) {
        const int g = warp + 8 * it, r0 = 4 * g, I = g >> 2;
        float gr[4], qrb[4], kdb[4], krb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int64_t gi = (rowbase + r0 + a) * Dk + cb0 + i;
            qrb[a] = p.qrb[gi];
            kdb[a] = p.kdb[gi];
            krb[a] = p.wb[gi];
            gr[a] = Gm[(r0 + a) * LB + i];
        }
        float LG[4] = {0.f, 0.f, 0.f, 0.f}, LP[4] = {0.f, 0.f, 0.f, 0.f};
        float RG[4] = {0.f, 0.f, 0.f, 0.f}, RP[4] = {0.f, 0.f, 0.f, 0.f};
        // left sums, off the diagonal block: per pivot block J < I
        for (int J = 0; J < I; ++J) {
            float sG[4] = {0.f, 0.f, 0.f, 0.f}, sP[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 16 * J; s < 16 * J + 16; s += 4) {
                const float rs[4] = {Rm[s * LB + i], Rm[(s + 1) * LB + i], Rm[(s + 2) * LB + i],
                                     Rm[(s + 3) * LB + i]};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float4 g4 = *reinterpret_cast<const float4*>(Gg + (r0 + a) * LDT + s);
                    const float4 p4 = *reinterpret_cast<const float4*>(Pb + (r0 + a) * LDT + s);
                    sG[a] = fmaf(g4.x, rs[0], fmaf(g4.y, rs[1], fmaf(g4.z, rs[2], fmaf(g4.w, rs[3], sG[a]))));
                    sP[a] = fmaf(p4.x, rs[0], fmaf(p4.y, rs[1], fmaf(p4.z, rs[2], fmaf(p4.w, rs[3], sP[a]))));
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float fo = Fm[frow(J, r0 + a) * LB + i];
                LG[a] = fmaf(fo, sG[a], LG[a]);
                LP[a] = fmaf(fo, sP[a], LP[a]);
            }
        }
        // left sums on the diagonal block
        for (int s = 16 * I; s <= r0 + 3; ++s) {
            const float ks0 = kb[s * LB + i], gs = Gm[s * LB + i];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (s <= r0 + a) {
                    const float ks = ks0 * __expf(gr[a] - gs);
                    if (s < r0 + a) LG[a] = fmaf(Gg[(r0 + a) * LDT + s], ks, LG[a]);
                    LP[a] = fmaf(Pb[(r0 + a) * LDT + s], ks, LP[a]);
                }
            }
        }
        // right sums (the rows as columns s), off the diagonal block
        if (I < 3) {
            const int b = 16 * I + 15;
            float sG[4] = {0.f, 0.f, 0.f, 0.f}, sP[4] = {0.f, 0.f, 0.f, 0.f};
            for (int t = b + 1; t < C; ++t) {
                const float ft = Fm[frow(I, t) * LB + i];
                const float kt = kb[t * LB + i] * ft, qt = qb[t * LB + i] * ft;
                const float4 g4 = *reinterpret_cast<const float4*>(Gg + t * LDT + r0);
                const float4 p4 = *reinterpret_cast<const float4*>(Pb + t * LDT + r0);
                sG[0] = fmaf(g4.x, kt, sG[0]);
                sG[1] = fmaf(g4.y, kt, sG[1]);
                sG[2] = fmaf(g4.z, kt, sG[2]);
                sG[3] = fmaf(g4.w, kt, sG[3]);
                sP[0] = fmaf(p4.x, qt, sP[0]);
                sP[1] = fmaf(p4.y, qt, sP[1]);
                sP[2] = fmaf(p4.z, qt, sP[2]);
                sP[3] = fmaf(p4.w, qt, sP[3]);
            }
            const float gb = Gm[b * LB + i];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float fr = __expf(gb - gr[a]);
                RG[a] = fr * sG[a];
                RP[a] = fr * sP[a];
            }
        }
        // right sums on the diagonal block
        for (int t = r0; t < 16 * I + 16; ++t) {
            const float gt = Gm[t * LB + i], kt0 = kb[t * LB + i], qt0 = qb[t * LB + i];
            const float4 g4 = *reinterpret_cast<const float4*>(Gg + t * LDT + r0);
            const float4 p4 = *reinterpret_cast<const float4*>(Pb + t * LDT + r0);
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (t >= r0 + a) {
                    const float e = __expf(gt - gr[a]);
                    if (t > r0 + a) RG[a] = fmaf(gv[a], kt0 * e, RG[a]);
                    RP[a] = fmaf(pv[a], qt0 * e, RP[a]);
                }
            }
        }
        const float g63 = Gm[(C - 1) * LB + i];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int r = r0 + a;
            const float k_r = kb[r * LB + i], q_r = qb[r * LB + i];
            const float E = __expf(gr[a]), ed = __expf(g63 - gr[a]);
            const int64_t gi = (rowbase + r) * Dk + cb0 + i;
            const float Kd = k_r * ed;
            p.dqh[gi] = fmaf(qrb[a], E, LP[a]);
            p.dkh[gi] = krb[a] * E + kdb[a] * ed + LG[a] + RG[a] + RP[a];
            Gb[r * LB + i] = qrb[a] * q_r * E + krb[a] * k_r * E - kdb[a] * Kd + q_r * LP[a] +
                             k_r * (LG[a] - RG[a] - RP[a]);
            colK = fmaf(kdb[a], Kd, colK);
        }
    }
    part[warp * CB + i] = colK;
    __syncthreads();
    if (tid < CB) {  // Gammabar_63: the K_d column sums (warp order) and the state decay
        float tot = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) tot += part[w * CB + tid];
        Gb[(C - 1) * LB + tid] += tot + p.ecb[ci * Dk + cb0 + tid] * __expf(Gm[(C - 1) * LB + tid]);
    }
    __syncthreads();
    // lbar: sums of Gammabar from the end of the chunk; warp w takes rows 8 w .. 8 w + 7
    float piece = 0.f;
    for (int t = 8 * warp; t < 8 * warp + 8; ++t) piece += Gb[t * LB + i];
    part[warp * CB + i] = piece;
    __syncthreads();
    float acc = 0.f;
    for (int w = kThreads / 32 - 1; w > warp; --w) acc += part[w * CB + i];
    __nv_bfloat16* dlg = static_cast<__nv_bfloat16*>(p.da);
    for (int t = 8 * warp + 7; t >= 8 * warp; --t) {
        acc += Gb[t * LB + i];
        if (t < nvalid)
            dlg[(((int64_t)bb * d.T + t0 + t) * d.Hv + h) * Dk + cb0 + i] = __float2bfloat16_rn(on[t] != 0.f ? acc : 0.f);
    }
}

inline size_t kc_gate_smem() { return 3 * kBlkMat + 3 * C * 4; }
inline size_t kc_chan_smem() { return 2 * kBlkMat + 4 * kBlkArr + (96 + 48) * LB * 4 + (8 * CB + 4 * C) * 4; }

}  // namespace

bool kc_chunked_supported(const Dims& d) {
    return d.dtype == 1 && d.Dv == 128 && (d.Dk == 64 || d.Dk == 128 || d.Dk == 192) &&
           scan_ta_supported(d) && kf_plan((int)d.Dk, (int)d.Dv).total + 1024 <= 227u * 1024u;
}

cudaError_t launch_kc_bwd_prod(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = kp_plan((int)d.Dv).total + 1024;
    auto kern = kc_bwd_prod_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kThreads, smem, s>>>(d, p, *p.tmaps);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_kc_bwd_gate(const Dims& d, const Ptrs& p, cudaStream_t s) {
    auto kern = kc_bwd_gate_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kc_gate_smem());
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B), kThreads, kc_gate_smem(), s>>>(d, p);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_kc_bwd_chan(const Dims& d, const Ptrs& p, cudaStream_t s) {
    auto kern = kc_bwd_chan_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kc_chan_smem());
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(d.NC * (d.Dk / CB)), (unsigned)d.Hv, (unsigned)d.B), kThreads, kc_chan_smem(), s>>>(d, p);
    count_launches(1);
    return cudaPeekAtLastError();
}

cudaError_t launch_kc_chunk(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = kf_plan((int)d.Dk, (int)d.Dv).total;
    auto kern = kc_chunk_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)d.NC, (unsigned)d.Hv, (unsigned)d.B);
    kern<<<grid, kChunkThreads, smem, s>>>(d, p);
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace gdn
