// gdn_bwd_tc.cu -- per-chunk gradient kernel of the VJP on the tensor cores
// (tcgen05, bf16 operands, fp32 accumulators in TMEM) for bf16 inputs.
//
// Same equations as the CUDA-core version in gdn_bwd.cu (reverse-mode
// derivative of the chunked WY/UT form; mlx-lm PR "Add gated_delta_update
// VJP", "What this PR adds" and "Scope and follow-ups").  One persistent CTA
// per SM walks the work items (chunk, value head, batch), loading the next
// item's operands while it stores the current one's results; every product
// has 64 rows as its M dimension
// (M = 64 MMAs, accumulator row r in TMEM lane 32 (r / 16) + r % 16):
//   phase 0:  Pbar = Obar Delta^T,  Dbar V^T,  Y = T^T Dbar
//   phase 1:  per 64-wide block of Dk:  Delta Sbar'^T,  Obar S^T,  Wbar = -Dbar S^T
//   phase 1b: Wbar K^T,  diag(beta gam) T^T Wbar,  K K^T
//   phase 2:  X = Tbar T^T,  Q K^T,  Abar = -T^T X,  then the gate / log-decay
//             cotangents element-wise in fp32 (fp64 for the cancelling sums)
//   phase 3:  (Pbar o M) K  and  (Pbar o M)^T Q + (Gb + Gb^T) K
// The cotangents of the normalised q and k rows accumulate in TMEM from
// phase 1 on (the state products of phase 1, rescaled in place, then Z and
// the phase-3 products on top) and are stored once at the end.
// Delta (a cancelling difference) enters as two bf16 terms (hi + lo).  q and k
// are staged as the exact bf16 inputs; the norms r_q, r_k (and 1/sqrt(Dk)) are
// applied in fp32 in the epilogues or folded into the other operand, so the
// normalised rows are never rounded.  The saved intermediates (Delta hi / lo,
// -Dbar, T, the state checkpoints S and the chunk-end cotangents Sbar') are
// bf16 operand images written by the earlier kernels; each arrives with one
// bulk copy, and the 64-wide Dk blocks of S / Sbar' stream through one buffer so the
// next block streams in while the current block's epilogue runs.
#include "gdn_internal.cuh"
#include "gdn_scan_ta.cuh"
#include "gdn_tc.cuh"

namespace gdn {

GDN_ERROR_WORD(bwdtc)

namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int kBlkK = 64;  // Dk block of the state products (the last one may be 32)
// TMEM column map (Dk <= 192): scratch S1 = [0, 64); dk accumulator AK = [64, 64 + Dk);
// dq accumulator AQ = [64 + Dk, 64 + 2 Dk); scratch S2 = 64 columns from
// 64 + max(2 Dk, Dv).  Phase 0 parks Y (Dv <= 256 columns) at 64, before AK /
// AQ are live.
constexpr uint32_t kS1 = 0, kAK = 64;
// fp32 64 x 64 scratch matrices have rows of 68 floats: 16-byte aligned rows
// (row-wise runs move as float4) four banks apart, so eight lanes that own eight
// rows touch 32 distinct banks; an unpadded 256-byte row stride would put every
// lane in one bank
constexpr int LDM = C + 4;

__device__ __forceinline__ void ld_row8(const float* src, float* v) {
    const float4 a = reinterpret_cast<const float4*>(src)[0], b = reinterpret_cast<const float4*>(src)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st_row8(float* dst, const float* v) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

struct Smem {
    // byte offsets inside dynamic shared memory
    uint32_t K, Q, W, R1, O, D, Dlo, NB, V, S, Sp, Gkk, Gqk, Tbh, Xh, PMk, PMq, Hk, Tsc, Tt, Pf,
        Tbf, vec, total;
};

__host__ __device__ inline Smem smem_plan(int Dk, int Dv) {
    Smem s{};
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
        const uint32_t r = o;
        o += (bytes + 1023u) & ~1023u;
        return r;
    };
    const uint32_t tk = C * Dk * 2, tv = C * Dv * 2, t64 = C * C * 2, f64x64 = C * LDM * 4;
    s.K = take(tk);
    s.Q = take(tk);
    s.W = take(tk);
    // region R1: Dv-wide operands of phases 0-1, then phase-2/3 scratch
    const uint32_t r1_ops = 5 * tv + 2 * (tv / 2);
    const uint32_t r1_late = 2 * f64x64 + 6 * t64;
    s.R1 = take(r1_ops > r1_late ? r1_ops : r1_late);
    s.O = s.R1;
    s.D = s.O + tv;
    s.Dlo = s.D + tv;
    s.NB = s.Dlo + tv;
    s.V = s.NB + tv;
    s.S = s.V + tv;  // with V: one Dk block of S and of Sbar' (2 x 64 x Dv bf16)
    s.Sp = s.S + tv / 2;
    s.Gkk = s.R1;            // fp32, later Mbar o M in place
    s.Gqk = s.Gkk + f64x64;  // fp32, later Gb in place
    s.Tbh = s.Gqk + f64x64;
    s.Xh = s.Tbh + t64;
    s.PMk = s.Xh + t64;
    s.PMq = s.PMk + t64;
    s.Hk = s.PMq + t64;
    s.Tsc = s.Hk + t64;      // diag(beta gam)-scaled T image
    s.Tt = take(t64);
    s.Pf = take(f64x64);
    s.Tbf = take(f64x64);
    s.vec = take(40 * C * 4 + 2 * C * 8 + 1024);
    s.total = o;
    return s;
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
__device__ __forceinline__ void ld_bf16x8(const uint8_t* src, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ uint32_t canon(int x, int y, int ncols) {
    return (uint32_t)(x >> 3) * 128u + (uint32_t)(y >> 3) * (uint32_t)ncols * 16u +
           (uint32_t)(y & 7) * 16u + (uint32_t)(x & 7) * 2u;
}
// 16 consecutive elements (x0 multiple of 8) of row y of a 64-row panel tile
__device__ __forceinline__ void panel_row16(const uint8_t* tile, int x0, int y, float* v) {
    ld_bf16x8(tile + tc::panel_off(x0, y, C), v);
    ld_bf16x8(tile + tc::panel_off(x0 + 8, y, C), v + 8);
}
__device__ __forceinline__ void tile_put16(uint8_t* tile, int ncols, int x0, int y, const float* v) {
    st_bf16x8(tile + canon(x0, y, ncols), v);
    st_bf16x8(tile + canon(x0 + 8, y, ncols), v + 8);
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

// Walk an M = 64 accumulator of `ncols` columns (a multiple of 32) at TMEM
// column col0 with every thread of the eight warps busy: 32-column pieces,
// taken in turn by the two warp groups g = warp / 4; in a piece at column c,
// thread l < 16 of warp w holds row 16 (w % 4) + l at columns c .. c + 15 and
// thread l + 16 the same row at columns c + 16 .. c + 31 (the 16x32bx2 TMEM
// shape).  f(row, first column, 16 values) is called by all 32 lanes; a
// per-row sum adds its two lane halves with row_pair_sum.
template <typename F>
__device__ __forceinline__ void acc_rows1(uint32_t tbase, uint32_t col0, int ncols, F&& f) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int sp = w & 3, g = w >> 2, hl = l >> 4;
    for (int c = 32 * g; c < ncols; c += 64) {
        float v[16];
        tc::tmem_ld16x2<16>(tc::tmem_addr(tbase, 32 * sp, col0 + c), v);
        tc::tmem_wait_ld();
        f(16 * sp + (l & 15), c + 16 * hl, v);
    }
}
// As acc_rows1 with two pieces in flight per wait
template <typename F>
__device__ __forceinline__ void acc_rows2(uint32_t tbase, uint32_t col0, int ncols, F&& f) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int sp = w & 3, g = w >> 2, hl = l >> 4;
    for (int c = 32 * g; c < ncols; c += 128) {
        float v[2][16];
        const bool two = c + 64 < ncols;  // warp-uniform
        tc::tmem_ld16x2<16>(tc::tmem_addr(tbase, 32 * sp, col0 + c), v[0]);
        if (two) tc::tmem_ld16x2<16>(tc::tmem_addr(tbase, 32 * sp, col0 + c + 64), v[1]);
        tc::tmem_wait_ld();
        f(16 * sp + (l & 15), c + 16 * hl, v[0]);
        if (two) f(16 * sp + (l & 15), c + 64 + 16 * hl, v[1]);
    }
}
// A row's two lane halves (lanes l and l + 16) summed; every lane gets the total
__device__ __forceinline__ float row_pair_sum(float s) { return s + __shfl_xor_sync(0xffffffffu, s, 16); }
// As acc_rows1, handing each lane's 16 columns to f in two 8-column runs:
// f(row, first column, 8 values, lane half)
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
        f(16 * sp + (l & 15), c + 16 * hl, x, hl);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = v[8 + i];
        f(16 * sp + (l & 15), c + 16 * hl + 8, x, hl);
    }
}

// Unevaluated sums hi + lo of two floats (Knuth's two-sum, Dekker's fast
// two-sum): ~48-bit sums in fp32 arithmetic, for the cancelling log-decay sums
struct f2 {
    float hi, lo;
};
__device__ __forceinline__ f2 two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ f2 f2_add(f2 x, f2 y) {
    const f2 s = two_sum(x.hi, y.hi);
    const float lo = s.lo + (x.lo + y.lo);
    const float h = s.hi + lo;
    return {h, lo - (h - s.hi)};
}

// Completion of an MMA round on `bar`: waiting threads wait for it; every thread
// advances its copy of the barrier's phase
__device__ __forceinline__ void sync_after_mma(uint64_t* bar, uint32_t& phase, bool& ok, bool wait) {
    if (wait) {
        ok = tc::mbar_wait(bar, phase, &g_err_bwdtc) && ok;
        tc::tc_fence_after();
    }
    phase ^= 1u;
}
__device__ __forceinline__ void cta_sync_tc() {
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
}

// Work items are (chunk, value head, batch) in order of decreasing chunk, the
// (batch, value head) pairs of a chunk consecutive (the value heads of a key head
// share their q / k images).  Each CTA takes its next item from the counter
// *sched (zero before the launch).  progress (null: the inputs are all there):
// the reverse scan's per-(b, h) count of finished chunks (ntiles value tiles per
// head); item (c, h, b) waits until it reaches ntiles (NC - c).
__device__ __forceinline__ void bwd_chunk_body(const Dims& d, const Ptrs& p, const Tmaps& tm,
                                               unsigned int* sched, const unsigned int* progress,
                                               int ntiles) {
    extern __shared__ __align__(1024) uint8_t sm[];
    // bar: MMA rounds outside phase 1; barOV, barL, barKQ: arrivals of an item's
    // operands.  Phase 1 (one of each per Dk block b, completing once per item):
    // barMa1[b] the block's Delta Sbar'^T products done, barM2[b] its Obar S^T and
    // -Dbar S^T products done, barG2[b] its tiles read by the <S, Sbar'> sums,
    // barE2[b] its epilogue done (Wbar scratch free); barT[s]: arrivals of the
    // tiles of slot s (several per item)
    __shared__ uint64_t bar, barOV, barL, barKQ, barAQ, barT[5], barMa1[4], barM2[4], barG2[4], barE2[4];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int next_item;
    const int Dk = (int)d.Dk, Dv = (int)d.Dv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps 0-7: epilogues (row quarter warp % 4, column half g); warp 8: loads and MMA
    // issue; warp 9: MMA issue of the second of two independent product chains.  One
    // thread issues a tcgen05.mma about every 80 cycles whatever its size, so small
    // products from two issuing warps run side by side on the tensor core.
    const bool epi = tid < kThreads;
    const bool prod = tid == kThreads;
    const bool prod2 = tid == kThreads + 32;
    const int g = (warp >> 2) & 1;
    const Smem L = smem_plan(Dk, Dv);
    float* vec = reinterpret_cast<float*>(sm + L.vec);
    float* gm = vec;             // exp(Gamma)
    float* ev = gm + C;          // exp(Gamma_63 - Gamma)
    float* bt = ev + C;          // beta
    float* rqv = bt + C;         // r_q / sqrt(Dk)
    float* rkv = rqv + C;        // r_k
    float* gq = rkv + C;         // [2][64] row-dot partials: gambar * gam
    float* ee = gq + 2 * C;      // [2][64] ebar * e
    float* bb0 = ee + 2 * C;     // [2][64] betabar (Y . V)
    float* zk = bb0 + 2 * C;     // [2][64] Z . K
    float* sbp = zk + 2 * C;     // [4][64] sum_j Abar M Gkk
    float* betab = sbp + 4 * C;  // [64]
    float* red = betab + C;      // [256]
    // Gamma as an unevaluated sum hi + lo of two floats: for steps i, j whose
    // Gamma are within a factor of two (the only case where exp(Gamma_i - Gamma_j)
    // is not negligible), (hi_i - hi_j) is exact and the difference keeps fp64
    // accuracy without fp64 arithmetic
    float* Ghi = red + 256;     // [64]
    float* Glo = Ghi + C;       // [64]
    float* rsp = Glo + C;       // [4][64] row sums of Mbar o M (compensated)
    float* rsc = rsp + 4 * C;   // [4][64] their compensation terms
    float* csp = rsc + 4 * C;   // [4][64] column sums (compensated, folded)
    float* gbh = csp + 4 * C;   // [64] Gammabar as hi + lo
    float* gbl = gbh + C;       // [64]
    // Off the diagonal 16 x 16 blocks, M_ij = exp(Gamma_i - Gamma_j) is the
    // product of two factors through the last step b = 16 J + 15 of the column
    // block J of j: uf[J][i] = exp(Gamma_i - Gamma_b) (i > b) and wf[J][j] =
    // exp(Gamma_b - Gamma_j) (j <= b), both in (0, 1] since Gamma does not increase
    float* uf = gbl + C;        // [3][64]
    float* wf = uf + 3 * C;     // [3][64]

    // Persistent: the next item's operands load while the current one ends.
    const int nitems = (int)(d.NC * d.Hv * d.B);
    const int nbh = (int)(d.Hv * d.B);
    auto item_c = [&](int it) { return (int)d.NC - 1 - it / nbh; };
    auto item_h = [&](int it) { return (it % nbh) % (int)d.Hv; };
    auto item_b = [&](int it) { return (it % nbh) / (int)d.Hv; };
    // producer: the reverse scan has finished chunk c of this head (bounded wait)
    auto wait_ready = [&](int it) -> bool {
        if (progress == nullptr) return true;
        const unsigned int* f = progress + (int64_t)item_b(it) * d.Hv + item_h(it);
        const unsigned int need = (unsigned int)(ntiles * ((int)d.NC - item_c(it)));
        if (!tc::poll_geq(f, need, &g_err_bwdtc, tc::kWaitLimitNs)) return false;
        tc::fence_async_global();  // the images it saw released, before the copies read them
        return true;
    };
    __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(p.dv);
    const int64_t ldv = d.Hv * Dv;
    const uint32_t tv = (uint32_t)(C * Dv * 2);         // one 64 x Dv bf16 tile
    const uint32_t tk = (uint32_t)(C * Dk * 2);         // one 64 x Dk bf16 tile
    const uint32_t blk = (uint32_t)(kBlkK * Dv * 2);    // one full Dk block of S (or Sbar')
    // Dk block b of S / Sbar' (panels 8b .. 8b + nk(b) / 8 - 1 of the images of
    // chunk image ci) goes to one of five tile slots: slot 0 in the space of the V
    // tile (free once phase 0 is done), slot 1 right after it (never used by phase
    // 0), slots 2 and 3 in the space of the Delta hi / lo tiles (free once the
    // Delta Sbar'^T products are done), slot 4 in the Wbar staging tile (free until
    // walk 2's epilogues write Wbar).  Walk 1 (Delta Sbar'^T) with three blocks
    // reads Sbar' block 1 from slot 1 and block 2 from slot 4, both loaded with the
    // phase-1 group of copies, and block 0 from slot 0, loaded once phase 0 is
    // done, so that blocks 0 and 1 lie side by side and go through one 128-wide
    // product while the second issuer takes block 2; with fewer blocks, block 0
    // comes early in slot 1 and block 1 in slot 0, one per issuer.  The blocks stay
    // there for the <S, Sbar'> sums of walk 2, which so loads only S: walk-2
    // position p takes block w2_blk(p) (order 2, 0, 1 for three blocks, so that
    // the Wbar of block 2 is written first, beside Sbar' block 2) from slot 2
    // (even p) or 3 (odd p), the third position once the first is done.  Per item,
    // slot 0 takes one tile when nblk > 1, slot 1 one, slot 2 ceil(nblk / 2), slot 3
    // floor(nblk / 2), slot 4 one when nblk = 3; a wait on slot s for its occ-th tile
    // of the item uses parity (iord * uses(s) + occ) & 1.
    const int nblk = (Dk + kBlkK - 1) / kBlkK;  // 1 .. 3 (Dk <= 192)
    auto nkb = [&](int b) { return Dk - b * kBlkK < kBlkK ? Dk - b * kBlkK : kBlkK; };
    auto slot_ptr = [&](int sl) -> uint8_t* {
        return sm + (sl == 0 ? L.V : sl == 1 ? L.V + blk : sl == 2 ? L.D : sl == 3 ? L.Dlo : L.W);
    };
    auto slot_uses = [&](int sl) -> uint32_t {
        return sl == 0 ? (uint32_t)(nblk > 1) : sl == 1 ? 1u : sl == 2 ? (uint32_t)((nblk + 1) / 2)
               : sl == 3 ? (uint32_t)(nblk / 2) : (uint32_t)(nblk == 3);
    };
    auto sbar_slot = [&](int b) { return b == 2 ? 4 : (nblk == 3) == (b == 1) ? 1 : 0; };
    auto w2_blk = [&](int p) { return nblk == 3 ? (p == 0 ? 2 : p - 1) : p; };
    auto load_tile = [&](const void* img, int64_t ci, int b, int sl) {
        const uint32_t bytes = (uint32_t)(nkb(b) * Dv * 2);
        tc::mbar_arrive_expect_tx(&barT[sl], bytes);
        tc::bulk_g2s(slot_ptr(sl), static_cast<const uint8_t*>(img) + ci * (int64_t)Dk * Dv * 2 + (int64_t)b * blk,
                     bytes, &barT[sl]);
    };
    // ---- operands of item it, all issued by the producer, in two groups.  Phase 0:
    // raw dO, v by TMA in the panel layout, Delta (hi + lo), -Dbar and T by bulk
    // copies.  Phase 1 (issued once the phase-0 products are, so that the first
    // group, which every SM wants at about the same time, is smaller): the k, q
    // images and the first Sbar' block (its half of the block buffer is not used
    // by phase 0).
    auto issue_loads = [&](int it) {
        const int c = item_c(it), h = item_h(it), bb = item_b(it);
        const int64_t ci = ((int64_t)bb * d.Hv + h) * d.NC + c;
        tc::mbar_arrive_expect_tx(&barOV, 2 * tv);
        tc::tma_load_5d(sm + L.O, &tm.dOf, 0, c * C, 0, h, bb, &barOV);
        tc::tma_load_5d(sm + L.V, &tm.v, 0, c * C, 0, h, bb, &barOV);
        const uint8_t* dl_img = reinterpret_cast<const uint8_t*>(p.Delta) + ci * (int64_t)C * Dv * 4;
        tc::mbar_arrive_expect_tx(&barL, 3 * tv + C * C * 2);
        tc::bulk_g2s(sm + L.D, dl_img, tv, &barL);
        tc::bulk_g2s(sm + L.Dlo, dl_img + tv, tv, &barL);
        tc::bulk_g2s(sm + L.NB, reinterpret_cast<const uint8_t*>(p.Dbar) + ci * (int64_t)tv, tv, &barL);
        tc::bulk_g2s(sm + L.Tt, reinterpret_cast<const uint8_t*>(p.Tinv) + ci * (int64_t)C * C * 2,
                     C * C * 2, &barL);
        // the state and state-cotangent images that phase 1 streams through its
        // slots, into L2 now: a slot's copy then waits for L2, not for DRAM
        const uint32_t sbytes = (uint32_t)(Dk * Dv * 2);
        tc::bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(p.dSck) + ci * (int64_t)sbytes, sbytes);
        tc::bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(p.ckpt) + ci * (int64_t)sbytes, sbytes);
    };
    auto issue_loads_kq = [&](int it) {
        const int c = item_c(it), h = item_h(it), bb = item_b(it);
        const int j = h / (int)d.G;
        const int64_t ci = ((int64_t)bb * d.Hv + h) * d.NC + c;
        const int64_t kqi = ((int64_t)bb * d.Hk + j) * d.NC + c;  // q / k images of this chunk
        tc::mbar_arrive_expect_tx(&barKQ, 2 * tk);
        tc::bulk_g2s(sm + L.K, static_cast<const uint8_t*>(p.kimg) + kqi * tk, tk, &barKQ);
        tc::bulk_g2s(sm + L.Q, static_cast<const uint8_t*>(p.qimg) + kqi * tk, tk, &barKQ);
        load_tile(p.dSck, ci, nblk == 3 ? 1 : 0, 1);
        if (nblk == 3) load_tile(p.dSck, ci, 2, 4);
    };
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base_sh, 512);
        tc::tmem_relinquish();
    }
    if (prod) {
        tc::mbar_init(&bar, 2);  // every MMA round: one commit (or arrival) from each issuer
        tc::mbar_init(&barOV, 1);
        tc::mbar_init(&barL, 1);
        tc::mbar_init(&barKQ, 1);
        tc::mbar_init(&barAQ, 1);  // the producer's phase-3 chain (dq complete), once per item
        tc::mbar_init(&barT[4], 1);
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(&barT[i], 1);
            tc::mbar_init(&barMa1[i], 1);
            tc::mbar_init(&barM2[i], 2);
            tc::mbar_init(&barG2[i], kThreads);
            tc::mbar_init(&barE2[i], kThreads);
        }
        tc::fence_mbar_init();
        const int first = (int)atomicAdd(sched, 1u);
        next_item = first;
        if (first < nitems && !wait_ready(first)) next_item = nitems;  // gave up: no item
        else if (first < nitems) issue_loads(first);
    }
    cta_sync_tc();
    const uint32_t tb = tmem_base_sh;
    uint32_t phase = 0;        // parity of the next completion of bar (MMA rounds)
    uint32_t pit = 0;          // parity of the per-item arrivals (barOV, barL, barKQ)
    uint32_t iord = 0;         // items this CTA has run before (parities of the phase-1 barriers)
    bool ok = true;
    // producer: an item whose operands are in flight but not yet waited for
    bool pending = false;
    uint32_t pend_pit = 0;
    for (int it = next_item; it < nitems; it = next_item, pit ^= 1u, ++iord) {
    pending = false;
    const int c = item_c(it), h = item_h(it), bb = item_b(it);
    const int j = h / (int)d.G;
    const int64_t t0 = (int64_t)c * C;
    const int nvalid = (int)(d.T - t0 < C ? d.T - t0 : C);
    const int64_t gbase = ((int64_t)bb * d.Hv + h) * d.Tp + t0;
    const int64_t rbase = ((int64_t)bb * d.Hk + j) * d.Tp + t0;
    const int64_t ci = ((int64_t)bb * d.Hv + h) * d.NC + c;  // chunk image index
    if (tid < C) {
        const double G = p.gam[gbase + tid];
        const float ghi = (float)G;
        Ghi[tid] = ghi;
        Glo[tid] = (float)(G - (double)ghi);
        gm[tid] = expf((float)G);
        ev[tid] = expf((float)(p.gam[gbase + C - 1] - G));
        bt[tid] = p.beta[gbase + tid];
        rqv[tid] = p.rq[rbase + tid] * rsqrtf((float)Dk);
        rkv[tid] = p.rk[rbase + tid];
    }
    for (int i = tid; i < 12 * C; i += blockDim.x) gq[i] = 0.f;  // gq, ee, bb0, zk, sbp
    for (int i = tid; i < 8 * C; i += blockDim.x) rsp[i] = 0.f;  // rsp, rsc
    cta_sync_tc();
    if (tid < 3 * C) {  // decay factors (read first by the element-wise phase)
        const int J = tid / C, i = tid % C, b = 16 * J + 15;
        const float dg = (Ghi[i] - Ghi[b]) + (Glo[i] - Glo[b]);
        uf[tid] = i > b ? expf(dg) : 0.f;
        wf[tid] = i <= b ? expf(-dg) : 0.f;
    }
    ok = tc::mbar_wait(&barOV, pit, &g_err_bwdtc) && ok;
    ok = tc::mbar_wait(&barL, pit, &g_err_bwdtc) && ok;

    // k, q, dO, v tiles: panel layout (x = column, 64 rows); Wbar tile: canonical
    const tc::Tile tK = tc::panel_tile(sm + L.K, C, true), tQ = tc::panel_tile(sm + L.Q, C, true);
    const tc::Tile tKmn = tc::panel_tile(sm + L.K, C, false), tQmn = tc::panel_tile(sm + L.Q, C, false);
    const tc::Tile tW = tc::panel_tile(sm + L.W, C, true), tWmn = tc::panel_tile(sm + L.W, C, false);
    const tc::Tile tO = tc::panel_tile(sm + L.O, C, true), tV = tc::panel_tile(sm + L.V, C, true);
    // Delta / -Dbar images: x = step t (canonical, 8-row groups of Dv 1024 bytes apart)
    const tc::Tile tDmn = mnmaj(sm, L.D, C), tDlomn = mnmaj(sm, L.Dlo, C);
    const tc::Tile tNB = kmaj(sm, L.NB, C), tNBmn = mnmaj(sm, L.NB, C);
    // T image: panel layout, x = column j
    const tc::Tile tTt = tc::panel_tile(sm + L.Tt, C, true), tTmn = tc::panel_tile(sm + L.Tt, C, false);

    // S2 also clears Y (Dv columns from kAK) of phase 0
    const uint32_t kAQ = kAK + (uint32_t)Dk, kS2 = kAK + (uint32_t)(2 * Dk > Dv ? 2 * Dk : Dv);

    // ---- phase 0: Pbar = Obar Delta^T | -Dbar V^T | -T^T Dbar
    if (prod) {
        tc::mma_tile(tb + kS1, tO, tDmn, C, C, Dv, false);
        tc::mma_tile(tb + kS1, tO, tDlomn, C, C, Dv, true);
        tc::mma_commit(&bar);
        issue_loads_kq(it);
    } else if (prod2) {
        tc::mma_tile(tb + kS2, tNBmn, tV, C, C, Dv, false);
        tc::mma_tile(tb + kAK, tTmn, tNB, C, Dv, C, false);
        tc::mma_commit(&bar);
    }
    float* Pf = reinterpret_cast<float*>(sm + L.Pf);
    float* Tbf = reinterpret_cast<float*>(sm + L.Tbf);
    sync_after_mma(&bar, phase, ok, epi);
    if (epi) {
        if (ok) {
            acc_rows2(tb, kS1, C, [&](int r, int c0, const float (&x)[16]) {
                float m[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) m[i] = (c0 + i <= r) ? x[i] : 0.f;
                st_row8(Pf + r * LDM + c0, m);
                st_row8(Pf + r * LDM + c0 + 8, m + 8);
            });
            acc_rows2(tb, kS2, C, [&](int r, int c0, const float (&x)[16]) {
                float m[16];
#pragma unroll
                for (int i = 0; i < 16; i += 8) ld_row8(bt + c0 + i, m + i);  // per-column vectors as float4
#pragma unroll
                for (int i = 0; i < 16; ++i) m[i] = -m[i] * x[i];
                st_row8(Tbf + r * LDM + c0, m);
                st_row8(Tbf + r * LDM + c0 + 8, m + 8);
            });
            acc_rows1(tb, kAK, Dv, [&](int r, int c0, const float (&x)[16]) {
                float vv[16], y[16];
                panel_row16(sm + L.V, c0, r, vv);
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    s = fmaf(-x[i], vv[i], s);
                    y[i] = -bt[r] * x[i];
                }
                s = row_pair_sum(s);
                if (lane < 16) bb0[g * C + r] += s;
                if (r < nvalid) {
                    uint8_t* dst = reinterpret_cast<uint8_t*>(dv + ((int64_t)bb * d.T + t0 + r) * ldv +
                                                              (int64_t)h * Dv + c0);
                    st_bf16x8(dst, y);
                    st_bf16x8(dst + 16, y + 8);
                }
            });
        }
    }
    cta_sync_tc();  // phase-0 reads of TMEM and of the V tile are done

    // ---- phase 1: state products per kBlkK-wide block of Dk, in two walks over
    // the blocks (slots: see load_tile above).  Walk 1: Delta Sbar'^T (hi + lo)
    // into the dk accumulator, the blocks' products issued as their Sbar' tiles
    // arrive (block 1 by the second issuer); the epilogue rescales dk by e and
    // forms <dk, k> per row.  Walk 2, once every walk-1 product is done (slots 2
    // and 3 free): per position p, Obar S^T into the dq accumulator (producer) and
    // -Dbar S^T into the Wbar scratch (second issuer; S1 for even, S2 for odd p,
    // reused once the epilogue of position p - 2 released it); the epilogue forms
    // <S, Sbar'> from the S tile and the Sbar' tile of walk 1, rescales dq by gam,
    // forms <dq, q> per row and stages Wbar as a bf16 panel tile.
    float gcb = 0.f;
    const uint32_t ip = iord & 1u;  // parity of the per-block barriers in this item
    auto slot_par = [&](int sl, int occ) { return (iord * slot_uses(sl) + (uint32_t)occ) & 1u; };
    // walk-1 products of blocks b0 .. b0 + nb - 1 (one or two adjacent tiles from
    // slot sbar_slot(b0)), committed to each block's barrier
    auto walk1_blocks = [&](int b0, int nb) {
        const int sl = sbar_slot(b0);
        int nk = 0;
        for (int b = b0; b < b0 + nb; ++b) {
            ok = tc::mbar_wait(&barT[sbar_slot(b)], slot_par(sbar_slot(b), 0), &g_err_bwdtc) && ok;
            nk += nkb(b);
        }
        const tc::Tile tSp = tc::panel_tile(slot_ptr(sl), Dv, false);
        tc::mma_tile(tb + kAK + b0 * kBlkK, tDmn, tSp, C, nk, Dv, false);
        tc::mma_tile(tb + kAK + b0 * kBlkK, tDlomn, tSp, C, nk, Dv, true);
        for (int b = b0; b < b0 + nb; ++b) tc::mma_commit(&barMa1[b]);
    };
    if (prod) {
        if (nblk >= 2) load_tile(p.dSck, ci, nblk == 3 ? 0 : 1, 0);  // the V tile is dead: phase 0 is done
        walk1_blocks(0, nblk == 3 ? 2 : 1);
        for (int b = 0; b < nblk; ++b)  // every walk-1 product done: slots 2, 3 free
            ok = tc::mbar_wait(&barMa1[b], ip, &g_err_bwdtc) && ok;
        load_tile(p.ckpt, ci, w2_blk(0), 2);
        if (nblk >= 2) load_tile(p.ckpt, ci, w2_blk(1), 3);
        for (int q = 0; q < nblk; ++q) {  // walk 2: Obar S^T
            const int b = w2_blk(q), sS = (q & 1) ? 3 : 2;
            if (q == 2) {  // slot 2 again, once position 0's products and sums are done
                ok = tc::mbar_wait(&barM2[0], ip, &g_err_bwdtc) && ok;
                ok = tc::mbar_wait(&barG2[0], ip, &g_err_bwdtc) && ok;
                load_tile(p.ckpt, ci, w2_blk(2), 2);
            }
            ok = tc::mbar_wait(&barT[sS], slot_par(sS, q >> 1), &g_err_bwdtc) && ok;
            const tc::Tile tS = tc::panel_tile(slot_ptr(sS), Dv, false);
            tc::mma_tile(tb + kAQ + b * kBlkK, tO, tS, C, nkb(b), Dv, false);
            tc::mma_commit(&barM2[q]);
        }
    } else if (prod2) {
        if (nblk >= 2) walk1_blocks(nblk == 3 ? 2 : 1, 1);
        for (int q = 0; q < nblk; ++q) {  // walk 2: -Dbar S^T
            const int b = w2_blk(q), sS = (q & 1) ? 3 : 2;
            ok = tc::mbar_wait(&barT[sS], slot_par(sS, q >> 1), &g_err_bwdtc) && ok;
            if (q >= 2) ok = tc::mbar_wait(&barE2[q - 2], ip, &g_err_bwdtc) && ok;
            const uint32_t wcol = (q & 1) ? kS2 : kS1;
            const tc::Tile tS = tc::panel_tile(slot_ptr(sS), Dv, false);
            tc::mma_tile(tb + wcol, tNBmn, tS, C, nkb(b), Dv, false);
            tc::mma_commit(&barM2[q]);
        }
    } else if (epi) {
        ok = tc::mbar_wait(&barKQ, pit, &g_err_bwdtc) && ok;
        const int sp = warp & 3, hl = lane >> 4;
        const int r = 16 * sp + (lane & 15);  // the accumulator row of this lane
        // a block's 32-column pieces (nk is 64 or 32) go to the warp groups in
        // turn; lanes l and l + 16 take columns 16 (l / 16) .. + 15 of a piece
        for (int b = 0; b < nblk; ++b) {  // walk 1: dk *= e, <dk, k> per row
            const int dk0 = b * kBlkK, nk = nkb(b);
            ok = tc::mbar_wait(&barMa1[b], ip, &g_err_bwdtc) && ok;
            tc::tc_fence_after();
            if (ok) {
                for (int cc = 32 * g; cc < nk; cc += 64) {
                    float ak[16];
                    const uint32_t ta = tc::tmem_addr(tb, 32 * sp, kAK + dk0 + cc);
                    tc::tmem_ld16x2<16>(ta, ak);
                    tc::tmem_wait_ld();
                    float kk[16];
                    panel_row16(sm + L.K, dk0 + cc + 16 * hl, r, kk);
                    float sk = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        ak[i] *= ev[r];
                        sk = fmaf(ak[i], kk[i], sk);
                    }
                    sk = row_pair_sum(sk);
                    if (lane < 16) ee[g * C + r] += sk;
                    tc::tmem_st16x2<16>(ta, ak);  // rescaled values back in place
                }
                tc::tmem_wait_st();
            }
        }
        for (int q = 0; q < nblk; ++q) {  // walk 2: <S, Sbar'>, dq *= gam, <dq, q>, Wbar tile
            const int b = w2_blk(q), dk0 = b * kBlkK, nk = nkb(b);
            const int sS = (q & 1) ? 3 : 2, sP = sbar_slot(b);
            ok = tc::mbar_wait(&barT[sS], slot_par(sS, q >> 1), &g_err_bwdtc) && ok;
            ok = tc::mbar_wait(&barT[sP], slot_par(sP, 0), &g_err_bwdtc) && ok;
            const uint8_t* tSs = slot_ptr(sS);
            const uint8_t* tSps = slot_ptr(sP);
            const int bytes = nk * Dv * 2;
            for (int e = tid; e < bytes / 16; e += kThreads) {
                float a8[8], b8[8];
                ld_bf16x8(tSs + 16 * e, a8);
                ld_bf16x8(tSps + 16 * e, b8);
#pragma unroll
                for (int i = 0; i < 8; ++i) gcb = fmaf(a8[i], b8[i], gcb);
            }
            tc::mbar_arrive(&barG2[q]);
            ok = tc::mbar_wait(&barM2[q], ip, &g_err_bwdtc) && ok;
            // Wbar of blocks 0 and 1 overwrites Sbar' block 2 in slot 4: every
            // thread's sums over it (position 0) are done first
            if (nblk == 3 && q >= 1) ok = tc::mbar_wait(&barG2[0], ip, &g_err_bwdtc) && ok;
            tc::tc_fence_after();
            if (ok) {
                const uint32_t wcol = (q & 1) ? kS2 : kS1;
                for (int cc = 32 * g; cc < nk; cc += 64) {
                    float aq[16], wv[16];
                    const uint32_t ta = tc::tmem_addr(tb, 32 * sp, kAQ + dk0 + cc);
                    tc::tmem_ld16x2<16>(ta, aq);
                    tc::tmem_ld16x2<16>(tc::tmem_addr(tb, 32 * sp, wcol + cc), wv);
                    tc::tmem_wait_ld();
                    const int c0 = dk0 + cc + 16 * hl;
                    float qq[16];
                    panel_row16(sm + L.Q, c0, r, qq);
                    float sq = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        aq[i] *= gm[r];
                        sq = fmaf(aq[i], qq[i], sq);
                    }
                    sq = row_pair_sum(sq);
                    if (lane < 16) gq[g * C + r] += sq;
                    st_bf16x8(sm + L.W + tc::panel_off(c0, r, C), wv);  // Wbar: panel tile
                    st_bf16x8(sm + L.W + tc::panel_off(c0 + 8, r, C), wv + 8);
                    tc::tmem_st16x2<16>(ta, aq);
                }
                tc::tmem_wait_st();
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&barE2[q]);
        }
        // <S, Sbar'> of this CTA: warp sums by a fixed shuffle tree, then in warp order
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) gcb += __shfl_xor_sync(0xffffffffu, gcb, off);
        if (lane == 0) red[warp] = gcb;
    }
    cta_sync_tc();  // phase 1 done: its operand space (under the phase-2/3 scratch) is free
    // diag(beta gam) T^T as an operand: T image columns scaled by beta gam
    for (int e = tid; e < C * (C / 8); e += blockDim.x) {
        const int j0 = (e / C) * 8;  // panel chunk e: row e % 64, columns j0 .. j0 + 7
        float t8[8];
        ld_bf16x8(sm + L.Tt + 16 * e, t8);
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] *= bt[j0 + i] * gm[j0 + i];
        st_bf16x8(sm + L.Tsc + 16 * e, t8);
    }
    tc::fence_async_smem();  // Wbar and scaled-T tiles written by generic stores -> MMA operands
    cta_sync_tc();

    // ---- phase 1b: Wbar K^T | dk += diag(beta gam) T^T Wbar | K K^T
    if (prod) {
        ok = tc::mbar_wait(&barKQ, pit, &g_err_bwdtc) && ok;
        tc::mma_tile(tb + kS1, tW, tK, C, C, Dk, false);
        tc::mma_tile(tb + kAK, tc::panel_tile(sm + L.Tsc, C, false), tWmn, C, Dk, C, true);
        tc::mma_commit(&bar);
    } else if (prod2) {
        ok = tc::mbar_wait(&barKQ, pit, &g_err_bwdtc) && ok;
        tc::mma_tile(tb + kS2, tK, tK, C, C, Dk, false);
        tc::mma_commit(&bar);
    }
    float gCb = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) gCb += red[w];
    float* Gkk = reinterpret_cast<float*>(sm + L.Gkk);
    float* Gqk = reinterpret_cast<float*>(sm + L.Gqk);
    float* ZP = Gqk;  // T o (Wbar K^T), until Gqk is formed in phase 2
    sync_after_mma(&bar, phase, ok, epi);
    if (epi && ok) {
        acc_rows2(tb, kS2, C, [&](int r, int c0, const float (&x)[16]) {
            float m[16];
#pragma unroll
            for (int i = 0; i < 16; i += 8) ld_row8(rkv + c0 + i, m + i);
#pragma unroll
            for (int i = 0; i < 16; ++i) m[i] = rkv[r] * m[i] * x[i];
            st_row8(Gkk + r * LDM + c0, m);
            st_row8(Gkk + r * LDM + c0 + 8, m + 8);
        });
        acc_rows2(tb, kS1, C, [&](int r, int c0, const float (&x)[16]) {
            float tt[16];
            ld_bf16x8(sm + L.Tt + tc::panel_off(c0, r, C), tt);
            ld_bf16x8(sm + L.Tt + tc::panel_off(c0 + 8, r, C), tt + 8);
            float tb16[16], zp[16];
            ld_row8(Tbf + r * LDM + c0, tb16);
            ld_row8(Tbf + r * LDM + c0 + 8, tb16 + 8);
            float cb[16], cg[16], ck[16];
#pragma unroll
            for (int i = 0; i < 16; i += 8) {
                ld_row8(bt + c0 + i, cb + i);
                ld_row8(gm + c0 + i, cg + i);
                ld_row8(rkv + c0 + i, ck + i);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                tb16[i] += cb[i] * cg[i] * ck[i] * x[i];
                zp[i] = tt[i] * x[i];
            }
            st_row8(Tbf + r * LDM + c0, tb16);
            st_row8(Tbf + r * LDM + c0 + 8, tb16 + 8);
            st_row8(ZP + r * LDM + c0, zp);
            st_row8(ZP + r * LDM + c0 + 8, zp + 8);
        });
    }
    __syncthreads();
    if (epi) {  // <Z_i, k_i> = sum_m T_mi (Wbar K^T)_mi, Z = T^T Wbar: four 16-row partials
        const int i = tid & (C - 1), qd = tid >> 6;
        float z = 0.f;
#pragma unroll 4
        for (int m = 16 * qd; m < 16 * qd + 16; ++m) z += ZP[m * LDM + i];
        csp[qd * C + i] = z;  // scratch until the column sums of phase 2
    }
    __syncthreads();
    if (tid < C) zk[tid] = (csp[tid] + csp[C + tid]) + (csp[2 * C + tid] + csp[3 * C + tid]);
    __syncthreads();
    if (tid < C) {
        const int i = tid;
        const float z = rkv[i] * zk[i];  // <Z_i, k_hat_i>
        betab[i] = bb0[i] + bb0[C + i] + gm[i] * z;
        gq[i] = rqv[i] * (gq[i] + gq[C + i]) + bt[i] * z * gm[i];  // gambar * gam
        ee[i] = rkv[i] * (ee[i] + ee[C + i]);                      // ebar * e
    }
    // Tbar as a bf16 operand (x = j, y = i)
    for (int e = tid; e < C * (C / 8); e += blockDim.x) {
        const int i = e / (C / 8), j0 = (e % (C / 8)) * 8;
        float t8[8];
        ld_row8(Tbf + i * LDM + j0, t8);
        st_bf16x8(sm + L.Tbh + canon(j0, i, C), t8);
    }
    tc::fence_async_smem();
    cta_sync_tc();

    // ---- phase 2: X = Tbar T^T | Q K^T, then Abar' = T^T X (Abar = -Abar')
    if (prod) {
        tc::mma_tile(tb + kS1, kmaj(sm, L.Tbh, C), tTt, C, C, C, false);
        tc::mma_commit(&bar);
    } else if (prod2) {
        tc::mma_tile(tb + kS2, tQ, tK, C, C, Dk, false);
        tc::mma_commit(&bar);
    }
    sync_after_mma(&bar, phase, ok, epi);
    if (epi && ok) {
        acc_rows2(tb, kS1, C, [&](int r, int c0, const float (&x)[16]) {
            tile_put16(sm + L.Xh, C, c0, r, x);  // X row-major (x = l, y = j)
        });
        acc_rows2(tb, kS2, C, [&](int r, int c0, const float (&x)[16]) {
            float m[16];
#pragma unroll
            for (int i = 0; i < 16; i += 8) ld_row8(rkv + c0 + i, m + i);
#pragma unroll
            for (int i = 0; i < 16; ++i) m[i] = rqv[r] * m[i] * x[i];
            st_row8(Gqk + r * LDM + c0, m);
            st_row8(Gqk + r * LDM + c0 + 8, m + 8);
        });
    }
    tc::fence_async_smem();
    cta_sync_tc();
    if (prod) {
        tc::mma_tile(tb + kS1, tTmn, mnmaj(sm, L.Xh, C), C, C, C, false);
        tc::mma_commit(&bar);
    } else if (prod2) {
        tc::mbar_arrive(&bar);  // nothing to issue in this round
    }
    sync_after_mma(&bar, phase, ok, epi);
    if (epi && ok) {
        // element-wise: M, Abar, Mbar o M (in place of Gkk), Gb (in place of Gqk),
        // Pbar o M scaled by r_k (columns) and by r_q (rows) as bf16 operands;
        // every lane takes 8 columns of a row
        acc_rows_all(tb, kS1, C, [&](int r, int c0, const float (&x)[8], int hl) {
            const int pi = 2 * g + hl;
            float sb = 0.f;
            float rs = rsp[pi * C + r], rc = rsc[pi * C + r];  // Kahan-compensated row sum
            float pk[8], pq[8], mv[8];
            // the column block of the piece and the row block of the warp are
            // warp-uniform, so is the choice between factored and direct decay
            const int J = c0 >> 4, I = r >> 4;
            if (J < I) {
                const float u = uf[J * C + r];
                ld_row8(wf + J * C + c0, mv);
#pragma unroll
                for (int i = 0; i < 8; ++i) mv[i] *= u;
            } else if (J == I) {
                const float ghr = Ghi[r], glr = Glo[r];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int jj = c0 + i;
                    mv[i] = jj <= r ? expf((ghr - Ghi[jj]) + (glr - Glo[jj])) : 0.f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) mv[i] = 0.f;
            }
            float gk8[8], pf8[8], gq8[8], kc8[8];
            ld_row8(rkv + c0, kc8);
            ld_row8(Gkk + r * LDM + c0, gk8);
            ld_row8(Pf + r * LDM + c0, pf8);
            ld_row8(Gqk + r * LDM + c0, gq8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int jj = c0 + i;
                const float m = mv[i];
                const float ab = jj < r ? -x[i] : 0.f;
                const float gk = gk8[i];
                const float mb = ab * bt[r] * gk + pf8[i] * gq8[i];
                sb = fmaf(ab * m, gk, sb);
                const float mm = mb * m;
                gk8[i] = mm;
                gq8[i] = ab * bt[r] * m;
                const float yk = mm - rc;
                const float tk = rs + yk;
                rc = (tk - rs) - yk;
                rs = tk;
                const float pm = pf8[i] * m;
                pk[i] = pm * kc8[i];
                pq[i] = pm * rqv[r];
            }
            st_row8(Gkk + r * LDM + c0, gk8);
            st_row8(Gqk + r * LDM + c0, gq8);
            st_bf16x8(sm + L.PMk + canon(c0, r, C), pk);
            st_bf16x8(sm + L.PMq + canon(c0, r, C), pq);
            sbp[pi * C + r] += sb;  // two 8-column pieces per lane
            rsp[pi * C + r] = rs;
            rsc[pi * C + r] = rc;
        });
    }
    __syncthreads();
    // H = (Gb + Gb^T) diag(r_k) as a bf16 operand; column sums of Mbar o M (fp64)
    for (int e = tid; e < C * (C / 8); e += blockDim.x) {
        // lanes take consecutive rows i: the row-wise float4 reads and the
        // transposed column reads both stay conflict-free
        const int i = e % C, j0 = (e / C) * 8;
        float h8[8];
        ld_row8(Gqk + i * LDM + j0, h8);
#pragma unroll
        for (int s = 0; s < 8; ++s) h8[s] = (h8[s] + Gqk[(j0 + s) * LDM + i]) * rkv[j0 + s];
        st_bf16x8(sm + L.Hk + canon(j0, i, C), h8);
    }
    if (epi) {
        const int i = tid & (C - 1), qd = tid >> 6;
        float cs = 0.f, cc = 0.f;  // Kahan-compensated column sum
#pragma unroll 4
        for (int kk = 16 * qd; kk < 16 * qd + 16; ++kk) {
            const float yk = Gkk[kk * LDM + i] - cc;
            const float tk = cs + yk;
            cc = (tk - cs) - yk;
            cs = tk;
        }
        csp[qd * C + i] = cs - cc;
    }
    tc::fence_async_smem();
    cta_sync_tc();

    // ---- phase 3: dq += (Pbar o M) K;  dk += (Pbar o M)^T Q + (Gb + Gb^T) K
    if (prod) {
        tc::mma_tile(tb + kAQ, kmaj(sm, L.PMk, C), tKmn, C, Dk, C, true);
        tc::mma_commit(&bar);
        tc::mma_commit(&barAQ);
    } else if (prod2) {
        tc::mma_tile(tb + kAK, mnmaj(sm, L.PMq, C), tQmn, C, Dk, C, true);
        tc::mma_tile(tb + kAK, kmaj(sm, L.Hk, C), tKmn, C, Dk, C, true);
        tc::mma_commit(&bar);
    }
    // Gammabar_i = sum_j (Mbar o M)_ij - sum_k (Mbar o M)_ki + gambar_i gam_i - ebar_i e_i,
    // plus the chunk-end terms at i = 63; the log-decay cotangent is its reverse
    // cumulative sum (one warp, two-float sums, two steps per lane)
    if (tid < C) {
        const int i = tid;
        betab[i] += sbp[i] + sbp[C + i] + sbp[2 * C + i] + sbp[3 * C + i];
        f2 gb{0.f, 0.f};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            gb = f2_add(gb, f2{rsp[q4 * C + i], -rsc[q4 * C + i]});
            gb = f2_add(gb, f2{-csp[q4 * C + i], 0.f});
        }
        gb = f2_add(gb, f2{gq[i], 0.f});
        gb = f2_add(gb, f2{-ee[i], 0.f});
        gbh[i] = gb.hi;
        gbl[i] = gb.lo;
    }
    __syncthreads();
    if (warp == 0) {
        // chunk-end terms at i = 63: <S, Sbar'> gam_63 + sum_j ebar_j e_j
        f2 se = f2_add(f2{ee[2 * lane], 0.f}, f2{ee[2 * lane + 1], 0.f});
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            se = f2_add(se, f2{__shfl_xor_sync(0xffffffffu, se.hi, off), __shfl_xor_sync(0xffffffffu, se.lo, off)});
        const f2 x0{gbh[2 * lane], gbl[2 * lane]};
        f2 x1{gbh[2 * lane + 1], gbl[2 * lane + 1]};
        if (lane == 31) x1 = f2_add(f2_add(x1, two_sum(gCb * gm[C - 1], 0.f)), se);
        // suffix sums: element i gets sum_{k >= i}
        const f2 tot = f2_add(x0, x1);
        f2 suf = tot;  // inclusive suffix over lanes >= lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            // every lane adds (zero past the last lane: the sum is unchanged, and no
            // lane branches between the shuffles)
            const float yh = __shfl_down_sync(0xffffffffu, suf.hi, off);
            const float yl = __shfl_down_sync(0xffffffffu, suf.lo, off);
            const bool in = lane + off < 32;
            suf = f2_add(suf, f2{in ? yh : 0.f, in ? yl : 0.f});
        }
        const f2 after = f2_add(suf, f2{-tot.hi, -tot.lo});  // lanes > lane
        const f2 d1 = f2_add(x1, after);
        const f2 d0 = f2_add(x0, d1);
        p.dl[gbase + 2 * lane + 1] = d1.hi + d1.lo;
        p.dl[gbase + 2 * lane] = d0.hi + d0.lo;
        p.dbeta[gbase + 2 * lane] = betab[2 * lane];
        p.dbeta[gbase + 2 * lane + 1] = betab[2 * lane + 1];
    }
    // dq is complete once the producer's phase-3 chain is: its partials go out
    // while the second issuer's dk products still run
    const int64_t prow = d.Hv * Dk;  // partials [B, Tp, Hv, Dk]: elements from one step's rows to the next
    const int64_t pbase = (((int64_t)bb * d.Tp + t0) * d.Hv + h) * Dk;
    if (epi) {
        ok = tc::mbar_wait(&barAQ, ip, &g_err_bwdtc) && ok;
        tc::tc_fence_after();
        if (ok) {
            uint8_t* dqh = reinterpret_cast<uint8_t*>(p.dqh) + pbase * 2;
            acc_rows2(tb, kAQ, Dk, [&](int r, int c0, const float (&x)[16]) {
                st_bf16x8(dqh + ((int64_t)r * prow + c0) * 2, x);
                st_bf16x8(dqh + ((int64_t)r * prow + c0 + 8) * 2, x + 8);
            });
        }
    }
    // the producer waits too: once the phase-3 products are done, every operand
    // tile of this item is dead and the next item's loads go out, under the
    // final stores below
    sync_after_mma(&bar, phase, ok, epi || prod);
    if (prod) {
        const int next = (int)atomicAdd(sched, 1u);
        next_item = next;
        if (ok && next < nitems) {
            ok = wait_ready(next);
            if (ok) {
                issue_loads(next);
                pending = true;
                pend_pit = pit ^ 1u;
            }
        }
    }
    if (epi && ok) {
        // per-value-head partials as bf16 [B, Tp, Hv, Dk] (summed over the group
        // and normalised in fp32; a group's rows of one step are then contiguous
        // for the reduction)
        uint8_t* dkh = reinterpret_cast<uint8_t*>(p.dkh) + pbase * 2;
        acc_rows2(tb, kAK, Dk, [&](int r, int c0, const float (&x)[16]) {
            st_bf16x8(dkh + ((int64_t)r * prow + c0) * 2, x);
            st_bf16x8(dkh + ((int64_t)r * prow + c0 + 8) * 2, x + 8);
        });
    }
    tc::tc_fence_before();
    const int failed = __syncthreads_or(!ok);  // a bounded wait gave up: stop here
    tc::tc_fence_after();
    if (failed) break;
    }  // items
    if (prod && pending) {
        // only after a failed wait: the copies of an item that will not run land
        // before the CTA exits (each wait bounded)
        tc::mbar_wait(&barOV, pend_pit, &g_err_bwdtc);
        tc::mbar_wait(&barL, pend_pit, &g_err_bwdtc);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

__global__ void __launch_bounds__(kThreads + 64, 1)
    bwd_chunk_tc_kernel(Dims d, Ptrs p, const __grid_constant__ Tmaps tm) {
    bwd_chunk_body(d, p, tm, p.sched, nullptr, 0);
}

// The reverse scan and the per-chunk gradients in one cooperative launch (one
// CTA per SM, all resident at once).  CTAs [0, nscan) first run the reverse scan
// of one value tile each, publishing every finished chunk; then every CTA takes
// gradient items, each once the reverse scan has published its chunk for all
// value tiles of its head.  The scan CTAs never wait on the gradient CTAs, so
// every wait ends; the SMs the scan leaves idle run gradient items meanwhile.
__global__ void __launch_bounds__(kThreads + 64, 1)
    bwd_fused_tc_kernel(Dims d, Ptrs p, const __grid_constant__ Tmaps tm) {
    const int ntiles = (int)(d.Dv / ta::DVT);
    const int nscan = ntiles * (int)(d.Hv * d.B);
    unsigned int* progress = p.sched + 1;
    const int t = (int)blockIdx.x;
    if (t < nscan) {
        const ScanSeg whole{1, (int)d.NC, 0, nullptr, nullptr};
        ta::bwd_scan_ta_body<false>(d, p, tm, t % ntiles, (t / ntiles) % (int)d.Hv, t / (ntiles * (int)d.Hv),
                             whole, 0, &g_err_bwdtc, progress, false);
        __syncthreads();
    }
    bwd_chunk_body(d, p, tm, p.sched, progress, ntiles);
}

size_t fused_smem(const Dims& d) {
    const uint32_t a = smem_plan((int)d.Dk, (int)d.Dv).total, b = ta::tb_plan((int)d.Dk).total;
    return (size_t)(a > b ? a : b) + 1024;  // slack for the 1024-byte alignment of the base
}

}  // namespace

bool bwd_chunk_tc_supported(const Dims& d) {
    if (d.dtype != 1) return false;
    // TMEM: scratch 64 + dk and dq accumulators 2 Dk + scratch 64 <= 512
    if (d.Dk % 32 || d.Dv % 32 || d.Dk > 192 || d.Dv > 256) return false;
    // the third Dk block of Sbar' sits in the Wbar tile ahead of that block's Wbar
    if (d.Dk > 128 && (d.Dk - 128) * d.Dv * 2 > 16 * C * 16) return false;
    return smem_plan((int)d.Dk, (int)d.Dv).total + 2048 <= 227u * 1024u;
}

cudaError_t launch_bwd_chunk_tc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const Smem L = smem_plan((int)d.Dk, (int)d.Dv);
    const size_t smem = L.total + 1024;  // slack for the 1024-byte alignment of the base
    auto kern = bwd_chunk_tc_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (the shared memory allows no second one)
    const int64_t nitems = d.NC * d.Hv * d.B;
    const int grid = (int)(nitems < sm_count() ? nitems : sm_count());
    e = cudaMemsetAsync(p.sched, 0, sizeof(unsigned int), s);  // the item counter
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads + 64, smem, s>>>(d, p, *p.tmaps);
    count_launches(1);
    return cudaPeekAtLastError();
}

bool bwd_fused_tc_supported(const Dims& d) {
    if (!bwd_chunk_tc_supported(d) || !scan_ta_supported(d)) return false;
    if (fused_smem(d) + 1024 > 227u * 1024u) return false;
    // the reverse scan's CTAs leave SMs to the gradient items from the start
    const int64_t nscan = (d.Dv / ta::DVT) * d.Hv * d.B;
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return false;
    return nscan + 8 <= sm_count();
}

cudaError_t launch_bwd_fused_tc(const Dims& d, const Ptrs& p, cudaStream_t s) {
    const size_t smem = fused_smem(d);
    auto kern = bwd_fused_tc_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads + 64, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    // the item counter and the per-(b, h) progress counts start at zero
    e = cudaMemsetAsync(p.sched, 0, (size_t)(1 + d.B * d.Hv) * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    Dims dd = d;
    Ptrs pp = p;
    Tmaps tm = *p.tmaps;
    void* args[] = {&dd, &pp, &tm};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)sm_count()),
                                    dim3(kThreads + 64), args, smem, s);
    count_launches(1);
    return e;
}

}  // namespace gdn
