// gdn_tc.cuh -- sm_100-family tensor-core primitives (tcgen05, TMEM, mbarrier,
// bulk/tensor TMA) written as inline PTX, used by the bf16 kernels.
//
// Shared-memory operand layout ("canonical, no swizzle"): a tile is stored
// as 8 x 16-byte core matrices.  For a tile indexed (x, y) where x is the
// dimension whose 8 consecutive elements share one 16-byte row of a core
// matrix and y the other dimension:
//     byte(x, y) = (x / 8) * XS + (y / 8) * YS + (y % 8) * 16 + (x % 8) * 2
// A K-major operand has x = K (then LBO = XS, SBO = YS); an MN-major operand
// has x = M or N (then SBO = XS, LBO = YS).  One bf16 MMA consumes K = 16,
// i.e. two core matrices along K: the next K step starts 2 * LBO further.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc {

// Error word bit set when a bounded wait gives up (kernels never trap).  Each
// translation unit that waits owns one word (GDN_ERROR_WORD) and a host
// accessor that reads and clears it.
constexpr unsigned int kErrWaitTimeout = 1u;

#define GDN_ERROR_WORD(tu)                                                       \
    static __device__ unsigned int g_err_##tu = 0;                                \
    unsigned int read_clear_error_##tu() {                                       \
        unsigned int v = 0, z = 0;                                               \
        if (cudaMemcpyFromSymbol(&v, g_err_##tu, sizeof(v)) != cudaSuccess) return ~0u; \
        cudaMemcpyToSymbol(g_err_##tu, &z, sizeof(z));                           \
        return v;                                                                \
    }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete is
// suspended until the phase completes or hint_ns pass, instead of returning at
// once and spinning
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t kWaitSleepNs = 10000;  // suspend-time hint of one try_wait
// Every wait on another agent gives up after this much wall time.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

// Bounded wait on an mbarrier phase.  On timeout it records kErrWaitTimeout in
// *err and returns false; callers then skip work.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned int* err,
                                              uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err) {
    return mbar_wait_for(bar, parity, err, kWaitLimitNs);
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// ---- proxy / ordering fences ----------------------------------------------------
// generic-proxy shared-memory writes -> visible to the async proxy (tcgen05.mma, TMA)
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- TMEM ----------------------------------------------------------------------
// executed by one full warp; writes the TMEM base address to *dst (shared)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// TMEM address of (lane, column)
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// 32 lanes x 32 bits, 16 consecutive columns per thread (thread t <-> lane base + t)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 16 lanes x 32 bits in two column halves (shape 16x32bx2): thread t < 16 reads
// lane base + t at columns col .. col + 15, thread t >= 16 reads lane
// base + t - 16 at columns col + OFF .. col + OFF + 15.  The rows of an M = 64
// accumulator sit in the first 16 lanes of each warp's 32, so this shape keeps
// every thread of the warp on accumulator data.
template <int OFF>
__device__ __forceinline__ void tmem_ld16x2(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16], %17;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr), "n"(OFF));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// the store of the same shape: thread t < 16 writes lane base + t, columns
// col .. col + 15; thread t >= 16 lane base + t - 16, columns col + OFF ..
template <int OFF>
__device__ __forceinline__ void tmem_st16x2(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, "
        "{%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17};" ::"r"(taddr),
        "n"(OFF), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns per thread
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- 16-byte asynchronous global -> shared copies (zero-filled when src_bytes = 0)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---- bulk (non-tensor) asynchronous copies through the async proxy ------------------
// Addresses 16-byte aligned, size a multiple of 16.  global -> shared completes
// `bytes` of transaction count on *bar (the issuer arms it with arrive_expect_tx);
// shared -> global is tracked in the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... all but the most recent committed group
__device__ __forceinline__ void bulk_wait_read_but1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// load with acquire semantics at GPU scope (pairs with a release by another CTA)
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Bounded poll until the global word *f (written by other CTAs with release
// semantics) reaches `need`; acquire ordering on success.  On timeout it
// records kErrWaitTimeout in *err and returns false.
__device__ __forceinline__ bool poll_geq(const unsigned int* f, unsigned int need, unsigned int* err,
                                         uint64_t limit_ns) {
    if (ld_acquire_gpu(f) >= need) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; ld_acquire_gpu(f) < need; ++i) {
        __nanosleep(64);
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
    return true;
}
// ... all but the most recent committed group
__device__ __forceinline__ void bulk_wait_but1() { asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); }
// global-memory accesses of the generic proxy (an acquire that saw another CTA's
// release) ordered before this thread's later bulk / tensor copies
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- tensor (TMA) loads -----------------------------------------------------------
// 5-d tiled load of the box at coordinates c0..c4 of the tensor map `map` (the
// address of a __grid_constant__ kernel parameter) into shared memory; the box
// bytes complete on *bar (armed by the issuer with arrive_expect_tx)
__device__ __forceinline__ void tma_load_5d(void* dst, const void* map, int c0, int c1, int c2,
                                            int c3, int c4, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(smem_u32(bar))
        : "memory");
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned global
// address: no shared memory, no completion to wait for
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-d tiled load (coordinates c0 = innermost, c1) into shared memory
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
// 3-d tiled store of a box from shared memory to the tensor map's tensor at
// coordinates c0..c2 (all non-negative; elements past the tensor's extent are
// not written), tracked in this thread's bulk groups
__device__ __forceinline__ void tma_store_3d(const void* map, const void* src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}

// 2-d tiled store of a box from shared memory at coordinates c0 (innermost), c1
// (non-negative), tracked in this thread's bulk groups
__device__ __forceinline__ void tma_store_2d(const void* map, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

// ---- descriptors -------------------------------------------------------------------
// shared-memory matrix descriptor, no swizzle, sm_100 version field = 1
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}
// instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulator
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], one thread issues
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]: A (M x K, bf16) held in TMEM, row m in the
// accumulator's lane for row m, K elements packed two per 32-bit column
// (element 2i in the low half of column i)
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on *bar once every MMA issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Operand tile geometry in the canonical layout above.
struct Tile {
    uint32_t base;  // shared address of the tile
    uint32_t xs;    // byte stride between 8-element groups along x
    uint32_t ys;    // byte stride between 8-row groups along y
    bool k_major;   // x is the K dimension
    __device__ __forceinline__ uint32_t off(uint32_t x, uint32_t y) const {
        return (x >> 3) * xs + (y >> 3) * ys + (y & 7u) * 16u + (x & 7u) * 2u;
    }
    // descriptor for the K slice starting at k0 (multiple of 16)
    __device__ __forceinline__ uint64_t desc(uint32_t k0) const {
        if (k_major) return sdesc(base + (k0 >> 3) * xs, xs, ys);
        return sdesc(base + (k0 >> 3) * ys, ys, xs);
    }
    // desc(k0 + 16) - desc(k0): the next K slice moves only the start-address
    // field (addresses below 256 KB never carry into the next field).  Issuing
    // loops add it instead of rebuilding the descriptor, which keeps the single
    // issuing thread from becoming the bottleneck of small MMAs.
    __device__ __forceinline__ uint64_t desc_step() const {
        return (uint64_t)((2u * (k_major ? xs : ys)) >> 4);
    }
};

// "Panel" image of a bf16 operand with `rows` rows (y) and 8-column groups (x):
// the canonical layout with XS = rows * 16 and YS = 128, so every 8-column group
// is one contiguous panel of rows x 16 bytes and a run of groups is one block.
// Saved intermediates are stored in global memory in this form and moved with a
// single bulk copy.
__host__ __device__ __forceinline__ uint32_t panel_off(uint32_t x, uint32_t y, uint32_t rows) {
    return (x >> 3) * rows * 16u + y * 16u + (x & 7u) * 2u;
}
__device__ __forceinline__ Tile panel_tile(const void* smem, uint32_t rows, bool k_major) {
    Tile t;
    t.base = smem_u32(smem);
    t.xs = rows * 16u;
    t.ys = 128u;
    t.k_major = k_major;
    return t;
}

// issue D = A (M x K) * B (K x N) (+ D if accumulate) as K / 16 MMAs
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, const Tile& A, const Tile& B, int M,
                                         int N, int K, bool accumulate) {
    const uint32_t id = idesc_bf16(M, N, !A.k_major, !B.k_major);
    uint64_t da = A.desc(0), db = B.desc(0);
    const uint64_t ia = A.desc_step(), ib = B.desc_step();
    for (int k = 0; k < K; k += 16) {
        mma_bf16(d_tmem, da, db, id, (accumulate || k > 0) ? 1u : 0u);
        da += ia;
        db += ib;
    }
}

// issue D = A (M x K, in TMEM at column a_col) * B (K x N) (+ D) as K / 16 MMAs
__device__ __forceinline__ void mma_tile_ta(uint32_t d_tmem, uint32_t a_tmem, const Tile& B, int M,
                                            int N, int K, bool accumulate) {
    const uint32_t id = idesc_bf16(M, N, false, !B.k_major);
    uint64_t db = B.desc(0);
    const uint64_t ib = B.desc_step();
    for (int k = 0; k < K; k += 16) {
        mma_bf16_ta(d_tmem, a_tmem + (uint32_t)(k >> 1), db, id, (accumulate || k > 0) ? 1u : 0u);
        db += ib;
    }
}
// 32 lanes x 32 bits, 16 consecutive columns per thread, raw 32-bit words
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
// 32 lanes x 32 bits, 8 consecutive columns per thread, raw 32-bit words v[0 .. 7]
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}
// One arrival on `bar` for the calling warp, once every lane's tcgen05.st have
// completed (each lane has executed tcgen05.wait::st): the waiter may then
// issue MMAs that read those TMEM columns.
__device__ __forceinline__ void warp_arrive_after_st(uint64_t* bar) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
// named barrier `id` (1 .. 15) over `count` threads of the CTA, a multiple of 32
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void tmem_ld16u(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// two floats -> packed bf16 pair (x in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace tc
}  // namespace gdn
