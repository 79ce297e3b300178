// gdn_selftest.cu -- plain matrix product through the library's tcgen05 path
// (staging into the canonical shared-memory layout, MMA issue, TMEM read-back).
#include "../../include/gdn_selftest.h"
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

GDN_ERROR_WORD(selftest)

namespace {

__global__ void __launch_bounds__(128) selftest_mma_kernel(int M, int N, int K, int a_mn, int b_mn,
                                                           const __nv_bfloat16* __restrict__ A,
                                                           const __nv_bfloat16* __restrict__ B,
                                                           float* __restrict__ D, int rows16x2) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    uint8_t* sa = smem;                 // A tile: up to 128 x 256 bf16 = 64 KB
    uint8_t* sb = smem + 128 * 256 * 2; // B tile: up to 256 x 256 bf16 = 128 KB
    const int tid = threadIdx.x, warp = tid >> 5;
    // A: K-major -> x = k, y = m; MN-major -> x = m, y = k.  x groups fastest.
    tc::Tile ta, tb;
    ta.base = tc::smem_u32(sa);
    ta.k_major = !a_mn;
    const int ax = a_mn ? M : K;
    ta.xs = 128;
    ta.ys = (uint32_t)(ax / 8) * 128;
    tb.base = tc::smem_u32(sb);
    tb.k_major = !b_mn;
    const int bx = b_mn ? N : K;
    tb.xs = 128;
    tb.ys = (uint32_t)(bx / 8) * 128;
    for (int e = tid; e < M * K; e += blockDim.x) {
        const int m = e / K, k = e % K;
        const uint32_t o = a_mn ? ta.off(m, k) : ta.off(k, m);
        *reinterpret_cast<__nv_bfloat16*>(sa + o) = A[e];
    }
    for (int e = tid; e < K * N; e += blockDim.x) {
        const int k = e / N, n = e % N;
        const uint32_t o = b_mn ? tb.off(n, k) : tb.off(k, n);
        *reinterpret_cast<__nv_bfloat16*>(sb + o) = B[e];
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 256);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = tmem_base;
    if (tid == 0) {
        tc::mma_tile(tbase, ta, tb, M, N, K, false);
        tc::mma_commit(&bar);
    }
    const bool ok = tc::mbar_wait(&bar, 0, &g_err_selftest);
    tc::tc_fence_after();
    if (ok && !rows16x2) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tc::tmem_ld16(tc::tmem_addr(tbase, 32 * (warp & 3), c0), v);
            tc::tmem_wait_ld();
            const int row = 32 * (warp & 3) + (tid & 31);
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + c0 + i] = v[i];
        }
    } else if (ok) {
        // M = 64 rows through the 16x32bx2 shape: load, negate, store back with
        // the same shape, load again; D is [64][N] (row 16 (warp % 4) + lane % 16)
        const int l = tid & 31;
        const int row = 16 * (warp & 3) + (l & 15);
        for (int c0 = 0; c0 < N; c0 += 32) {
            const uint32_t ta = tc::tmem_addr(tbase, 32 * (warp & 3), c0);
            float v[16];
            tc::tmem_ld16x2<16>(ta, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = -v[i];
            tc::tmem_st16x2<16>(ta, v);
            tc::tmem_wait_st();
            tc::tmem_ld16x2<16>(ta, v);
            tc::tmem_wait_ld();
            const int col = c0 + 16 * (l >> 4);
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + col + i] = v[i];
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, 256);
}

// Same product with A held in TMEM (the form the scans use for the state):
// thread m writes row m of A as packed bf16 pairs into columns 256 .. 256 + K/2.
__global__ void __launch_bounds__(128) selftest_mma_ta_kernel(int N, int K, int b_mn,
                                                              const __nv_bfloat16* __restrict__ A,
                                                              const __nv_bfloat16* __restrict__ B,
                                                              float* __restrict__ D) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    uint8_t* sb = smem;
    const int tid = threadIdx.x, warp = tid >> 5;
    tc::Tile tb;
    tb.base = tc::smem_u32(sb);
    tb.k_major = !b_mn;
    const int bx = b_mn ? N : K;
    tb.xs = 128;
    tb.ys = (uint32_t)(bx / 8) * 128;
    for (int e = tid; e < K * N; e += blockDim.x) {
        const int k = e / N, n = e % N;
        const uint32_t o = b_mn ? tb.off(n, k) : tb.off(k, n);
        *reinterpret_cast<__nv_bfloat16*>(sb + o) = B[e];
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t acol = 256;
    for (int k0 = 0; k0 < K; k0 += 32) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k = k0 + 2 * i;
            const float x = k < K ? __bfloat162float(A[tid * K + k]) : 0.f;
            const float y = k + 1 < K ? __bfloat162float(A[tid * K + k + 1]) : 0.f;
            w[i] = tc::pack_bf16(x, y);
        }
        tc::tmem_st16u(tc::tmem_addr(tbase, 32 * warp, acol + k0 / 2), w);
    }
    tc::tmem_wait_st();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid == 0) {
        tc::mma_tile_ta(tbase, tbase + acol, tb, 128, N, K, false);
        tc::mma_commit(&bar);
    }
    const bool ok = tc::mbar_wait(&bar, 0, &g_err_selftest);
    tc::tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tc::tmem_ld16(tc::tmem_addr(tbase, 32 * warp, c0), v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) D[tid * N + c0 + i] = v[i];
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

// One TMA tile load through a row-tile tensor map, copied back verbatim.
__global__ void __launch_bounds__(128) selftest_tma_kernel(const __grid_constant__ CUtensorMap map,
                                                           int b, int t0, int h, int xg0, int cols,
                                                           uint8_t* __restrict__ out) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    const int tid = threadIdx.x;
    const uint32_t bytes = (uint32_t)(kChunk * cols * 2);
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(&bar, bytes);
        tc::tma_load_5d(smem, &map, 0, t0, xg0, h, b, &bar);
    }
    const bool ok = tc::mbar_wait(&bar, 0, &g_err_selftest);
    if (ok)
        for (uint32_t e = tid; e < bytes / 16; e += blockDim.x)
            reinterpret_cast<uint4*>(out)[e] = reinterpret_cast<const uint4*>(smem)[e];
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_selftest_mma(int M, int N, int K, int a_mn_major, int b_mn_major,
                                       const void* A, const void* B, float* D_raw, void* stream) {
    if (!(M == 64 || M == 128) || N < 16 || N > 256 || N % 16 || K < 16 || K > 256 || K % 16)
        return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!A || !B || !D_raw) return GDN_ERR_INVALID_ARG;
    const size_t smem = (size_t)128 * 256 * 2 + (size_t)256 * 256 * 2;
    auto kern = gdn::selftest_mma_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        M, N, K, a_mn_major, b_mn_major, static_cast<const __nv_bfloat16*>(A),
        static_cast<const __nv_bfloat16*>(B), D_raw, 0);
    gdn::count_launches(1);
    return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_selftest_mma_m64_rows(int N, int K, const void* A, const void* B,
                                                float* D, void* stream) {
    if (N < 32 || N > 256 || N % 32 || K < 16 || K > 256 || K % 16) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!A || !B || !D) return GDN_ERR_INVALID_ARG;
    const size_t smem = (size_t)128 * 256 * 2 + (size_t)256 * 256 * 2;
    auto kern = gdn::selftest_mma_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        64, N, K, 0, 0, static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D, 1);
    gdn::count_launches(1);
    return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_selftest_mma_tmem_a(int N, int K, int b_mn_major, const void* A,
                                              const void* B, float* D, void* stream) {
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 256 || K % 32) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!A || !B || !D) return GDN_ERR_INVALID_ARG;
    const size_t smem = (size_t)256 * 256 * 2;
    auto kern = gdn::selftest_mma_ta_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        N, K, b_mn_major, static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D);
    gdn::count_launches(1);
    return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_selftest_tma_tile(int64_t B, int64_t T, int64_t H, int64_t D, int cols,
                                            int b, int t0, int h, int xg0, const void* src,
                                            void* out, void* stream) {
    if (!src || !out) return GDN_ERR_INVALID_ARG;
    if (cols % 8 || cols < 8 || cols > 256 || D % 8 || xg0 < 0 || xg0 * 8 + cols > D)
        return GDN_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap m;
    if (!gdn::encode_row_tile_map(&m, src, B, T, H, D, cols)) return GDN_ERR_CUDA;
    const size_t smem = (size_t)gdn::kChunk * cols * 2;
    auto kern = gdn::selftest_tma_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(m, b, t0, h, xg0, cols,
                                                              static_cast<uint8_t*>(out));
    gdn::count_launches(1);
    return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

namespace gdn {
namespace {

// A bounded wait that nobody ends: the CTA takes TMEM as the tensor-core
// kernels do, then waits for an mbarrier phase no thread completes (mode 0)
// or for a global word the host left below 1 (mode 1, the form of the fused
// backward's progress poll), with a limit of limit_ns.  On timeout the wait
// sets the error word; the CTA then frees its TMEM, records out[0] = 1 if the
// wait succeeded (0 if it gave up) and out[1] = 1 once the TMEM is freed, and
// returns.
__global__ void __launch_bounds__(128) selftest_wait_timeout_kernel(int mode, uint64_t limit_ns,
                                                                    const unsigned int* word,
                                                                    unsigned int* out) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int waited;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 32);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);  // one arrival expected; none comes
        tc::fence_mbar_init();
        waited = 1;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = tmem_base;
    bool ok = true;
    if (mode == 0) {
        ok = tc::mbar_wait_for(&bar, 0, &g_err_selftest, limit_ns);
    } else if (tid == 0) {
        ok = tc::poll_geq(word, 1u, &g_err_selftest, limit_ns);
    }
    if (!ok) waited = 0;  // benign: every writer stores 0
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tmem_dealloc(tbase, 32);
        if (tid == 0) {
            out[0] = (unsigned int)waited;
            __threadfence();
            out[1] = 1u;
        }
    }
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_selftest_wait_timeout(int mode, uint64_t limit_ns,
                                                const unsigned int* word, unsigned int* out,
                                                void* stream) {
    if (!out || (mode == 1 && !word)) return GDN_ERR_INVALID_ARG;
    if ((mode != 0 && mode != 1) || limit_ns < 1000ull || limit_ns > gdn::tc::kWaitLimitNs)
        return GDN_ERR_INVALID_ARG;
    gdn::selftest_wait_timeout_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        mode, limit_ns, word, out);
    gdn::count_launches(1);
    return cudaPeekAtLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_device_error(unsigned int* flag) {
    if (!flag) return GDN_ERR_INVALID_ARG;
    const unsigned int v = gdn::read_clear_error_all();
    if (v == ~0u) return GDN_ERR_CUDA;
    *flag = v;
    return GDN_OK;
}
