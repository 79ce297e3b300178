/*
 * gdn_selftest.h -- hardware self-check of the tensor-core path of libgdn.so.
 *
 * Not an operation of the method (the pages have no counterpart): it runs the
 * library's own shared-memory staging, tcgen05 MMA issue and TMEM read-back on
 * a plain matrix product so that tests can check operand layouts and
 * accumulator lane placement against a reference product.
 */
#ifndef GDN_SELFTEST_H
#define GDN_SELFTEST_H

#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* D_raw = A * B on one CTA with tcgen05.mma (bf16 in, fp32 accumulate).
 *   A: device bf16 [M][K] row-major, B: device bf16 [K][N] row-major.
 *   M in {64, 128}; N in 16..256 (multiple of 16); K in 16..256 (multiple of 16).
 *   a_mn_major / b_mn_major choose the shared-memory operand orientation.
 *   D_raw: device fp32 [128][N]: every TMEM lane (row) of the accumulator as read
 *   back by 32x32b loads, so the lane placement of M = 64 results is visible.
 * Enqueued on `stream`; returns GDN_ERR_UNSUPPORTED_SHAPE for other sizes. */
gdn_status gdn_selftest_mma(int M, int N, int K, int a_mn_major, int b_mn_major, const void* A,
                            const void* B, float* D_raw, void* stream);

/* The rows of an M = 64 accumulator read through the 16x32bx2 TMEM shape (every
 * thread of a warp on accumulator data; the form the gradient kernel's
 * epilogues use): D = -(A * B) after one load, a negated store back with the
 * same shape and a second load.
 *   A: device bf16 [64][K] row-major, B: device bf16 [K][N] row-major, both
 *   staged K-major.  N in 32..256 (multiple of 32); K in 16..256 (multiple of 16).
 *   D: device fp32 [64][N].
 * Enqueued on `stream`; returns GDN_ERR_UNSUPPORTED_SHAPE for other sizes. */
gdn_status gdn_selftest_mma_m64_rows(int N, int K, const void* A, const void* B, float* D,
                                     void* stream);

/* D = A * B on one CTA with tcgen05.mma taking A from tensor memory (the form
 * the scans use for the state operand), M = 128.
 *   A: device bf16 [128][K] row-major, written by its 128 threads into TMEM
 *   (row m in lane m, two elements per 32-bit column); B: device bf16 [K][N]
 *   row-major, staged in shared memory in the orientation b_mn_major selects.
 *   N in 16..256 (multiple of 16); K in 32..256 (multiple of 32).
 *   D: device fp32 [128][N].
 * Enqueued on `stream`; returns GDN_ERR_UNSUPPORTED_SHAPE for other sizes. */
gdn_status gdn_selftest_mma_tmem_a(int N, int K, int b_mn_major, const void* A, const void* B,
                                   float* D, void* stream);

/* One 64-row tile of a bf16 [B][T][H][D] tensor loaded by TMA through the
 * library's row-tile tensor map (the path the scans and the gradient kernel use
 * for q, k, v and dO), copied back verbatim: out receives 64 * cols * 2 bytes in
 * the panel layout, byte (g * 64 + r) * 16 + 2 i = element (b, t0 + r, h,
 * 8 (xg0 + g) + i), zero where t0 + r >= T.  cols: multiple of 8 in 8..256.
 * Enqueued on `stream`. */
gdn_status gdn_selftest_tma_tile(int64_t B, int64_t T, int64_t H, int64_t D, int cols, int b,
                                 int t0, int h, int xg0, const void* src, void* out,
                                 void* stream);

/* Failure detection check: one CTA takes tensor memory as the tensor-core
 * kernels do, then waits on something nothing will complete, bounded by
 * limit_ns (1 us .. 1 s; the kernels use 1 s):
 *   mode 0: an mbarrier phase that no thread arrives at;
 *   mode 1: the device word *word reaching 1 (pass a word holding 0), polled
 *           with acquire loads as the fused backward polls its progress words.
 * When the wait gives up, the kernel sets the timeout bit (1) of the device
 * error word (read it with gdn_device_error), frees its tensor memory, writes
 * out[0] = 0 (1 had the wait succeeded) and then out[1] = 1, and returns; the
 * context stays usable.  out: device, 2 words.  Enqueued on `stream`; returns
 * GDN_ERR_INVALID_ARG for a bad mode, limit or pointer. */
gdn_status gdn_selftest_wait_timeout(int mode, uint64_t limit_ns, const unsigned int* word,
                                     unsigned int* out, void* stream);

/* Reads and clears the library's device error word (nonzero after a bounded
 * wait inside a kernel gave up).  Synchronises the device. */
gdn_status gdn_device_error(unsigned int* flag);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SELFTEST_H */
