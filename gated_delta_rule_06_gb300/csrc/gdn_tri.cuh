// gdn_tri.cuh -- the 64 x 64 unit lower-triangular inverse T = (I + A)^-1 of
// the chunked WY/UT form, in fp32 on the CUDA cores, shared by the forward
// chunk kernels of the scalar and the per-key-channel gates.
#pragma once

#include "gdn_internal.cuh"

namespace gdn {
namespace tri {

constexpr int C = kChunk;

// fp32 64 x 64 matrices in shared memory have rows of LDT floats: 68 keeps
// rows 16-byte aligned and moves consecutive rows four banks apart
constexpr int LDT = C + 4;

// T = (I + A)^-1 for a 64 x 64 strictly lower A (fp32, row stride LDT in shared
// memory), on 16 x 16 blocks.  (1) The diagonal blocks T_II = (I + A_II)^-1 by
// forward substitution, one column per thread.  (2) N_IK = T_II A_IK for the six
// blocks below the diagonal (into X).  (3) The block sub-diagonals d = 1, 2, 3 in
// turn: the block rows I > J of (I + A) T = I give
//   T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ = -sum_{K=J}^{I-1} N_IK T_KJ.
// Steps (2) and (3) give each thread eight or four adjacent columns of a row,
// with the 16-byte shared loads of several steps issued before their FMAs.  All threads of the CTA
// take part; ends synchronised.  Only the blocks on and below the diagonal of
// T are written (the diagonal blocks in full, zeros above their diagonal); the
// solve reads no other.
static __device__ void tri_inverse64(const float* A, float* T, float* X) {
    const int tid = threadIdx.x;
    if (tid < C) {
        const int blk = tid >> 4, c = tid & 15, o = 16 * blk;
        float col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a[16];
#pragma unroll
            for (int q = 0; q < (i + 3) / 4; ++q) {
                const float4 v4 = *reinterpret_cast<const float4*>(A + (o + i) * LDT + o + 4 * q);
                a[4 * q] = v4.x;
                a[4 * q + 1] = v4.y;
                a[4 * q + 2] = v4.z;
                a[4 * q + 3] = v4.w;
            }
            float v = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int jj = 0; jj < i; ++jj) v = fmaf(-a[jj], col[jj], v);
            col[i] = (i < c) ? 0.f : v;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) T[(o + i) * LDT + o + c] = col[i];
    }
    __syncthreads();
    for (int e = tid; e < 6 * 32; e += blockDim.x) {
        // block b -> (I, K): (1,0) (2,0) (2,1) (3,0) (3,1) (3,2); eight columns per task
        const int b = e >> 5, r = (e >> 1) & 15, c8 = (e & 1) * 8;
        const int I = b < 1 ? 1 : (b < 3 ? 2 : 3);
        const int K = b - I * (I - 1) / 2;
        const float* trow = T + (16 * I + r) * LDT + 16 * I;
        const float* acol = A + 16 * I * LDT + 16 * K + c8;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
        for (int kb = 0; kb < 16; kb += 4) {
            // all loads of four steps first, then their FMAs
            const float4 t4 = *reinterpret_cast<const float4*>(trow + kb);
            float4 x0[4], x1[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                x0[q] = *reinterpret_cast<const float4*>(acol + (kb + q) * LDT);
                x1[q] = *reinterpret_cast<const float4*>(acol + (kb + q) * LDT + 4);
            }
            const float tq[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a0.x = fmaf(tq[q], x0[q].x, a0.x);
                a0.y = fmaf(tq[q], x0[q].y, a0.y);
                a0.z = fmaf(tq[q], x0[q].z, a0.z);
                a0.w = fmaf(tq[q], x0[q].w, a0.w);
                a1.x = fmaf(tq[q], x1[q].x, a1.x);
                a1.y = fmaf(tq[q], x1[q].y, a1.y);
                a1.z = fmaf(tq[q], x1[q].z, a1.z);
                a1.w = fmaf(tq[q], x1[q].w, a1.w);
            }
        }
        float4* xo = reinterpret_cast<float4*>(X + (16 * I + r) * LDT + 16 * K + c8);
        xo[0] = a0;
        xo[1] = a1;
    }
    __syncthreads();
    for (int dlt = 1; dlt < 4; ++dlt) {
        for (int e = tid; e < (4 - dlt) * 64; e += blockDim.x) {
            const int bj = e >> 6, r = (e >> 2) & 15, c4 = (e & 3) * 4;
            const int bi = bj + dlt;
            const float* nrow = X + (16 * bi + r) * LDT;
            const float* tcol = T + 16 * bj + c4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int kb = 16 * bj; kb < 16 * bi; kb += 8) {
                // all loads of eight steps first, then their FMAs
                const float4 n0 = *reinterpret_cast<const float4*>(nrow + kb);
                const float4 n1 = *reinterpret_cast<const float4*>(nrow + kb + 4);
                float4 t[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) t[q] = *reinterpret_cast<const float4*>(tcol + (kb + q) * LDT);
                const float nq[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    acc.x = fmaf(nq[q], t[q].x, acc.x);
                    acc.y = fmaf(nq[q], t[q].y, acc.y);
                    acc.z = fmaf(nq[q], t[q].z, acc.z);
                    acc.w = fmaf(nq[q], t[q].w, acc.w);
                }
            }
            *reinterpret_cast<float4*>(T + (16 * bi + r) * LDT + 16 * bj + c4) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
    }
}

}  // namespace tri
}  // namespace gdn
