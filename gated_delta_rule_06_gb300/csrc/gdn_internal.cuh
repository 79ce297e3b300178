// gdn_internal.cuh -- shapes, buffer layouts and device helpers shared by the
// CUDA kernels of the gated delta rule library.  Private to libgdn.so.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the library links the runtime alone)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kChunk = 64;           // chunk length (mlx-lm page, "Design notes")
constexpr int kConvMaxK = 16;        // longest causal conv1d kernel supported
constexpr float kNormEps = 1e-6f;    // L2-norm eps (torch-to-nnef page, op contract)
constexpr float kSoftplusClamp = 20.f;

struct Dims {
    int64_t B, T, Hk, Hv, Dk, Dv;
    int64_t G;   // Hv / Hk
    int64_t NC;  // number of chunks, ceil(T / 64)
    int64_t Tp;  // NC * 64 (sequence padded with identity steps)
    int dtype;   // 0 = fp32, 1 = bf16
    // gate inputs: 0 = (a, b, A_log, dt_bias), from which the kernels form
    // l = -exp(A_log) softplus(min(a + dt_bias, 20)) and beta = sigmoid(b);
    // 1 = the per-step log_decay l and beta themselves (in Ptrs::a, Ptrs::b;
    // A_log, dt_bias unused), whose cotangents the backward returns in da, db
    int gates = 0;
};

// TMA descriptors of the raw bf16 inputs v and dO (q and k reach the kernels as
// panel images written by prep) and of the output, encoded on the host for each call of
// the tensor-core path and handed to the kernels as __grid_constant__ params.
// Each describes a [B, T, H, D] tensor (row t of head h of batch b at
// ((b T + t) H + h) D) as 5-d {8, T, D / 8, H, B} with a box of 64 rows: one
// load brings a 64-row tile in the panel layout (8-column groups of 64 x 16
// bytes); rows past T arrive as zeros.
// `o` is the output [B, T, Hv, Dv] as 3-d {Hv Dv, T, B} with a row-major box of
// 64 rows x min(Dv, 128) columns, for TMA stores of staged output rows (rows past
// T are not written).
// `U` is the forward workspace U [B Hv Tp, Dv] fp32 with a box of 64 rows x
// min(Dv, 128) columns (row-major), for the forward scan.
struct Tmaps {
    CUtensorMap v, dO, dOf, o, U;  // dO: boxes min(Dv, 128) wide; dOf: Dv wide
    // U again for the chunk kernel's stores: boxes of 64 rows x 32 fp32, 128-byte swizzle
    CUtensorMap Us;
};
// box `cols` columns wide (multiple of 8, <= 256); false if the driver refuses
bool encode_row_tile_map(CUtensorMap* m, const void* base, int64_t B, int64_t T, int64_t H,
                         int64_t D, int cols);
bool encode_row_major_map(CUtensorMap* m, const void* base, int64_t B, int64_t T, int64_t rowlen,
                          int cols);
// fp32 [rows, cols_total] row-major, box of 64 rows x `cols` columns
bool encode_f32_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols_total, int cols);
// the same rows in boxes of 64 rows x 32 columns with the 128-byte swizzle: the
// 16-byte piece j of box row r sits at r * 128 + ((j ^ (r % 8)) * 16)
bool encode_f32_rows_map_sw128(CUtensorMap* m, const void* base, int64_t rows, int64_t cols_total);

// Every device buffer the kernels touch.  Inputs/outputs come from the
// caller; the rest are carved out of the caller's `saved` and `ws` buffers.
//
// Two storage formats exist for the saved intermediates.  The CUDA-core path
// (fp32 inputs, and shapes outside the tensor-core kernels' range) stores them
// row-major as annotated.  The tensor-core path (tc_path) stores every one of
// them as bf16 operand images per chunk, in the exact shared-memory layout the
// consuming MMA reads, so each is moved by one bulk copy:
//   ckpt   [B, Hv, NC] images of S^T (Dv rows x Dk, panel layout), bf16
//   Tinv   [B, Hv, NC] images of T (64 rows x 64, panel), bf16
//   W      [B, Hv, NC] images of W (64 rows x Dk, panel)
//   P      [B, Hv, NC] images of P (64 rows x 64, panel)
//   Delta  [B, Hv, NC] pairs {hi, lo} of images of Delta^T (Dv rows x 64,
//          canonical x = step, 8-row groups 1024 bytes apart), Delta = hi + lo
//   dSck   [B, Hv, NC] images of Sbar'^T (Dv rows x Dk, panel), bf16
//   kimg, qimg  [B, Hk, NC] images of the raw k / q rows (64 x Dk, panel)
//   Dbar   [B, Hv, NC] images of -Dbar^T (Dv rows x 64, as Delta), bf16
// U, gam, beta, rq, rk and the backward partials keep the row-major fp32 form.
struct Ptrs {
    // primal inputs
    const void *q, *k, *v, *a, *b;
    const float *A_log, *dt_bias, *state0;
    const uint8_t* mask;
    // forward outputs
    void* o;
    float* state_T;
    // saved (forward -> backward)
    float* ckpt;   // [B, Hv, NC, Dk, Dv] fp32 state at each chunk start
    double* gam;   // [B, Hv, Tp] in-chunk cumulative log-decay Gamma (fp64: the
                   // differences Gamma_i - Gamma_j must stay accurate when |Gamma| is large)
    float* beta;   // [B, Hv, Tp] write strength (0 on masked / padded steps)
    float* rq;     // [B, Hk, Tp] 1 / sqrt(|q|^2 + eps)   (0 on padded steps)
    float* rk;     // [B, Hk, Tp] 1 / sqrt(|k|^2 + eps)
    float* Tinv;   // [B, Hv, NC, 64, 64] fp32 (I + A)^-1 per chunk
    void* W;       // [B, Hv, Tp, Dk]  T diag(beta gam) K   (input dtype)
    void* P;       // [B, Hv, NC, 64, 64] (Q K^T) o M, lower incl. diagonal
    float* Delta;  // [B, Hv, Tp, Dv]  U - W S  per chunk (fp32: Delta cancels, see U)
    void* kimg;    // tensor-core path: [B, Hk, NC] images of the raw k rows of each
    void* qimg;    // chunk (64 rows x Dk, panel; rows past T zero), written by prep
    // forward workspace
    float* U;      // [B, Hv, Tp, Dv]  T diag(beta) V (fp32: Delta = U - W S cancels,
                   // so a rounded U would dominate the error of the log-decay gradient)
    // backward inputs / outputs
    const void* d_o;
    const float* d_state_T;
    void *dq, *dk, *dv, *da, *db;
    float *dA_log, *ddt_bias, *dstate0;
    // backward workspace
    float* dSck;   // [B, Hv, NC, Dk, Dv] state cotangent at each chunk END
    float* Dbar;   // [B, Hv, Tp, Dv] cotangent of Delta
    float* dqh;    // [B, Hv, Tp, Dk] cotangent of the normalised q, per value head
    float* dkh;    // [B, Hv, Tp, Dk]  (both bf16 [B, Tp, Hv, Dk] on the tensor-core path)
    float* dl;     // [B, Hv, Tp] cotangent of the log-decay
    float* dbeta;  // [B, Hv, Tp]
    float* part;   // [2, B, NC, Hv] per-chunk partial sums for dA_log, ddt_bias
    float* ecd;    // per-key-channel chunked form: [B, Hv, NC, Dk] exp(Gamma_63, i) of
                   // each chunk and key channel i (the state's per-chunk decay)
    void* krimg;   // per-key-channel chunked form: [B, Hv, NC] panel images of
                   // K_r = kh o exp(Gamma) (64 rows x Dk), bf16
    float* gram;   // per-key-channel chunked form: [B, Hv, NC, 64, 64] the decayed
                   // Gram sum_i kh_ti kh_si exp(Gamma_ti - Gamma_si), s < t (fp32)
    // per-key-channel chunked backward: per-chunk products of the tensor-core pass
    float* kdb;    // [B, Hv, Tp, Dk] Delta Sbar'^T       (cotangent of K_d)
    float* qrb;    // [B, Hv, Tp, Dk] Obar S^T             (cotangent of Q_r)
    float* wb;     // [B, Hv, Tp, Dk] diag(beta) T^T Wbar  (cotangent of K_r)
    float* pbm;    // [B, Hv, NC, 64, 64] Obar Delta^T, lower incl. diagonal
    float* m1;     // [B, Hv, NC, 64, 64] Dbar V^T + Wbar K_r^T, then Gbar
    float* ecb;    // [B, Hv, NC, Dk] <Sbar'_i, S_i> per key channel i
    unsigned int* sched;  // tensor-core path: [1 + B Hv] the gradient kernel's item
                          // counter, then the reverse scan's per-(b, h) progress
    // host copy of the tensor maps (tensor-core path; read by the launchers only)
    const Tmaps* tmaps;
};

// ---- scalar load / store in the input dtype ---------------------------------
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + __expf(-x)); }

// ---- CTA-wide fp32 GEMM on shared memory ------------------------------------
// C[m, n] = beta_c * C[m, n] + alpha * rs[m] * sum_k A(m, k) B(k, n)
// with A(m, k) = A[m * sam + k * sak] and B(k, n) = B[k * sbk + n * sbn].
// rs may be nullptr (all ones).  Each thread owns TM x TN output micro tiles;
// M % TM == 0 and N % TN == 0 are required.  The caller synchronises.
template <int TM, int TN>
__device__ __forceinline__ void cta_gemm(int M, int N, int K, const float* A, int sam, int sak,
                                         const float* Bm, int sbk, int sbn, float* C, int ldc,
                                         float alpha, float beta_c, const float* rs) {
    const int tilesN = N / TN;
    const int ntiles = (M / TM) * tilesN;
    for (int t = threadIdx.x; t < ntiles; t += blockDim.x) {
        const int m0 = (t / tilesN) * TM, n0 = (t % tilesN) * TN;
        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
        for (int kk = 0; kk < K; ++kk) {
            float av[TM], bv[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) av[i] = A[(m0 + i) * sam + kk * sak];
#pragma unroll
            for (int j = 0; j < TN; ++j) bv[j] = Bm[kk * sbk + (n0 + j) * sbn];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float s = alpha * (rs ? rs[m0 + i] : 1.f);
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                float* c = C + (m0 + i) * ldc + n0 + j;
                *c = (beta_c != 0.f ? beta_c * *c : 0.f) + s * acc[i][j];
            }
        }
    }
}

// ---- launchers (defined in the .cu files) -----------------------------------
cudaError_t launch_prep(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_fwd_chunk(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_fwd_scan(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_bwd_scan(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_bwd_chunk(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_bwd_reduce(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_decode(const Dims& d, const Ptrs& p, cudaStream_t s);
// the decode step with the short convolution fused in front (q, k, v come from
// `hidden` [B, 2 Hk Dk + Hv Dv] through the K-tap convolution; p.q, p.k, p.v unused)
cudaError_t launch_decode_conv(const Dims& d, const Ptrs& p, const void* hidden,
                               const void* conv_state, const void* weight, void* final_state,
                               int K, cudaStream_t s);
bool decode_supported(int64_t Dk, int64_t Dv);
// depthwise causal conv1d + SiLU with a K-sample carry state (K <= kConvMaxK)
cudaError_t launch_causal_conv1d_update(int64_t B, int64_t C, int64_t S, int K, int dtype,
                                        const void* hidden, const void* conv_state,
                                        const void* weight, void* out, void* final_state,
                                        cudaStream_t s);
// streaming multiprocessors of the current device (cached per device)
int sm_count();
// q / k row norms alone (rq, rk), and the q / k part of the reduction alone
cudaError_t launch_prep_norms(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_qk_reduce(const Dims& d, const Ptrs& p, cudaStream_t s);
// per-key-channel gates (gdn_kc.cu)
bool kc_supported(const Dims& d);
size_t kc_bwd_smem_bytes(const Dims& d);
int64_t kc_tiles(const Dims& d);
int64_t kc_segments(const Dims& d);
cudaError_t launch_kc_forward(const Dims& d, const Ptrs& p, const void* log_decay,
                              const void* beta, float* ckpt, cudaStream_t s);
cudaError_t launch_kc_backward(const Dims& d, const Ptrs& p, const void* log_decay,
                               const void* beta, const float* ckpt, float* gpart, float* bpart,
                               void* d_log_decay, void* d_beta, cudaStream_t s);
// Records e as the library's last CUDA error (the text gdn_last_cuda_error
// returns) and gives GDN_ERR_CUDA; cudaSuccess gives GDN_OK and records nothing.
int note_cuda_error(cudaError_t e);
unsigned int read_clear_error_decode();
// tensor-core (tcgen05) variants for bf16 inputs
bool bwd_chunk_tc_supported(const Dims& d);
cudaError_t launch_bwd_chunk_tc(const Dims& d, const Ptrs& p, cudaStream_t s);
// the reverse scan and the gradient kernel in one cooperative launch (bf16,
// shapes both tensor-core kernels take, fewer reverse-scan tiles than SMs)
bool bwd_fused_tc_supported(const Dims& d);
cudaError_t launch_bwd_fused_tc(const Dims& d, const Ptrs& p, cudaStream_t s);
unsigned int read_clear_error_bwdtc();
bool scan_tc_supported(const Dims& d);
cudaError_t launch_fwd_scan_tc(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_bwd_scan_tc(const Dims& d, const Ptrs& p, cudaStream_t s);
unsigned int read_clear_error_scantc();
bool scan_ta_supported(const Dims& d);
cudaError_t launch_fwd_scan_ta(const Dims& d, const Ptrs& p, cudaStream_t s);
// Segmented forward scan.  The chunk transition S_{c+1} = A_c S_c + B_c is affine
// in the state, so a run of chunks composes into one affine segment map.  The
// chunks are cut into nseg segments of len chunks (the last may be shorter):
//   mode 1 (maps): for segments 0 .. nseg - 2, the scan from the zero state (the
//     offset B_s, value tiles of Dv) and, with U = 0, from the identity (the linear
//     part A_s, value tiles over Dk padded to the tile width); the end states go to
//     maps [nseg - 1][B][Hv][Dk][Wd], Wd = Dv + Dk padded, offset part first;
//   the chain kernel: S_{s+1} = A_s S_s + B_s from S_0 = state0 into start
//     [nseg - 1][B][Hv][Dk][Dv] (the start states of segments 1 ..);
//   mode 0 (the scan proper): every segment from its start state at once, writing
//     the checkpoints, Delta images and outputs of its chunks; the last segment
//     writes the final state.
// A launch may also cover segment `first` alone (grid z = B) with its start
// state read from `sin` and its end state written to `sout` ([B][Hv][Dk][Dv]
// fp32 each, null: the rules above): the chunk-by-chunk scans of the compressed
// forward and backward, which change the state between two chunks.
struct ScanSeg {
    int nseg, len, mode;
    float* start;
    float* maps;
    int first = 0;
    const float* sin = nullptr;
    float* sout = nullptr;
};
int64_t seg_map_width(const Dims& d);  // Wd
cudaError_t launch_fwd_scan_ta_seg(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s);
cudaError_t launch_seg_chain(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s);
// The same three passes for the reverse scan of the backward (segment t counted
// from the top, the bottom one possibly shorter): the maps of segments 0 .. nseg - 2
// (mode 1), the chain from d_state_T (launch_seg_chain with state0 = d_state_T),
// then every segment (mode 0); the per-chunk gradients follow as their own launch.
cudaError_t launch_bwd_scan_ta_seg(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s);
cudaError_t launch_bwd_scan_ta(const Dims& d, const Ptrs& p, cudaStream_t s);
// segment sg.first alone (mode 0, grid z = B), forward and reverse
cudaError_t launch_fwd_scan_ta_one(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s);
cudaError_t launch_bwd_scan_ta_one(const Dims& d, const Ptrs& p, const ScanSeg& sg, cudaStream_t s);
unsigned int read_clear_error_scanta();
// per-key-channel gates, chunked form: the scans with the chunk kernel's
// per-value-head Q_r / K_d images (p.qimg / p.kimg) and per-channel decays (p.ecd)
cudaError_t launch_fwd_scan_kc(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_bwd_scan_kc(const Dims& d, const Ptrs& p, cudaStream_t s);
// the chunk-local products of the chunked per-key-channel form (gdn_kc_tc.cu)
bool kc_chunked_supported(const Dims& d);
cudaError_t launch_kc_chunk(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_kc_bwd_prod(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_kc_bwd_gate(const Dims& d, const Ptrs& p, cudaStream_t s);
cudaError_t launch_kc_bwd_chan(const Dims& d, const Ptrs& p, cudaStream_t s);
unsigned int read_clear_error_kctc();
bool fwd_chunk_tc_supported(const Dims& d);
cudaError_t launch_fwd_chunk_tc(const Dims& d, const Ptrs& p, cudaStream_t s);
unsigned int read_clear_error_fwdtc();
// rank-r compressed chunk states: the truncation at boundary c of every (b, h)
// (chunk-end states S_end in, truncated states S_tr out, factors into slot c of
// Qf [B][Hv][NC][Dk][r] and Rf [B][Hv][NC][r][Dv], fp32), and the bf16
// checkpoint images of every chunk start state rebuilt from them (chunk 0 from
// S0f [B][Hv][Dk][Dv])
bool compress_supported(const Dims& d, int rank, int iters);
cudaError_t launch_trunc(const Dims& d, const float* S_end, const float* omega, int rank, int iters,
                         float* S_tr, float* Qf, float* Rf, int64_t c, cudaStream_t s);
cudaError_t launch_expand_ckpt(const Dims& d, const float* S0f, const float* Qf, const float* Rf,
                               int rank, void* img, cudaStream_t s);
// bf16 inputs whose shape every tensor-core kernel supports: the whole forward
// and backward run on the tensor-core kernels with the image formats above
bool tc_path(const Dims& d);
// adds n to the library's launch counter (called by every launcher)
void count_launches(int n);
// chunk index e of a 64-row (or 8k-row) canonical-tile copy -> (row, 8-column
// group) with row % 8 fastest: eight consecutive chunks fill one 128-byte core
// matrix (conflict-free shared-memory stores) and a warp covers 8 rows x 4
// column groups (whole 32-byte sectors of the global rows)
__device__ __forceinline__ void chunk_rc(int e, int cpr, int& row, int& cc) {
    const int t = e >> 3;
    cc = t % cpr;
    row = (t / cpr) * 8 + (e & 7);
}
// reads and clears the device error words of every translation unit
// (~0u if a read failed); defined in gdn_api.cu
unsigned int read_clear_error_all();
unsigned int read_clear_error_selftest();

}  // namespace gdn
