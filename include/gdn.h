/*
 * gdn.h -- C ABI of the GB300 gated delta rule library (libgdn.so).
 *
 * The operation (mlx-lm PR "Add gated_delta_update VJP - trainable
 * GatedDeltaNet on Apple Silicon", "What this PR adds"; torch-to-nnef
 * "custom_extractors/gdn", op contract):
 *
 *   per batch b and value head h (key head j = h / G, G = Hv / Hk):
 *     qh_t = q_t / sqrt(|q_t|^2 + 1e-6) / sqrt(Dk),  kh_t = k_t / sqrt(|k_t|^2 + 1e-6)
 *     g_t  = exp(-exp(A_log[h]) * softplus(min(a_t + dt_bias[h], 20)))
 *     beta_t = sigmoid(b_t)
 *     if mask[b, t]:  S <- g_t S;  delta = beta_t (v_t - S^T kh_t);  S <- S + kh_t delta^T
 *     o_t = S^T qh_t                       (a masked step leaves S unchanged)
 *
 * gdn_forward returns o and the final state; gdn_backward returns the
 * gradients of q, k, v, a, b, A_log, dt_bias and the initial state (the VJP
 * the mlx-lm page adds).  The sequence is processed in chunks of 64 steps
 * (mlx-lm page, "Design notes": CHUNK_SIZE = 64); the forward keeps the fp32
 * state at every chunk start in a caller-owned "saved" buffer that the
 * backward consumes.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or synchronises.  All work is enqueued
 *     on `stream` (a cudaStream_t passed as void*, NULL = legacy stream).
 *   - Tensors are dense row-major in these layouts:
 *       q, k, dq, dk        [B, T, Hk, Dk]   dtype
 *       v, o, d_o, dv       [B, T, Hv, Dv]   dtype
 *       a, b, da, db        [B, T, Hv]       dtype
 *       A_log, dt_bias, dA_log, ddt_bias   [Hv]  fp32
 *       state0, state_T, d_state_T, dstate0 [B, Hv, Dk, Dv] fp32
 *       mask                [B, T]  uint8, nonzero = step applied
 *     where dtype is GDN_DTYPE_F32 (float) or GDN_DTYPE_BF16 (bfloat16).
 *   - Every pointer must be 16-byte aligned (GDN_ERR_MISALIGNED otherwise).
 *   - Arguments are validated on the host before anything is launched; an
 *     error returns a status and leaves every output untouched.  A failed
 *     launch returns GDN_ERR_CUDA (the CUDA error is reported by
 *     gdn_last_cuda_error()).  Nothing aborts the process or throws.
 *   - Results are deterministic: no atomics; every reduction has a fixed order.
 *
 * Supported shapes: B >= 1, T >= 1, Hk >= 1, Hv % Hk == 0,
 * 8 <= Dk, Dv <= 256 and both multiples of 8.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,         /* null pointer where one is required, bad enum */
    GDN_ERR_UNSUPPORTED_SHAPE = 2,   /* shape outside the supported set above */
    GDN_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes or saved_bytes below the sizing call */
    GDN_ERR_MISALIGNED = 4,          /* a pointer is not 16-byte aligned */
    GDN_ERR_CUDA = 5                 /* a kernel launch failed */
} gdn_status;

typedef enum { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 } gdn_dtype;

typedef struct {
    int64_t B, T, Hk, Hv, Dk, Dv;
    int32_t dtype;    /* gdn_dtype of q, k, v, a, b, o and of their gradients */
    int32_t has_mask; /* 0: mask pointer ignored (every step applied) */
} gdn_shape;

/* Human-readable name of a status code (static string, never NULL). */
const char* gdn_status_string(gdn_status status);

/* Text of the last CUDA error seen by this thread inside the library. */
const char* gdn_last_cuda_error(void);

/* Bytes of scratch the caller must pass as `ws` to gdn_forward (pass = 0)
 * or gdn_backward (pass = 1).  Host-only; launches nothing. */
gdn_status gdn_workspace_bytes(const gdn_shape* shape, int pass, size_t* bytes);

/* Bytes of the `saved` buffer that gdn_forward fills and gdn_backward reads:
 * the fp32 state at each of the ceil(T/64) chunk starts plus per-chunk
 * intermediates of the WY/UT form (mlx-lm page, "Scope and follow-ups":
 * chunk-parallel form through a lower-triangular solve).  Host-only. */
gdn_status gdn_saved_bytes(const gdn_shape* shape, size_t* bytes);

/* The same number under the name the checkpoint sizing call also goes by: the
 * saved buffer is where the forward keeps the chunk-start states (the
 * checkpoints) together with the per-chunk intermediates the backward reads.
 * On the tensor-core path the checkpoints are stored as bf16 operand images,
 * so the buffer is not B*Hv*NC*Dk*Dv*4 bytes of fp32 states. */
gdn_status gdn_checkpoint_bytes(const gdn_shape* shape, size_t* bytes);

/* Forward pass.  state0 may be NULL (zero initial state); mask may be NULL
 * (every step applied).  state_T may alias state0 (in-place update).
 * saved may be NULL for inference (nothing kept for the backward); then,
 * when T == 1, the single-step decode kernel runs and ws may be NULL.
 * Otherwise ws must hold gdn_workspace_bytes(shape, 0) bytes. */
gdn_status gdn_forward(const gdn_shape* shape, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log,
                       const float* dt_bias, const float* state0, const uint8_t* mask,
                       void* o, float* state_T, void* saved, size_t saved_bytes, void* ws,
                       size_t ws_bytes, void* stream);

/* Backward pass (VJP).  Takes the same primal inputs and the `saved` buffer
 * of a gdn_forward call on them, the cotangent d_o of o and d_state_T of the
 * final state (NULL = zero), and writes dq, dk, dv, da, db (dtype),
 * dA_log, ddt_bias [Hv] and dstate0 [B, Hv, Dk, Dv] (fp32).  Every output
 * is written in full (no accumulation into existing contents).  ws must
 * hold gdn_workspace_bytes(shape, 1) bytes. */
gdn_status gdn_backward(const gdn_shape* shape, const void* q, const void* k, const void* v,
                        const void* a, const void* b, const float* A_log,
                        const float* dt_bias, const uint8_t* mask, const void* saved,
                        size_t saved_bytes, const void* d_o, const float* d_state_T,
                        void* dq, void* dk, void* dv, void* da, void* db, float* dA_log,
                        float* ddt_bias, float* dstate0, void* ws, size_t ws_bytes,
                        void* stream);

/* ---- log_decay / beta gate form --------------------------------------------- */

/* The op contract's other gate input (torch-to-nnef "custom_extractors/gdn",
 * op contract: log_decay and beta [b, S, hv]): the per-step log-decay
 * l_t = log g_t and beta_t are given directly instead of (a, b, A_log,
 * dt_bias); the recurrence is the one above with g_t = exp(l_t).
 *   - log_decay, beta, d_log_decay, d_beta: [B, T, Hv] in the shape's dtype.
 *   - log_decay must be finite and <= 0 (g in (0, 1], a decay), and beta
 *     finite; the chunked kernels rely on the cumulative log-decay not
 *     increasing within a chunk.  Values are not checked (they live on the
 *     device): outside that range results are unspecified.
 *   - Sizing, `saved`, `ws`, masking, decode (T == 1, saved == NULL) and every
 *     other convention are those of gdn_forward / gdn_backward, and a saved
 *     buffer from gdn_forward_lb is consumed by gdn_backward_lb.
 *   - gdn_backward_lb writes d_log_decay and d_beta (zero on masked steps) in
 *     place of da, db, dA_log and ddt_bias. */
gdn_status gdn_forward_lb(const gdn_shape* shape, const void* q, const void* k, const void* v,
                          const void* log_decay, const void* beta, const float* state0,
                          const uint8_t* mask, void* o, float* state_T, void* saved,
                          size_t saved_bytes, void* ws, size_t ws_bytes, void* stream);
gdn_status gdn_backward_lb(const gdn_shape* shape, const void* q, const void* k,
                           const void* v, const void* log_decay, const void* beta,
                           const uint8_t* mask, const void* saved, size_t saved_bytes,
                           const void* d_o, const float* d_state_T, void* dq, void* dk,
                           void* dv, void* d_log_decay, void* d_beta, float* dstate0,
                           void* ws, size_t ws_bytes, void* stream);

/* ---- segmented (associative) forward scan -------------------------------- */

/* The state recurrence of one chunk is an affine map of the state,
 * S_{c+1} = A_c S_c + B_c with A_c = gam_C I - K^T diag(e) W and
 * B_c = K^T diag(e) U, and affine maps compose associatively (mlx-lm page,
 * "Post-initial-submission extensions", Extension 5: the recurrence as an
 * associative monoid, for scans that are not one sequential pass).
 * gdn_forward_segmented cuts the chunks into `segments` runs of equal length
 * (the last may be shorter), forms every run's composed map but the last in
 * parallel (the scan from the zero state gives its offset, the scan from the
 * identity with U = 0 its linear part), chains the run start states
 * S_{s+1} = A_s S_s + B_s in fp32, and then scans every run from its start state
 * at once.  Its results are those of gdn_forward up to rounding, and its saved
 * buffer is the same (gdn_backward consumes it unchanged): it only shortens
 * the sequential chain when B * Hv * (Dv / 128) leaves SMs idle and T is long.
 *   - Arguments, layouts and saved-buffer rules as gdn_forward (a, b, A_log,
 *     dt_bias gates).  ws must hold gdn_workspace_bytes(shape, 0) bytes
 *     (gdn_workspace_bytes(shape, 2) when saved is NULL) plus
 *     gdn_segment_bytes(shape, segments) bytes.
 *   - segments = 1: the plain scan (as gdn_forward); 0: the count
 *     gdn_segments_auto picks; above the number of chunks it is clamped.
 *   - segments > 1 requires bf16 with Dv % 128 == 0 and Dk in {64, 128, 192}
 *     (the tensor-core scan), and B * segments <= 65535; otherwise
 *     GDN_ERR_UNSUPPORTED_SHAPE.  T == 1 with saved == NULL runs the decode
 *     kernel as gdn_forward does. */
gdn_status gdn_forward_segmented(const gdn_shape* shape, int segments, const void* q,
                                 const void* k, const void* v, const void* a, const void* b,
                                 const float* A_log, const float* dt_bias, const float* state0,
                                 const uint8_t* mask, void* o, float* state_T, void* saved,
                                 size_t saved_bytes, void* ws, size_t ws_bytes, void* stream);

/* The reverse scan of the backward is affine in the state cotangent too, with
 * the transposed chunk transition as its linear part, so gdn_backward_segmented
 * runs it in the same three passes (segments counted from the end of the
 * sequence, the first one possibly shorter): the maps, the chain from
 * d_state_T, every segment's reverse scan; the per-chunk gradients then run as
 * their own launch on every SM instead of beside a single scan.  gdn_backward
 * takes the automatic count of a model that weighs that against the single
 * fused launch (one segment at the benched 9B layer shape).
 *   - Arguments as gdn_backward.  ws must hold gdn_workspace_bytes(shape, 1)
 *     plus gdn_segment_bytes(shape, segments) bytes.
 *   - segments = 1: one reverse pass (as gdn_backward picks it for one
 *     segment); 0: the automatic count; requirements as gdn_forward_segmented.
 *   - Any saved buffer of gdn_forward / gdn_forward_segmented of the same
 *     inputs is accepted: the segment counts of the two need not agree. */
gdn_status gdn_backward_segmented(const gdn_shape* shape, int segments, const void* q,
                                  const void* k, const void* v, const void* a, const void* b,
                                  const float* A_log, const float* dt_bias, const uint8_t* mask,
                                  const void* saved, size_t saved_bytes, const void* d_o,
                                  const float* d_state_T, void* dq, void* dk, void* dv, void* da,
                                  void* db, float* dA_log, float* ddt_bias, float* dstate0,
                                  void* ws, size_t ws_bytes, void* stream);

/* Extra workspace bytes of gdn_forward_segmented / gdn_backward_segmented with
 * `segments` segments (0: the forward's automatic count): the segment maps
 * [segments - 1][B][Hv][Dk][Dv + Dk rounded up to 128] and the chained states
 * [segments - 1][B][Hv][Dk][Dv], fp32.  0 for one segment.  gdn_workspace_bytes
 * already includes the buffers of the automatic counts.  Host-only. */
gdn_status gdn_segment_bytes(const gdn_shape* shape, int segments, size_t* bytes);

/* The segment count the automatic choice takes (1 = the plain scan): the count
 * that minimises a model of the sequential chain, in waves of the GPU's SMs times
 * chunks per run.  Reads the SM count of the current device. */
gdn_status gdn_segments_auto(const gdn_shape* shape, int* segments);

/* The backward's automatic segment count (1 = one reverse pass, fused with the
 * per-chunk gradients where that fits).  Reads the SM count of the current
 * device. */
gdn_status gdn_backward_segments_auto(const gdn_shape* shape, int* segments);

/* ---- per-key-channel gates ------------------------------------------------ */

/* The vectorised gating the mlx-lm page lists (g.ndim == 4, "Scope and
 * follow-ups": on its Python path only): one decay per key channel.  Taken in
 * the op contract's log_decay form with a key-channel axis (torch-to-nnef
 * "custom_extractors/gdn", op contract):
 *   - log_decay, d_log_decay: [B, T, Hv, Dk]; beta, d_beta: [B, T, Hv]; both in
 *     the shape's dtype.  l_{t,i} = log g_{t,i} <= 0 for key channel i.
 *   - An applied step scales row i of the state by g_{t,i} before the delta
 *     rule: S_a = diag(g_t) S, delta = beta_t (v_t - S_a^T kh_t),
 *     S = S_a + kh_t delta^T, o_t = S^T qh_t.  Masking, norms, layouts of q, k,
 *     v, o, the states and their cotangents are those of gdn_forward /
 *     gdn_backward.
 *   - Two forms, chosen by the shape.  bf16 inputs with Dk 64, 128 or 192 and
 *     Dv 128 take the chunked form: per 64-step chunk the decayed key products
 *     (exp(Gamma_t,i - Gamma_s,i) through 16-step pivots, every factor <= 1, so
 *     any l <= 0 is safe) and the WY/UT solve on the CUDA cores in fp32, the
 *     scans and the value-long gradient products on the tensor cores; `saved`
 *     holds per-chunk bf16 images (checkpoints, Delta, W, P, T, Q_r, K_d, K_r)
 *     and fp32 decays and Grams.  Every other shape takes the recurrence on the
 *     CUDA cores with an fp32 state: one CTA per 16 value columns of a (b, h),
 *     the state at every 8th step kept in `saved` for the backward.
 *   - Requires Dk a multiple of 32 and Dv of 16 (Dk <= 256) on top of gdn.h's set,
 *     else GDN_ERR_UNSUPPORTED_SHAPE.  gdn_kc_saved_bytes and
 *     gdn_kc_workspace_bytes size the form the shape takes.
 *   - saved may be NULL in gdn_forward_kc (inference).  ws must hold
 *     gdn_kc_workspace_bytes(shape, 0) bytes for the forward and (shape, 1) for
 *     the backward; every output is written in full. */
gdn_status gdn_kc_saved_bytes(const gdn_shape* shape, size_t* bytes);
gdn_status gdn_kc_workspace_bytes(const gdn_shape* shape, int pass, size_t* bytes);
gdn_status gdn_forward_kc(const gdn_shape* shape, const void* q, const void* k, const void* v,
                          const void* log_decay, const void* beta, const float* state0,
                          const uint8_t* mask, void* o, float* state_T, void* saved,
                          size_t saved_bytes, void* ws, size_t ws_bytes, void* stream);
gdn_status gdn_backward_kc(const gdn_shape* shape, const void* q, const void* k, const void* v,
                           const void* log_decay, const void* beta, const uint8_t* mask,
                           const void* saved, size_t saved_bytes, const void* d_o,
                           const float* d_state_T, void* dq, void* dk, void* dv,
                           void* d_log_decay, void* d_beta, float* dstate0, void* ws,
                           size_t ws_bytes, void* stream);

/* ---- rank-r compressed chunk states ---------------------------------------- */

/* Compression-aware training (mlx-lm page, "Post-initial-submission
 * extensions", Extension 1: power-iteration rank-r truncation of the state at
 * every chunk boundary; three iterations there, ranks of at most 16 per
 * Extension 6).  Only rank-r factors of each chunk state are kept between the
 * forward and the backward.
 *   - Boundaries: between consecutive 64-step chunks.  The state S (Dk x Dv)
 *     reached at the end of a chunk is replaced, before the next chunk starts,
 *     by Q R: Y = S omega, Q = orth(Y), then `iters` times Y = S (S^T Q),
 *     Q = orth(Y); R = Q^T S.  orth is Gram-Schmidt with one reorthogonalisation
 *     pass; a column in the span of the earlier ones (to fp32 rounding) becomes
 *     zero.  state0 enters chunk 0 as given and state_T, after the last chunk, is
 *     not truncated.  Masking does not change where the truncation applies.
 *   - omega: device fp32 [Dv][rank] row-major, the start block of the power
 *     iteration, drawn by the caller (any fixed full-rank block; a Gaussian one is
 *     usual).  rank: 1 .. 16; iters: 0 .. 16.
 *   - The backward passes the state cotangent straight through each boundary:
 *     it is the chunked VJP along the compressed trajectory (each chunk from its
 *     truncated start state), with the truncation's derivative taken as the
 *     identity.
 *   - bf16 inputs whose shape runs every tensor-core kernel with 128-column
 *     value tiles (Dk in {64, 128, 192}, Dv = 128), a and b gates (A_log,
 *     dt_bias), else GDN_ERR_UNSUPPORTED_SHAPE.
 *   - gdn_compressed_bytes gives the saved buffer (the other saved
 *     intermediates, state0 in fp32 and the factors Q [B][Hv][NC][Dk][rank],
 *     R [B][Hv][NC][rank][Dv] in fp32) and the forward and backward workspaces;
 *     gdn_backward_compressed takes the saved buffer of gdn_forward_compressed
 *     with the same rank.  Buffers, streams and errors are as for gdn_forward /
 *     gdn_backward; the forward enqueues 2 NC + 1 launches and one device copy
 *     (or memset) of state0. */
gdn_status gdn_compressed_bytes(const gdn_shape* shape, int rank, size_t* saved_bytes,
                                size_t* fwd_ws_bytes, size_t* bwd_ws_bytes);
gdn_status gdn_forward_compressed(const gdn_shape* shape, int rank, int iters, const float* omega,
                                  const void* q, const void* k, const void* v, const void* a,
                                  const void* b, const float* A_log, const float* dt_bias,
                                  const float* state0, const uint8_t* mask, void* o, float* state_T,
                                  void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                                  void* stream);
gdn_status gdn_backward_compressed(const gdn_shape* shape, int rank, const void* q, const void* k,
                                   const void* v, const void* a, const void* b, const float* A_log,
                                   const float* dt_bias, const uint8_t* mask, const void* saved,
                                   size_t saved_bytes, const void* d_o, const float* d_state_T,
                                   void* dq, void* dk, void* dv, void* da, void* db, float* dA_log,
                                   float* ddt_bias, float* dstate0, void* ws, size_t ws_bytes,
                                   void* stream);

/* ---- causal conv1d update ------------------------------------------------- */

/* Depthwise causal conv1d + SiLU with a K-sample carry state, the short
 * convolution in front of the recurrence (torch-to-nnef "custom_extractors/gdn",
 * CausalConvUpdateReified: hidden [b, C, S], conv_state [b, C, k], weight
 * [C, k] -> out [b, C, S], final_state [b, C, k]).  Per (b, c), the K carried
 * samples followed by the S new ones form one sequence x, and
 *     out_t = SiLU(sum_{i<K} weight[c, i] x_{t+1+i}),   t = 0 .. S-1
 *     final_state = the last K samples of x
 * (no bias; the oldest carried sample lies outside every window).
 *   - hidden, out [B, C, S]; conv_state, final_state [B, C, K]; weight [C, K];
 *     all in `dtype` (gdn_dtype), fp32 arithmetic.  final_state may alias
 *     conv_state (in-place update); out must not alias an input.
 *   - B, C, S >= 1 and 1 <= K <= 16 (GDN_ERR_UNSUPPORTED_SHAPE otherwise);
 *     pointers 16-byte aligned; device pointers; enqueued on `stream`. */
gdn_status gdn_causal_conv1d_update(int64_t B, int64_t C, int64_t S, int64_t K, int32_t dtype,
                                    const void* hidden, const void* conv_state,
                                    const void* weight, void* out, void* final_state,
                                    void* stream);

/* ---- decode step with the convolution fused in front ----------------------- */

/* One T = 1 step of the recurrence whose q, k, v come from the short
 * convolution (gdn_causal_conv1d_update) of the layer's mixed projection, in
 * one kernel (mlx-lm page, "Scope and follow-ups": a mega-fused T = 1 kernel;
 * torch-to-nnef page: the conv update and the recurrence as the two ops of the
 * decode path).
 *   - hidden [B, C] (the S = 1 column of [B, C, 1]), C = 2 Hk Dk + Hv Dv,
 *     holding q | k | v along C, each head-major (q channel j Dk + i, k channel
 *     Hk Dk + j Dk + i, v channel 2 Hk Dk + h Dv + i); conv_state,
 *     final_conv_state [B, C, K]; conv_weight [C, K]; all in shape->dtype.
 *   - final_conv_state receives the shifted windows and must not overlap
 *     conv_state (the G value heads of a key head read the same q / k channels).
 *   - gates = 0: a, b [B, Hv] with A_log, dt_bias [Hv] as in gdn_forward;
 *     gates = 1: a = log_decay, b = beta [B, Hv] as in gdn_forward_lb (A_log,
 *     dt_bias ignored).
 *   - state0 [B, Hv, Dk, Dv] (NULL = zeros), state_T may alias it; o
 *     [B, 1, Hv, Dv].  A masked row (mask[b] == 0) keeps both its carried
 *     conv state and its recurrent state; its o reads the unchanged state.
 *   - Requires shape->T == 1, 1 <= K <= 16, Dv % 4 == 0 and the state of one
 *     head within shared memory (Dk * Dv <= 32768 at Dv = 128). */
gdn_status gdn_decode_conv(const gdn_shape* shape, int32_t gates, int64_t K, const void* hidden,
                           const void* conv_state, const void* conv_weight,
                           void* final_conv_state, const void* a, const void* b,
                           const float* A_log, const float* dt_bias, const float* state0,
                           const uint8_t* mask, void* o, float* state_T, void* stream);

/* ---- forward without any allocation -------------------------------------- */

/* Inference forward (no saved buffer) that allocates nothing and takes no
 * workspace: for callers that cannot allocate device memory where they run the
 * op (an inference runtime or plugin host that forbids allocation while work
 * is enqueued, code inside a CUDA stream capture, a host whose device memory
 * is fixed up front).  The pages have no counterpart: it is a packaging of
 * gdn_forward (saved = NULL) whose scratch lives in a fixed device array owned
 * by the library.
 *   - Inputs, outputs, layouts and results are those of gdn_forward with
 *     saved = NULL; the caller passes only inputs and outputs.
 *   - The scratch is a static device array of gdn_noalloc_scratch_bytes()
 *     bytes (64 MiB) that every GPU which loads the library holds until the
 *     process exits.  When gdn_workspace_bytes(shape, 2) exceeds it but the
 *     same less gdn_segment_bytes(shape, 0) fits, the single-pass scan runs
 *     (as gdn_forward_segmented with one segment); shapes for which that does
 *     not fit either are rejected with GDN_ERR_WORKSPACE_TOO_SMALL before
 *     anything is launched.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the one array and leave their intermediates in it:
 *     calls whose work overlaps on the GPU (other streams, other threads)
 *     race; serialise them.  Nothing in it needs to start at zero.
 *   - Returns GDN_ERR_CUDA if the address lookup or a launch fails. */
size_t gdn_noalloc_scratch_bytes(void);
gdn_status gdn_forward_noalloc(const gdn_shape* shape, const void* q, const void* k,
                               const void* v, const void* a, const void* b, const float* A_log,
                               const float* dt_bias, const float* state0, const uint8_t* mask,
                               void* o, float* state_T, void* stream);

/* ---- instrumentation (host-only bookkeeping, off by default) -------------- */

/* Number of CUDA kernels this library has launched in this process so far. */
uint64_t gdn_launch_count(void);

/* Per-phase device time.  gdn_timing_begin() makes every later gdn_forward /
 * gdn_backward record a CUDA event pair around each of its phases, on the
 * call's stream.  gdn_timing_end() waits for those events, writes up to
 * `max` entries {phase name, launches, total milliseconds} in first-seen
 * order, sets *count, and switches recording off.  Returns GDN_ERR_CUDA if an
 * event failed.  Phases: "prep", "fwd_chunk", "fwd_scan", "bwd_scan",
 * "bwd_chunk", "bwd_scan_chunk" (the reverse scan and the gradient kernel in one
 * launch), "bwd_reduce", "decode", "kc_fwd", "kc_bwd" (the recurrent
 * per-key-channel form), "kc_chunk", "kc_scan", "kc_bwd_scan", "kc_bwd_prod",
 * "kc_bwd_gate", "kc_bwd_chan" (its chunked form).  Not thread-safe: one
 * caller at a time. */
typedef struct {
    const char* name;
    int64_t launches;
    double total_ms;
} gdn_phase_time;

gdn_status gdn_timing_begin(void);
gdn_status gdn_timing_end(gdn_phase_time* out, int max, int* count);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
