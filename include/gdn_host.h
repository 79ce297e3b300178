/*
 * gdn_host.h -- steps of the gated delta rule on HOST buffers (libgdn.so).
 *
 * The operation, layouts, dtypes and results are those of gdn_forward /
 * gdn_backward (or gdn_forward_lb / gdn_backward_lb) in gdn.h (mlx-lm PR "Add
 * gated_delta_update VJP", "What this PR adds": the forward and its VJP;
 * torch-to-nnef "custom_extractors/gdn", op contract).  The pages have no
 * counterpart to this packaging: it is the host-facing wrapper a training or
 * serving loop calls with its tensors in host memory.
 *
 * A session moves each step's inputs from host to device memory, runs the
 * forward (and the backward), and moves the results back.  It keeps three
 * slots of device buffers and three streams (the caller's `stream` for compute,
 * and an upload and a download stream of its own), so the copies of one step
 * run under the compute of the steps next to it.
 *
 *   - The session allocates no device memory.  The caller passes one device
 *     arena of gdn_host_session_bytes() bytes, 256-byte aligned, that it owns
 *     and keeps alive until gdn_host_session_destroy returns.
 *   - The session creates two CUDA streams and fifteen events on the current device
 *     and destroys them in gdn_host_session_destroy.
 *   - gdn_host_step only enqueues.  The caller must leave that step's host
 *     input buffers unchanged and must not read its host output buffers until
 *     gdn_host_session_sync (or destroy) returns.
 *   - Host buffers should be page-locked (cudaHostAlloc / pinned) for the copies
 *     to be asynchronous; pageable buffers give the same results, but their copies
 *     are not asynchronous.
 *   - Steps of one session are ordered; a session is not thread-safe.
 *   - Errors are those of gdn.h: GDN_ERR_INVALID_ARG (a required pointer is
 *     NULL, a flag is out of range), GDN_ERR_UNSUPPORTED_SHAPE,
 *     GDN_ERR_MISALIGNED (arena), GDN_ERR_WORKSPACE_TOO_SMALL (arena_bytes),
 *     GDN_ERR_CUDA (a copy, event or launch failed; gdn_last_cuda_error() has
 *     the text).  After an error in gdn_host_step the session should be
 *     destroyed.
 */
#ifndef GDN_HOST_H
#define GDN_HOST_H

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gdn_host_session gdn_host_session; /* opaque */

/* One step's host inputs.  Layouts as in gdn.h.
 *   q, k, v                     required
 *   a, b                        required: gates = 0 takes a, b; gates = 1 takes
 *                               log_decay, beta in these two fields
 *   A_log, dt_bias              required when gates = 0, ignored when 1
 *   state0                      NULL = zero initial state
 *   mask                        required iff shape->has_mask
 *   d_o                         required in a backward session, else ignored
 *   d_state_T                   NULL = zero cotangent (backward sessions) */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
    const float* state0;
    const uint8_t* mask;
    const void* d_o;
    const float* d_state_T;
} gdn_host_inputs;

/* One step's host outputs.  o and state_T always; in a backward session also
 * dq, dk, dv, da, db (d_log_decay, d_beta when gates = 1) and dstate0, and
 * dA_log, ddt_bias when gates = 0.  Fields a session does not write are
 * ignored. */
typedef struct {
    void* o;
    float* state_T;
    void* dq;
    void* dk;
    void* dv;
    void* da;
    void* db;
    float* dA_log;
    float* ddt_bias;
    float* dstate0;
} gdn_host_outputs;

/* Bytes of the device arena a session of this shape needs: three slots of one
 * step's inputs and outputs, plus (backward = 1) the saved buffer and the
 * larger of the two workspaces, or (backward = 0) the inference workspace.
 * Host-only. */
gdn_status gdn_host_session_bytes(const gdn_shape* shape, int32_t backward, size_t* bytes);

/* Creates a session.  gates: 0 = (a, b, A_log, dt_bias), 1 = (log_decay,
 * beta).  backward: 1 = each step runs the forward and the backward (a
 * training step), 0 = the forward only (inference; T = 1 runs the decode
 * kernel).  stream: the compute stream (cudaStream_t as void*, NULL = legacy
 * stream).  Arguments are checked before any CUDA call. */
gdn_status gdn_host_session_create(const gdn_shape* shape, int32_t gates, int32_t backward,
                                   void* arena, size_t arena_bytes, void* stream,
                                   gdn_host_session** out);

/* Enqueues one step on host buffers (see the conventions above). */
gdn_status gdn_host_step(gdn_host_session* session, const gdn_host_inputs* in,
                         const gdn_host_outputs* out);

/* Waits until every step enqueued so far has finished; their host outputs are
 * then complete. */
gdn_status gdn_host_session_sync(gdn_host_session* session);

/* Waits as gdn_host_session_sync does, then releases the session's streams and
 * events (NULL is a no-op). */
gdn_status gdn_host_session_destroy(gdn_host_session* session);

#ifdef __cplusplus
}
#endif

#endif /* GDN_HOST_H */
