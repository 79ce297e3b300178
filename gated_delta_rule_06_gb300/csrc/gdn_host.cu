// gdn_host.cu -- training (or inference) steps on HOST buffers.
//
// A session owns no device memory: the caller hands it one device arena
// (gdn_host_session_bytes) that holds kSlots = 3 slots of step inputs and
// outputs, the saved buffer and the workspace.  Each gdn_host_step enqueues, for
// step n in slot n % 3:
//   up stream       wait until step n - 3 has finished with the slot;
//                   host -> device copies of the forward inputs, then of the
//                   backward-only inputs (d_o, d_state_T)
//   compute stream  forward, then backward (the caller's stream)
//   down stream     device -> host copies of o and the final state once the
//                   forward is done, of the gradients once the backward is
//                   done; then the slot is released
// so the copies of a step run under the compute of its neighbours while each
// step still moves all of its own inputs and results.  A slot's turn (its
// uploads, its compute, its downloads) is longer than a step when the copies
// take about as long as the compute; with two slots the next step but one
// waited for it, with three the uploads of step n + 3 wait only for step n's
// downloads.  The forward and backward
// are gdn_forward / gdn_backward (or the log_decay / beta form) on the slot's
// device buffers; the saved buffer and the workspace are shared by all steps,
// whose compute is serialised on the one compute stream.
#include <gdn_host.h>

#include <cstdlib>
#include <cstring>

#include "gdn_internal.cuh"

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// byte sizes of one step's tensors
struct Sizes {
    size_t q, v, g, h, st, mask;  // q/k, v/o/d_o/dv, a/b/da/db, per-head fp32, state, mask
};
Sizes sizes_of(const gdn_shape& s) {
    const size_t es = s.dtype == GDN_DTYPE_BF16 ? 2 : 4;
    Sizes z;
    z.q = (size_t)(s.B * s.T * s.Hk * s.Dk) * es;
    z.v = (size_t)(s.B * s.T * s.Hv * s.Dv) * es;
    z.g = (size_t)(s.B * s.T * s.Hv) * es;
    z.h = (size_t)s.Hv * 4;
    z.st = (size_t)(s.B * s.Hv * s.Dk * s.Dv) * 4;
    z.mask = s.has_mask ? (size_t)(s.B * s.T) : 0;
    return z;
}

struct Slot {
    // inputs
    void *q, *k, *v, *a, *b;
    float *A_log, *dt_bias, *state0;
    uint8_t* mask;
    void* d_o;
    float* d_state_T;
    // outputs
    void *o, *dq, *dk, *dv, *da, *db;
    float *state_T, *dA_log, *ddt_bias, *dstate0;
};

constexpr int kSlots = 3;

struct Plan {
    size_t slot_bytes, saved, ws, total;
};

// Offsets are handed out in a fixed order; `base` null only measures.
size_t carve_slot(const gdn_shape& s, int backward, uint8_t* base, Slot* sl) {
    const Sizes z = sizes_of(s);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* p = base ? base + off : nullptr;
        off += align_up(bytes ? bytes : 1);
        return p;
    };
    Slot t{};
    t.q = take(z.q);
    t.k = take(z.q);
    t.v = take(z.v);
    t.a = take(z.g);
    t.b = take(z.g);
    t.A_log = (float*)take(z.h);
    t.dt_bias = (float*)take(z.h);
    t.state0 = (float*)take(z.st);
    t.mask = (uint8_t*)take(z.mask);
    t.o = take(z.v);
    t.state_T = (float*)take(z.st);
    if (backward) {
        t.d_o = take(z.v);
        t.d_state_T = (float*)take(z.st);
        t.dq = take(z.q);
        t.dk = take(z.q);
        t.dv = take(z.v);
        t.da = take(z.g);
        t.db = take(z.g);
        t.dA_log = (float*)take(z.h);
        t.ddt_bias = (float*)take(z.h);
        t.dstate0 = (float*)take(z.st);
    }
    if (sl) *sl = t;
    return off;
}

gdn_status make_plan(const gdn_shape* s, int backward, Plan* p) {
    size_t saved = 0, ws = 0;
    gdn_status st = gdn_saved_bytes(s, &saved);  // validates the shape
    if (st != GDN_OK) return st;
    if (backward) {
        size_t w0 = 0, w1 = 0;
        if ((st = gdn_workspace_bytes(s, 0, &w0)) != GDN_OK) return st;
        if ((st = gdn_workspace_bytes(s, 1, &w1)) != GDN_OK) return st;
        ws = w0 > w1 ? w0 : w1;
    } else {
        saved = 0;  // inference: nothing is kept for a backward
        if ((st = gdn_workspace_bytes(s, 2, &ws)) != GDN_OK) return st;
    }
    p->slot_bytes = carve_slot(*s, backward, nullptr, nullptr);
    p->saved = align_up(saved);
    p->ws = align_up(ws);
    p->total = kSlots * p->slot_bytes + p->saved + p->ws;
    return GDN_OK;
}

}  // namespace

struct gdn_host_session {
    gdn_shape shape;
    int gates, backward;
    cudaStream_t compute, up, down;
    cudaEvent_t ev_in[kSlots], ev_in_b[kSlots], ev_fwd[kSlots], ev_bwd[kSlots], ev_free[kSlots];
    Slot slot[kSlots];
    void *saved, *ws;
    size_t saved_bytes, ws_bytes;
    int64_t step;
};

namespace {

void release(gdn_host_session* s) {
    for (int i = 0; i < kSlots; ++i) {
        cudaEvent_t* evs[] = {&s->ev_in[i], &s->ev_in_b[i], &s->ev_fwd[i], &s->ev_bwd[i],
                              &s->ev_free[i]};
        for (cudaEvent_t* e : evs)
            if (*e) cudaEventDestroy(*e);
    }
    if (s->up) cudaStreamDestroy(s->up);
    if (s->down) cudaStreamDestroy(s->down);
    std::free(s);
}

}  // namespace

extern "C" {

gdn_status gdn_host_session_bytes(const gdn_shape* shape, int32_t backward, size_t* bytes) {
    if (bytes == nullptr || (backward != 0 && backward != 1)) return GDN_ERR_INVALID_ARG;
    Plan p;
    gdn_status st = make_plan(shape, backward, &p);
    if (st != GDN_OK) return st;
    *bytes = p.total;
    return GDN_OK;
}

gdn_status gdn_host_session_create(const gdn_shape* shape, int32_t gates, int32_t backward,
                                   void* arena, size_t arena_bytes, void* stream,
                                   gdn_host_session** out) {
    if (out == nullptr || arena == nullptr || (gates != 0 && gates != 1) ||
        (backward != 0 && backward != 1))
        return GDN_ERR_INVALID_ARG;
    *out = nullptr;
    Plan p;
    gdn_status st = make_plan(shape, backward, &p);
    if (st != GDN_OK) return st;
    if ((reinterpret_cast<uintptr_t>(arena) & (kAlign - 1)) != 0) return GDN_ERR_MISALIGNED;
    if (arena_bytes < p.total) return GDN_ERR_WORKSPACE_TOO_SMALL;
    gdn_host_session* s = static_cast<gdn_host_session*>(std::calloc(1, sizeof(gdn_host_session)));
    if (s == nullptr) return GDN_ERR_INVALID_ARG;
    s->shape = *shape;
    s->gates = gates;
    s->backward = backward;
    s->compute = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(arena);
    for (int i = 0; i < kSlots; ++i) carve_slot(*shape, backward, base + i * p.slot_bytes, &s->slot[i]);
    s->saved = backward ? base + kSlots * p.slot_bytes : nullptr;
    s->saved_bytes = backward ? p.saved : 0;
    s->ws = base + kSlots * p.slot_bytes + p.saved;
    s->ws_bytes = p.ws;
    cudaError_t e = cudaStreamCreateWithFlags(&s->up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s->down, cudaStreamNonBlocking);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i) {
        cudaEvent_t* evs[] = {&s->ev_in[i], &s->ev_in_b[i], &s->ev_fwd[i], &s->ev_bwd[i],
                              &s->ev_free[i]};
        for (cudaEvent_t* ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        release(s);
        return (gdn_status)gdn::note_cuda_error(e);
    }
    *out = s;
    return GDN_OK;
}

gdn_status gdn_host_step(gdn_host_session* s, const gdn_host_inputs* in,
                         const gdn_host_outputs* out) {
    if (s == nullptr || in == nullptr || out == nullptr) return GDN_ERR_INVALID_ARG;
    const gdn_shape& sh = s->shape;
    const bool g0 = s->gates == 0;
    if (!in->q || !in->k || !in->v || !in->a || !in->b || !out->o || !out->state_T)
        return GDN_ERR_INVALID_ARG;
    if (g0 && (!in->A_log || !in->dt_bias)) return GDN_ERR_INVALID_ARG;
    if (sh.has_mask && !in->mask) return GDN_ERR_INVALID_ARG;
    if (s->backward) {
        if (!in->d_o || !out->dq || !out->dk || !out->dv || !out->da || !out->db || !out->dstate0)
            return GDN_ERR_INVALID_ARG;
        if (g0 && (!out->dA_log || !out->ddt_bias)) return GDN_ERR_INVALID_ARG;
    }
    const int sl = (int)(s->step % kSlots);
    const Slot& d = s->slot[sl];
    const Sizes z = sizes_of(sh);
    const uint8_t* mask = sh.has_mask ? d.mask : nullptr;
    const float* state0 = in->state0 ? d.state0 : nullptr;
    const float* dST = (s->backward && in->d_state_T) ? d.d_state_T : nullptr;

    // up: the slot's previous step (n - 3) must have released it (an event that
    // was never recorded counts as complete)
    cudaError_t e = cudaStreamWaitEvent(s->up, s->ev_free[sl], 0);
    auto h2d = [&](void* dst, const void* src, size_t n) {
        if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s->up);
    };
    auto d2h = [&](void* dst, const void* src, size_t n) {
        if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s->down);
    };
    auto record = [&](cudaEvent_t ev, cudaStream_t st) {
        if (e == cudaSuccess) e = cudaEventRecord(ev, st);
    };
    auto wait = [&](cudaStream_t st, cudaEvent_t ev) {
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev, 0);
    };
    h2d(d.q, in->q, z.q);
    h2d(d.k, in->k, z.q);
    h2d(d.v, in->v, z.v);
    h2d(d.a, in->a, z.g);
    h2d(d.b, in->b, z.g);
    if (g0) {
        h2d(d.A_log, in->A_log, z.h);
        h2d(d.dt_bias, in->dt_bias, z.h);
    }
    if (state0) h2d(d.state0, in->state0, z.st);
    if (mask) h2d(d.mask, in->mask, z.mask);
    record(s->ev_in[sl], s->up);
    if (s->backward) {
        h2d(d.d_o, in->d_o, z.v);
        if (dST) h2d(d.d_state_T, in->d_state_T, z.st);
        record(s->ev_in_b[sl], s->up);
    }
    wait(s->compute, s->ev_in[sl]);
    if (e != cudaSuccess) return (gdn_status)gdn::note_cuda_error(e);

    gdn_status st =
        g0 ? gdn_forward(&sh, d.q, d.k, d.v, d.a, d.b, d.A_log, d.dt_bias, state0, mask, d.o,
                         d.state_T, s->saved, s->saved_bytes, s->ws, s->ws_bytes, s->compute)
           : gdn_forward_lb(&sh, d.q, d.k, d.v, d.a, d.b, state0, mask, d.o, d.state_T, s->saved,
                            s->saved_bytes, s->ws, s->ws_bytes, s->compute);
    if (st != GDN_OK) return st;
    record(s->ev_fwd[sl], s->compute);
    wait(s->down, s->ev_fwd[sl]);
    d2h(out->o, d.o, z.v);
    d2h(out->state_T, d.state_T, z.st);
    if (s->backward) {
        wait(s->compute, s->ev_in_b[sl]);
        if (e != cudaSuccess) return (gdn_status)gdn::note_cuda_error(e);
        st = g0 ? gdn_backward(&sh, d.q, d.k, d.v, d.a, d.b, d.A_log, d.dt_bias, mask, s->saved,
                               s->saved_bytes, d.d_o, dST, d.dq, d.dk, d.dv, d.da, d.db, d.dA_log,
                               d.ddt_bias, d.dstate0, s->ws, s->ws_bytes, s->compute)
                : gdn_backward_lb(&sh, d.q, d.k, d.v, d.a, d.b, mask, s->saved, s->saved_bytes,
                                  d.d_o, dST, d.dq, d.dk, d.dv, d.da, d.db, d.dstate0, s->ws,
                                  s->ws_bytes, s->compute);
        if (st != GDN_OK) return st;
        record(s->ev_bwd[sl], s->compute);
        wait(s->down, s->ev_bwd[sl]);
        d2h(out->dq, d.dq, z.q);
        d2h(out->dk, d.dk, z.q);
        d2h(out->dv, d.dv, z.v);
        d2h(out->da, d.da, z.g);
        d2h(out->db, d.db, z.g);
        if (g0) {
            d2h(out->dA_log, d.dA_log, z.h);
            d2h(out->ddt_bias, d.ddt_bias, z.h);
        }
        d2h(out->dstate0, d.dstate0, z.st);
    }
    record(s->ev_free[sl], s->down);
    if (e != cudaSuccess) return (gdn_status)gdn::note_cuda_error(e);
    ++s->step;
    return GDN_OK;
}

gdn_status gdn_host_session_sync(gdn_host_session* s) {
    if (s == nullptr) return GDN_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(s->up);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s->compute);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s->down);
    return (gdn_status)gdn::note_cuda_error(e);
}

gdn_status gdn_host_session_destroy(gdn_host_session* s) {
    if (s == nullptr) return GDN_OK;
    const gdn_status st = gdn_host_session_sync(s);
    release(s);
    return st;
}

}  // extern "C"
