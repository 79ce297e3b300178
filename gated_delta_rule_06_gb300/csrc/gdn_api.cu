// gdn_api.cu -- the C ABI of include/gdn.h: argument validation, the layout
// of the `saved` and workspace buffers, and the launch sequence.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_internal.cuh"

namespace {

thread_local char g_cuda_err[256] = "no error";

std::atomic<uint64_t> g_launches{0};

// opt-in per-phase timing (gdn_timing_begin / gdn_timing_end)
struct PhaseEvent {
    const char* name;
    cudaEvent_t start, stop;
};
bool g_timing = false;
std::vector<PhaseEvent> g_events;

template <typename F>
cudaError_t run_phase(const char* name, cudaStream_t s, F&& launch) {
    if (!g_timing) return launch();
    PhaseEvent ev{name, nullptr, nullptr};
    cudaError_t e = cudaEventCreate(&ev.start);
    if (e == cudaSuccess) e = cudaEventCreate(&ev.stop);
    if (e == cudaSuccess) e = cudaEventRecord(ev.start, s);
    if (e != cudaSuccess) return e;
    e = launch();
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(ev.stop, s);
    g_events.push_back(ev);
    return e;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    // byte offsets into `saved`
    size_t ckpt, gam, beta, rq, rk, Tinv, W, P, Delta, kimg, qimg, saved_total;
    // byte offsets into the forward workspace
    size_t U, fwd_total;
    // byte offsets into the backward workspace
    size_t dSck, Dbar, dqh, dkh, dl, dbeta, part, sched, bwd_total;
};

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status validate_shape(const gdn_shape* s, gdn::Dims* d) {
    if (s == nullptr) return GDN_ERR_INVALID_ARG;
    if (s->dtype != GDN_DTYPE_F32 && s->dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARG;
    if (s->B < 1 || s->T < 1 || s->Hk < 1 || s->Hv < 1) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->Hv % s->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->Dk < 8 || s->Dk > 256 || s->Dk % 8 != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->Dv < 8 || s->Dv > 256 || s->Dv % 8 != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
    // grid dimensions: y <= 65535, z <= 65535
    if (s->Hv > 65535 || s->B > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->T > (int64_t(1) << 40) / 64) return GDN_ERR_UNSUPPORTED_SHAPE;
    d->B = s->B;
    d->T = s->T;
    d->Hk = s->Hk;
    d->Hv = s->Hv;
    d->Dk = s->Dk;
    d->Dv = s->Dv;
    d->G = s->Hv / s->Hk;
    d->NC = (s->T + gdn::kChunk - 1) / gdn::kChunk;
    d->Tp = d->NC * gdn::kChunk;
    d->dtype = s->dtype;
    if (d->NC > 2147483647LL) return GDN_ERR_UNSUPPORTED_SHAPE;
    return GDN_OK;
}

Layout make_layout(const gdn::Dims& d) {
    const size_t es = d.dtype == GDN_DTYPE_BF16 ? 2 : 4;
    // the tensor-core path keeps checkpoints, T, the state cotangents and Dbar
    // as bf16 operand images (half the fp32 size)
    const size_t img = gdn::tc_path(d) ? 2 : 4;
    const size_t BH = (size_t)d.B * d.Hv;
    const size_t state_ck = BH * d.NC * d.Dk * d.Dv * img;
    const size_t perstep = BH * d.Tp;
    Layout L{};
    size_t o = 0;
    L.ckpt = o; o = align_up(o + state_ck);
    L.gam = o; o = align_up(o + perstep * 8);
    L.beta = o; o = align_up(o + perstep * 4);
    L.rq = o; o = align_up(o + (size_t)d.B * d.Hk * d.Tp * 4);
    L.rk = o; o = align_up(o + (size_t)d.B * d.Hk * d.Tp * 4);
    L.Tinv = o; o = align_up(o + BH * d.NC * gdn::kChunk * gdn::kChunk * img);
    L.W = o; o = align_up(o + perstep * d.Dk * es);
    L.P = o; o = align_up(o + BH * d.NC * gdn::kChunk * gdn::kChunk * es);
    L.Delta = o; o = align_up(o + perstep * d.Dv * 4);
    const size_t qk_img = img == 2 ? (size_t)d.B * d.Hk * d.Tp * d.Dk * 2 : 0;
    L.kimg = o; o = align_up(o + qk_img);
    L.qimg = o; o = align_up(o + qk_img);
    L.saved_total = o;
    o = 0;
    L.U = o; o = align_up(o + perstep * d.Dv * 4);
    L.fwd_total = o;
    o = 0;
    L.dSck = o; o = align_up(o + state_ck);
    L.Dbar = o; o = align_up(o + perstep * d.Dv * img);
    // per-value-head q / k cotangents: bf16 on the tensor-core path, else fp32
    L.dqh = o; o = align_up(o + perstep * d.Dk * img);
    L.dkh = o; o = align_up(o + perstep * d.Dk * img);
    L.dl = o; o = align_up(o + perstep * 4);
    L.dbeta = o; o = align_up(o + perstep * 4);
    L.part = o; o = align_up(o + 2 * (size_t)d.B * d.NC * d.Hv * 4);
    L.sched = o; o = align_up(o + (1 + (size_t)d.B * d.Hv) * 4);  // item counter, progress
    L.bwd_total = o;
    return L;
}

void carve_saved(const Layout& L, void* saved, gdn::Ptrs* p) {
    char* s = static_cast<char*>(saved);
    p->ckpt = reinterpret_cast<float*>(s + L.ckpt);
    p->gam = reinterpret_cast<double*>(s + L.gam);
    p->beta = reinterpret_cast<float*>(s + L.beta);
    p->rq = reinterpret_cast<float*>(s + L.rq);
    p->rk = reinterpret_cast<float*>(s + L.rk);
    p->Tinv = reinterpret_cast<float*>(s + L.Tinv);
    p->W = s + L.W;
    p->P = s + L.P;
    p->Delta = reinterpret_cast<float*>(s + L.Delta);
    p->kimg = s + L.kimg;
    p->qimg = s + L.qimg;
}

// Compressed chunk states (rank-r factors in place of the checkpoint images).
// saved: the other saved regions of make_layout moved down to offset 0, then the
// initial state (fp32) and the factors Q [B][Hv][NC][Dk][r], R [B][Hv][NC][r][Dv]
// (fp32; slot 0 unused).  Forward workspace: make_layout's, then the checkpoint
// images the scan writes (not kept) and two fp32 state buffers (the chunk-end
// state and the truncated one).  Backward workspace: make_layout's and the
// segment buffers of its automatic count, then the images rebuilt from the
// factors.
struct CLayout {
    Layout L;  // saved offsets moved down (ckpt unused)
    size_t S0f, Qf, Rf, saved_total;
    size_t img, stA, stB, fwd_total;
    size_t bimg, bwd_total;
};

CLayout make_clayout(const gdn::Dims& d, int rank, size_t bwd_seg_bytes) {
    CLayout C{};
    C.L = make_layout(d);
    Layout& L = C.L;
    const size_t sh = L.gam;  // the checkpoint images come first
    L.ckpt = 0;
    for (size_t* o : {&L.gam, &L.beta, &L.rq, &L.rk, &L.Tinv, &L.W, &L.P, &L.Delta, &L.kimg, &L.qimg})
        *o -= sh;
    const size_t BH = (size_t)d.B * d.Hv;
    const size_t st = BH * d.Dk * d.Dv * 4;
    const size_t imgb = BH * d.NC * d.Dk * d.Dv * 2;
    C.S0f = L.saved_total - sh;
    C.Qf = align_up(C.S0f + st);
    C.Rf = align_up(C.Qf + BH * d.NC * d.Dk * rank * 4);
    C.saved_total = align_up(C.Rf + BH * d.NC * rank * d.Dv * 4);
    C.img = L.fwd_total;
    C.stA = align_up(C.img + imgb);
    C.stB = align_up(C.stA + st);
    C.fwd_total = align_up(C.stB + st);
    C.bimg = align_up(L.bwd_total + bwd_seg_bytes);
    C.bwd_total = align_up(C.bimg + imgb);
    return C;
}

// tensor maps of v (and dO, o, U) for the tensor-core kernels: full-width
// 64-row tiles, dO in tiles of at most 128 columns (the scans' value tile)
bool make_tmaps(const gdn::Dims& d, const void* v, const void* dO, const void* o, const void* U,
                gdn::Tmaps* m) {
    std::memset(m, 0, sizeof(*m));
    const int vt = (int)(d.Dv < 128 ? d.Dv : 128);
    bool ok = gdn::encode_row_tile_map(&m->v, v, d.B, d.T, d.Hv, d.Dv, (int)d.Dv);
    if (ok && dO)
        ok = gdn::encode_row_tile_map(&m->dO, dO, d.B, d.T, d.Hv, d.Dv, vt) &&
             gdn::encode_row_tile_map(&m->dOf, dO, d.B, d.T, d.Hv, d.Dv, (int)d.Dv);
    if (ok && o) ok = gdn::encode_row_major_map(&m->o, o, d.B, d.T, d.Hv * d.Dv, vt);
    if (ok && U) ok = gdn::encode_f32_rows_map(&m->U, U, d.B * d.Hv * d.Tp, d.Dv, vt);
    if (ok && U && d.Dv % 32 == 0) ok = gdn::encode_f32_rows_map_sw128(&m->Us, U, d.B * d.Hv * d.Tp, d.Dv);
    return ok;
}

gdn_status tmap_error() {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "cuTensorMapEncodeTiled refused a tensor map");
    return GDN_ERR_CUDA;
}

gdn_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return GDN_ERR_CUDA;
}

}  // namespace

namespace gdn {
int note_cuda_error(cudaError_t e) { return (int)cuda_status(e); }
int sm_count() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < kMaxDev) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev >= 0 && dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// the driver's tensor-map encoder, resolved once through the runtime
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return encode;
}

bool encode_row_tile_map(CUtensorMap* m, const void* base, int64_t B, int64_t T, int64_t H,
                         int64_t D, int cols) {
    const auto encode = tensor_map_encoder();
    if (encode == nullptr || cols % 8 || cols < 8 || cols > 256 || D % 8) return false;
    const cuuint64_t dims[5] = {8, (cuuint64_t)T, (cuuint64_t)(D / 8), (cuuint64_t)H, (cuuint64_t)B};
    // byte strides of dims 1..4: row, 8-column group, head, batch
    const cuuint64_t strides[4] = {(cuuint64_t)(H * D * 2), 16, (cuuint64_t)(D * 2),
                                   (cuuint64_t)(T * H * D * 2)};
    const cuuint32_t box[5] = {8, (cuuint32_t)kChunk, (cuuint32_t)(cols / 8), 1, 1};
    const cuuint32_t unit[5] = {1, 1, 1, 1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
                  unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_row_major_map(CUtensorMap* m, const void* base, int64_t B, int64_t T, int64_t rowlen,
                          int cols) {
    const auto encode = tensor_map_encoder();
    if (encode == nullptr || cols % 8 || cols < 8 || cols > 256 || rowlen % 8) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)rowlen, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)(rowlen * 2), (cuuint64_t)(T * rowlen * 2)};
    const cuuint32_t box[3] = {(cuuint32_t)cols, (cuuint32_t)kChunk, 1};
    const cuuint32_t unit[3] = {1, 1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols_total, int cols) {
    const auto encode = tensor_map_encoder();
    if (encode == nullptr || cols % 4 || cols < 4 || cols > 256 || cols_total % 4) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols_total, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(cols_total * 4)};
    const cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)kChunk};
    const cuuint32_t unit[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                  unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32_rows_map_sw128(CUtensorMap* m, const void* base, int64_t rows, int64_t cols_total) {
    const auto encode = tensor_map_encoder();
    if (encode == nullptr || cols_total % 32) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols_total, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(cols_total * 4)};
    const cuuint32_t box[2] = {32, (cuuint32_t)kChunk};
    const cuuint32_t unit[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                  unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_path(const Dims& d) {
    return d.dtype == GDN_DTYPE_BF16 && fwd_chunk_tc_supported(d) && scan_tc_supported(d) &&
           bwd_chunk_tc_supported(d);
}
void count_launches(int n) { g_launches.fetch_add((uint64_t)n); }
unsigned int read_clear_error_bwdr();  // the streamed q / k reduction (gdn_bwd.cu)
unsigned int read_clear_error_all() {
    const unsigned int words[] = {read_clear_error_selftest(), read_clear_error_bwdtc(),
                                  read_clear_error_scantc(), read_clear_error_fwdtc(),
                                  read_clear_error_scanta(), read_clear_error_decode(),
                                  read_clear_error_kctc(), read_clear_error_bwdr()};
    unsigned int v = 0;
    for (unsigned int w : words) {
        if (w == ~0u) return ~0u;
        v |= w;
    }
    return v;
}
}  // namespace gdn

namespace {
// ---- segmented forward scan: sizing and the automatic segment count -------------
bool seg_supported(const gdn::Dims& d) { return gdn::tc_path(d) && gdn::scan_ta_supported(d); }

// segments actually formed from a requested count: len chunks each, none empty
void seg_geometry(const gdn::Dims& d, int requested, int* nseg, int* len) {
    int64_t r = requested < 1 ? 1 : requested;
    if (r > d.NC) r = d.NC;
    const int64_t l = (d.NC + r - 1) / r;
    *len = (int)l;
    *nseg = (int)((d.NC + l - 1) / l);
}

// extra forward workspace of nseg segments: the maps [nseg - 1][B][Hv][Dk][Wd] and
// the chained start states [nseg - 1][B][Hv][Dk][Dv], fp32
size_t seg_bytes(const gdn::Dims& d, int nseg) {
    if (nseg <= 1) return 0;
    const size_t n = (size_t)(nseg - 1) * d.B * d.Hv * d.Dk;
    return align_up(n * gdn::seg_map_width(d) * 4) + align_up(n * d.Dv * 4);
}

// Segment count that minimises the modelled critical path, in units of one chunk
// step of the scan: the plain scan takes waves(B Hv Dv/128) NC; with P segments of
// L chunks, the maps take waves((P - 1) B Hv Wd/128) L, the chain (P - 1) steps of
// about (Dk / 128)^2 chunk steps each (measured on GB300) and the scan proper
// waves(P B Hv Dv/128) L, plus two launches (about one step each).
int seg_auto(const gdn::Dims& d) {
    if (!seg_supported(d)) return 1;
    const int64_t sms = gdn::sm_count();
    auto waves = [&](int64_t ctas) { return (double)((ctas + sms - 1) / sms); };
    const int64_t tiles = d.B * d.Hv * (d.Dv / 128), mtiles = d.B * d.Hv * (gdn::seg_map_width(d) / 128);
    double best = waves(tiles) * (double)d.NC;
    const double chain = (double)(d.Dk * d.Dk) / (128.0 * 128.0);
    int best_p = 1;
    const int64_t pmax = d.NC < 4096 ? d.NC : 4096;
    for (int64_t r = 2; r <= pmax; ++r) {
        int nseg = 1, len = 1;
        seg_geometry(d, (int)r, &nseg, &len);
        if ((int64_t)nseg * d.B > 65535) break;
        const double cost = (waves((nseg - 1) * mtiles) + waves(nseg * tiles)) * len + chain * (nseg - 1) + 2.0;
        if (cost < best) {
            best = cost;
            best_p = nseg;
        }
    }
    return best_p;
}

// The backward's segment count.  Same model for the reverse scan, plus the
// per-chunk gradient items (about 7.8 Dk / 192 chunk steps of one SM each,
// measured on GB300): with one segment they run in the fused launch beside the
// scan (or after it when the scan's tiles fill the GPU); with several, after the
// segmented scan on every SM.
int seg_auto_bwd(const gdn::Dims& d) {
    if (!seg_supported(d)) return 1;
    const int64_t sms = gdn::sm_count();
    auto waves = [&](int64_t ctas) { return (double)((ctas + sms - 1) / sms); };
    const int64_t tiles = d.B * d.Hv * (d.Dv / 128), mtiles = d.B * d.Hv * (gdn::seg_map_width(d) / 128);
    const double items = (double)(d.B * d.Hv * d.NC), item = 7.8 * (double)d.Dk / 192.0;
    const double grads = waves(d.B * d.Hv * d.NC) * item;
    double best = gdn::bwd_fused_tc_supported(d)
                      ? std::max((double)d.NC, (items * item + (double)(tiles * d.NC)) / (double)sms)
                      : waves(tiles) * (double)d.NC + grads;
    int best_p = 1;
    const double chain = (double)(d.Dk * d.Dk) / (128.0 * 128.0);
    const int64_t pmax = d.NC < 4096 ? d.NC : 4096;
    for (int64_t r = 2; r <= pmax; ++r) {
        int nseg = 1, len = 1;
        seg_geometry(d, (int)r, &nseg, &len);
        if ((int64_t)nseg * d.B > 65535) break;
        const double cost = (waves((nseg - 1) * mtiles) + waves(nseg * tiles)) * len + chain * (nseg - 1) +
                            grads + 3.0;
        if (cost < best) {
            best = cost;
            best_p = nseg;
        }
    }
    return best_p;
}

// segments and chunks per segment a request resolves to (0: the automatic count
// of the forward, or of the backward when bwd)
int seg_resolve(const gdn::Dims& d, int requested, int* len, bool bwd = false) {
    if (requested == 0) requested = bwd ? seg_auto_bwd(d) : seg_auto(d);
    int nseg = 1;
    *len = (int)d.NC;
    if (requested > 1) seg_geometry(d, requested, &nseg, len);
    return nseg;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null pointer or bad enum value";
        case GDN_ERR_UNSUPPORTED_SHAPE: return "GDN_ERR_UNSUPPORTED_SHAPE: shape outside the supported set";
        case GDN_ERR_WORKSPACE_TOO_SMALL: return "GDN_ERR_WORKSPACE_TOO_SMALL: workspace or saved buffer too small";
        case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a kernel launch failed";
    }
    return "unknown gdn_status";
}

const char* gdn_last_cuda_error(void) { return g_cuda_err; }

gdn_status gdn_workspace_bytes(const gdn_shape* shape, int pass, size_t* bytes) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (bytes == nullptr || pass < 0 || pass > 2) return GDN_ERR_INVALID_ARG;
    const Layout L = make_layout(d);
    // the segment buffers of the pass's automatic segment count
    int len = 0;
    const size_t seg = seg_bytes(d, seg_resolve(d, 0, &len, pass == 1));
    if (pass == 0) *bytes = L.fwd_total + seg;
    else if (pass == 1) *bytes = L.bwd_total + seg;
    else *bytes = L.fwd_total + L.saved_total + seg;  // inference forward without a saved buffer
    return GDN_OK;
}

gdn_status gdn_saved_bytes(const gdn_shape* shape, size_t* bytes) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (bytes == nullptr) return GDN_ERR_INVALID_ARG;
    *bytes = make_layout(d).saved_total;
    return GDN_OK;
}

namespace {
// gdn_forward and gdn_forward_lb: gates = 0 takes (a, b, A_log, dt_bias), 1 takes
// (log_decay, beta) in a, b
gdn_status forward_impl(const gdn_shape* shape, int gates, const void* q, const void* k,
                        const void* v, const void* a, const void* b, const float* A_log,
                        const float* dt_bias, const float* state0, const uint8_t* mask, void* o,
                        float* state_T, void* saved, size_t saved_bytes, void* ws,
                        size_t ws_bytes, void* stream, int segments = 1) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    d.gates = gates;
    // segments of the scan (1: the plain sequential scan; 0: the automatic choice)
    if (segments < 0) return GDN_ERR_INVALID_ARG;
    if (segments > 1 && !seg_supported(d)) return GDN_ERR_UNSUPPORTED_SHAPE;
    int len = 0;
    const int nseg = seg_resolve(d, segments, &len);
    if ((int64_t)nseg * d.B > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;
    const size_t sbytes = seg_bytes(d, nseg);
    if (!q || !k || !v || !a || !b || !o || !state_T) return GDN_ERR_INVALID_ARG;
    if (gates == 0 && (!A_log || !dt_bias)) return GDN_ERR_INVALID_ARG;
    if (shape->has_mask && !mask) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, b, A_log, dt_bias, state0, mask, o, state_T, saved, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::Ptrs p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias; p.state0 = state0;
    p.mask = shape->has_mask ? mask : nullptr;
    p.o = o; p.state_T = state_T;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Layout L = make_layout(d);
    if (saved == nullptr && d.T == 1 && gdn::decode_supported(d.Dk, d.Dv))
        return cuda_status(run_phase("decode", s, [&] { return gdn::launch_decode(d, p, s); }));
    char* wsb = static_cast<char*>(ws);
    size_t used = L.fwd_total;  // the segment buffers follow the workspace proper
    if (saved != nullptr) {
        if (saved_bytes < L.saved_total) return GDN_ERR_WORKSPACE_TOO_SMALL;
        if (ws == nullptr) return GDN_ERR_INVALID_ARG;
        if (ws_bytes < L.fwd_total + sbytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
        carve_saved(L, saved, &p);
    } else {
        if (ws == nullptr) return GDN_ERR_INVALID_ARG;
        if (ws_bytes < L.fwd_total + L.saved_total + sbytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
        carve_saved(L, wsb + L.fwd_total, &p);
        used += L.saved_total;
    }
    p.U = reinterpret_cast<float*>(wsb + L.U);
    gdn::Tmaps maps;
    if (gdn::tc_path(d)) {
        if (!make_tmaps(d, v, nullptr, o, p.U, &maps)) return tmap_error();
        p.tmaps = &maps;
    }
    cudaError_t e = run_phase("prep", s, [&] { return gdn::launch_prep(d, p, s); });
    if (e == cudaSuccess) e = run_phase("fwd_chunk", s, [&] { return gdn::launch_fwd_chunk(d, p, s); });
    if (e == cudaSuccess && nseg > 1) {
        // segment maps, their chain, then every segment's scan at once
        const size_t nmap = (size_t)(nseg - 1) * d.B * d.Hv * d.Dk;
        gdn::ScanSeg sg{nseg, len, 1, reinterpret_cast<float*>(wsb + used + align_up(nmap * gdn::seg_map_width(d) * 4)),
                        reinterpret_cast<float*>(wsb + used)};
        e = run_phase("fwd_seg_maps", s, [&] { return gdn::launch_fwd_scan_ta_seg(d, p, sg, s); });
        if (e == cudaSuccess) e = run_phase("fwd_seg_chain", s, [&] { return gdn::launch_seg_chain(d, p, sg, s); });
        sg.mode = 0;
        if (e == cudaSuccess) e = run_phase("fwd_scan", s, [&] { return gdn::launch_fwd_scan_ta_seg(d, p, sg, s); });
    } else if (e == cudaSuccess) {
        e = run_phase("fwd_scan", s, [&] { return gdn::launch_fwd_scan(d, p, s); });
    }
    return cuda_status(e);
}

// gdn_backward and gdn_backward_lb (gates as in forward_impl; with gates = 1, da
// and db receive the log_decay and beta cotangents and dA_log, ddt_bias are unused)
gdn_status backward_impl(const gdn_shape* shape, int gates, const void* q, const void* k,
                         const void* v, const void* a, const void* b, const float* A_log,
                         const float* dt_bias, const uint8_t* mask, const void* saved,
                         size_t saved_bytes, const void* d_o, const float* d_state_T, void* dq,
                         void* dk, void* dv, void* da, void* db, float* dA_log, float* ddt_bias,
                         float* dstate0, void* ws, size_t ws_bytes, void* stream, int segments = 0,
                         int rank = 0) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    d.gates = gates;
    // rank > 0: the saved buffer of gdn_forward_compressed (factors in place of
    // the checkpoint images; the images are rebuilt into the workspace first)
    if (rank > 0 && (gates != 0 || !gdn::tc_path(d) || !seg_supported(d) ||
                     !gdn::compress_supported(d, rank, 0)))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    // segments of the reverse scan (1: one pass, fused with the gradients when it
    // fits; 0: the automatic choice)
    if (segments < 0) return GDN_ERR_INVALID_ARG;
    if (segments > 1 && !seg_supported(d)) return GDN_ERR_UNSUPPORTED_SHAPE;
    int len = 0;
    const int nseg = seg_resolve(d, segments, &len, true);
    if ((int64_t)nseg * d.B > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;
    const size_t sbytes = seg_bytes(d, nseg);
    if (!q || !k || !v || !a || !b || !saved || !d_o || !dq || !dk || !dv || !da || !db ||
        !dstate0 || !ws)
        return GDN_ERR_INVALID_ARG;
    if (gates == 0 && (!A_log || !dt_bias || !dA_log || !ddt_bias)) return GDN_ERR_INVALID_ARG;
    if (shape->has_mask && !mask) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, b, A_log, dt_bias, mask, saved, d_o, d_state_T, dq, dk,
                          dv, da, db, dA_log, ddt_bias, dstate0, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    const Layout L = make_layout(d);
    const CLayout C = make_clayout(d, rank > 0 ? rank : 1, sbytes);
    if (rank > 0) {
        if (saved_bytes < C.saved_total || ws_bytes < C.bwd_total) return GDN_ERR_WORKSPACE_TOO_SMALL;
    } else if (saved_bytes < L.saved_total || ws_bytes < L.bwd_total + sbytes) {
        return GDN_ERR_WORKSPACE_TOO_SMALL;
    }
    gdn::Ptrs p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.mask = shape->has_mask ? mask : nullptr;
    carve_saved(rank > 0 ? C.L : L, const_cast<void*>(saved), &p);
    if (rank > 0) p.ckpt = reinterpret_cast<float*>(static_cast<char*>(ws) + C.bimg);
    p.d_o = d_o; p.d_state_T = d_state_T;
    p.dq = dq; p.dk = dk; p.dv = dv; p.da = da; p.db = db;
    p.dA_log = dA_log; p.ddt_bias = ddt_bias; p.dstate0 = dstate0;
    char* w = static_cast<char*>(ws);
    p.dSck = reinterpret_cast<float*>(w + L.dSck);
    p.Dbar = reinterpret_cast<float*>(w + L.Dbar);
    p.dqh = reinterpret_cast<float*>(w + L.dqh);
    p.dkh = reinterpret_cast<float*>(w + L.dkh);
    p.dl = reinterpret_cast<float*>(w + L.dl);
    p.dbeta = reinterpret_cast<float*>(w + L.dbeta);
    p.part = reinterpret_cast<float*>(w + L.part);
    p.sched = reinterpret_cast<unsigned int*>(w + L.sched);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gdn::Tmaps maps;
    if (gdn::tc_path(d)) {
        if (!make_tmaps(d, v, d_o, nullptr, nullptr, &maps)) return tmap_error();
        p.tmaps = &maps;
    }
    cudaError_t e = cudaSuccess;
    if (rank > 0) {
        const char* sv = static_cast<const char*>(saved);
        e = run_phase("expand", s, [&] {
            return gdn::launch_expand_ckpt(d, reinterpret_cast<const float*>(sv + C.S0f),
                                           reinterpret_cast<const float*>(sv + C.Qf),
                                           reinterpret_cast<const float*>(sv + C.Rf), rank, p.ckpt, s);
        });
    }
    if (e != cudaSuccess) {
    } else if (nseg > 1) {
        // segment maps, their chain from d_state_T, every segment's reverse scan,
        // then the per-chunk gradients on every SM
        const size_t nmap = (size_t)(nseg - 1) * d.B * d.Hv * d.Dk;
        gdn::ScanSeg sg{nseg, len, 1, reinterpret_cast<float*>(w + L.bwd_total + align_up(nmap * gdn::seg_map_width(d) * 4)),
                        reinterpret_cast<float*>(w + L.bwd_total)};
        gdn::Ptrs pc = p;
        pc.state0 = d_state_T;
        e = run_phase("bwd_seg_maps", s, [&] { return gdn::launch_bwd_scan_ta_seg(d, p, sg, s); });
        if (e == cudaSuccess) e = run_phase("bwd_seg_chain", s, [&] { return gdn::launch_seg_chain(d, pc, sg, s); });
        sg.mode = 0;
        if (e == cudaSuccess) e = run_phase("bwd_scan", s, [&] { return gdn::launch_bwd_scan_ta_seg(d, p, sg, s); });
        if (e == cudaSuccess) e = run_phase("bwd_chunk", s, [&] { return gdn::launch_bwd_chunk(d, p, s); });
    } else if (p.tmaps && gdn::bwd_fused_tc_supported(d)) {
        e = run_phase("bwd_scan_chunk", s, [&] { return gdn::launch_bwd_fused_tc(d, p, s); });
    } else {
        e = run_phase("bwd_scan", s, [&] { return gdn::launch_bwd_scan(d, p, s); });
        if (e == cudaSuccess) e = run_phase("bwd_chunk", s, [&] { return gdn::launch_bwd_chunk(d, p, s); });
    }
    if (e == cudaSuccess) e = run_phase("bwd_reduce", s, [&] { return gdn::launch_bwd_reduce(d, p, s); });
    return cuda_status(e);
}

// gdn_forward_compressed: prep and the chunk-local products as in forward_impl,
// then the scan one chunk at a time, the state truncated to rank r between
// chunks (the truncated state is the next chunk's start state; its factors are
// saved)
gdn_status forward_compressed_impl(const gdn_shape* shape, int rank, int iters, const float* omega,
                                   const void* q, const void* k, const void* v, const void* a,
                                   const void* b, const float* A_log, const float* dt_bias,
                                   const float* state0, const uint8_t* mask, void* o,
                                   float* state_T, void* saved, size_t saved_bytes, void* ws,
                                   size_t ws_bytes, void* stream) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (!gdn::tc_path(d) || !seg_supported(d) || !gdn::compress_supported(d, rank, iters))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !o || !state_T || !saved || !ws || !omega)
        return GDN_ERR_INVALID_ARG;
    if (shape->has_mask && !mask) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, b, A_log, dt_bias, state0, mask, o, state_T, saved, ws, omega};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return GDN_ERR_MISALIGNED;
    const CLayout C = make_clayout(d, rank, 0);
    if (saved_bytes < C.saved_total || ws_bytes < C.fwd_total) return GDN_ERR_WORKSPACE_TOO_SMALL;
    gdn::Ptrs p{};
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b;
    p.A_log = A_log; p.dt_bias = dt_bias; p.state0 = state0;
    p.mask = shape->has_mask ? mask : nullptr;
    p.o = o; p.state_T = state_T;
    carve_saved(C.L, saved, &p);
    char* wsb = static_cast<char*>(ws);
    char* sv = static_cast<char*>(saved);
    p.ckpt = reinterpret_cast<float*>(wsb + C.img);
    p.U = reinterpret_cast<float*>(wsb + C.L.U);
    float* S0f = reinterpret_cast<float*>(sv + C.S0f);
    float* Qf = reinterpret_cast<float*>(sv + C.Qf);
    float* Rf = reinterpret_cast<float*>(sv + C.Rf);
    float* stA = reinterpret_cast<float*>(wsb + C.stA);  // truncated state: next chunk's start
    float* stB = reinterpret_cast<float*>(wsb + C.stB);  // chunk-end state
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gdn::Tmaps maps;
    if (!make_tmaps(d, v, nullptr, o, p.U, &maps)) return tmap_error();
    p.tmaps = &maps;
    const size_t stbytes = (size_t)d.B * d.Hv * d.Dk * d.Dv * 4;
    cudaError_t e = state0 ? cudaMemcpyAsync(S0f, state0, stbytes, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(S0f, 0, stbytes, s);
    if (e == cudaSuccess) e = run_phase("prep", s, [&] { return gdn::launch_prep(d, p, s); });
    if (e == cudaSuccess) e = run_phase("fwd_chunk", s, [&] { return gdn::launch_fwd_chunk(d, p, s); });
    for (int64_t c = 0; c < d.NC && e == cudaSuccess; ++c) {
        gdn::ScanSeg sg{(int)d.NC, 1, 0, nullptr, nullptr};
        sg.first = (int)c;
        sg.sin = c > 0 ? stA : nullptr;            // chunk 0 starts from state0
        sg.sout = c + 1 < d.NC ? stB : nullptr;    // the last chunk writes state_T
        e = run_phase("fwd_scan", s, [&] { return gdn::launch_fwd_scan_ta_one(d, p, sg, s); });
        if (e == cudaSuccess && c + 1 < d.NC)
            e = run_phase("compress", s, [&] {
                return gdn::launch_trunc(d, stB, omega, rank, iters, stA, Qf, Rf, c + 1, s);
            });
    }
    return cuda_status(e);
}
}  // namespace

gdn_status gdn_checkpoint_bytes(const gdn_shape* shape, size_t* bytes) {
    return gdn_saved_bytes(shape, bytes);
}

gdn_status gdn_forward(const gdn_shape* shape, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log, const float* dt_bias,
                       const float* state0, const uint8_t* mask, void* o, float* state_T,
                       void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                       void* stream) {
    return forward_impl(shape, 0, q, k, v, a, b, A_log, dt_bias, state0, mask, o, state_T, saved,
                        saved_bytes, ws, ws_bytes, stream, 0);
}

gdn_status gdn_forward_lb(const gdn_shape* shape, const void* q, const void* k, const void* v,
                          const void* log_decay, const void* beta, const float* state0,
                          const uint8_t* mask, void* o, float* state_T, void* saved,
                          size_t saved_bytes, void* ws, size_t ws_bytes, void* stream) {
    return forward_impl(shape, 1, q, k, v, log_decay, beta, nullptr, nullptr, state0, mask, o,
                        state_T, saved, saved_bytes, ws, ws_bytes, stream, 0);
}

gdn_status gdn_segments_auto(const gdn_shape* shape, int* segments) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (segments == nullptr) return GDN_ERR_INVALID_ARG;
    int len = 0;
    *segments = seg_resolve(d, 0, &len);
    return GDN_OK;
}

gdn_status gdn_backward_segments_auto(const gdn_shape* shape, int* segments) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (segments == nullptr) return GDN_ERR_INVALID_ARG;
    int len = 0;
    *segments = seg_resolve(d, 0, &len, true);
    return GDN_OK;
}

gdn_status gdn_segment_bytes(const gdn_shape* shape, int segments, size_t* bytes) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (bytes == nullptr || segments < 0) return GDN_ERR_INVALID_ARG;
    if (segments > 1 && !seg_supported(d)) return GDN_ERR_UNSUPPORTED_SHAPE;
    int len = 0;
    *bytes = seg_bytes(d, seg_resolve(d, segments, &len));
    return GDN_OK;
}

gdn_status gdn_forward_segmented(const gdn_shape* shape, int segments, const void* q,
                                 const void* k, const void* v, const void* a, const void* b,
                                 const float* A_log, const float* dt_bias, const float* state0,
                                 const uint8_t* mask, void* o, float* state_T, void* saved,
                                 size_t saved_bytes, void* ws, size_t ws_bytes, void* stream) {
    return forward_impl(shape, 0, q, k, v, a, b, A_log, dt_bias, state0, mask, o, state_T, saved,
                        saved_bytes, ws, ws_bytes, stream, segments);
}

gdn_status gdn_backward(const gdn_shape* shape, const void* q, const void* k, const void* v,
                        const void* a, const void* b, const float* A_log, const float* dt_bias,
                        const uint8_t* mask, const void* saved, size_t saved_bytes,
                        const void* d_o, const float* d_state_T, void* dq, void* dk, void* dv,
                        void* da, void* db, float* dA_log, float* ddt_bias, float* dstate0,
                        void* ws, size_t ws_bytes, void* stream) {
    return backward_impl(shape, 0, q, k, v, a, b, A_log, dt_bias, mask, saved, saved_bytes, d_o,
                         d_state_T, dq, dk, dv, da, db, dA_log, ddt_bias, dstate0, ws, ws_bytes,
                         stream);
}

gdn_status gdn_backward_segmented(const gdn_shape* shape, int segments, const void* q,
                                  const void* k, const void* v, const void* a, const void* b,
                                  const float* A_log, const float* dt_bias, const uint8_t* mask,
                                  const void* saved, size_t saved_bytes, const void* d_o,
                                  const float* d_state_T, void* dq, void* dk, void* dv, void* da,
                                  void* db, float* dA_log, float* ddt_bias, float* dstate0,
                                  void* ws, size_t ws_bytes, void* stream) {
    return backward_impl(shape, 0, q, k, v, a, b, A_log, dt_bias, mask, saved, saved_bytes, d_o,
                         d_state_T, dq, dk, dv, da, db, dA_log, ddt_bias, dstate0, ws, ws_bytes,
                         stream, segments);
}

gdn_status gdn_compressed_bytes(const gdn_shape* shape, int rank, size_t* saved_bytes,
                                size_t* fwd_ws_bytes, size_t* bwd_ws_bytes) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (!saved_bytes || !fwd_ws_bytes || !bwd_ws_bytes) return GDN_ERR_INVALID_ARG;
    if (!gdn::tc_path(d) || !seg_supported(d) || !gdn::compress_supported(d, rank, 0))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    int len = 0;
    const CLayout C = make_clayout(d, rank, seg_bytes(d, seg_resolve(d, 0, &len, true)));
    *saved_bytes = C.saved_total;
    *fwd_ws_bytes = C.fwd_total;
    *bwd_ws_bytes = C.bwd_total;
    return GDN_OK;
}

gdn_status gdn_forward_compressed(const gdn_shape* shape, int rank, int iters, const float* omega,
                                  const void* q, const void* k, const void* v, const void* a,
                                  const void* b, const float* A_log, const float* dt_bias,
                                  const float* state0, const uint8_t* mask, void* o, float* state_T,
                                  void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                                  void* stream) {
    return forward_compressed_impl(shape, rank, iters, omega, q, k, v, a, b, A_log, dt_bias, state0,
                                   mask, o, state_T, saved, saved_bytes, ws, ws_bytes, stream);
}

gdn_status gdn_backward_compressed(const gdn_shape* shape, int rank, const void* q, const void* k,
                                   const void* v, const void* a, const void* b, const float* A_log,
                                   const float* dt_bias, const uint8_t* mask, const void* saved,
                                   size_t saved_bytes, const void* d_o, const float* d_state_T,
                                   void* dq, void* dk, void* dv, void* da, void* db, float* dA_log,
                                   float* ddt_bias, float* dstate0, void* ws, size_t ws_bytes,
                                   void* stream) {
    if (rank < 1) return GDN_ERR_INVALID_ARG;
    return backward_impl(shape, 0, q, k, v, a, b, A_log, dt_bias, mask, saved, saved_bytes, d_o,
                         d_state_T, dq, dk, dv, da, db, dA_log, ddt_bias, dstate0, ws, ws_bytes,
                         stream, 0, rank);
}

gdn_status gdn_backward_lb(const gdn_shape* shape, const void* q, const void* k,
                           const void* v, const void* log_decay, const void* beta,
                           const uint8_t* mask, const void* saved, size_t saved_bytes,
                           const void* d_o, const float* d_state_T, void* dq, void* dk,
                           void* dv, void* d_log_decay, void* d_beta, float* dstate0,
                           void* ws, size_t ws_bytes, void* stream) {
    return backward_impl(shape, 1, q, k, v, log_decay, beta, nullptr, nullptr, mask, saved,
                         saved_bytes, d_o, d_state_T, dq, dk, dv, d_log_decay, d_beta, nullptr,
                         nullptr, dstate0, ws, ws_bytes, stream);
}

/* ---- per-key-channel gates ---------------------------------------------------- */
namespace {
// Two forms.  The chunked form (bf16, shapes of the tensor-core scans, Dv = 128)
// keeps per-chunk images like the scalar tensor-core path; the recurrent form
// (everything else) keeps the state at every 8th step.
struct KcLayout {
    bool chunked;
    // recurrent form
    size_t ckpt, rq, rk, dqh, dkh, gpart, bpart;
    // chunked form, saved: checkpoints, Delta, W, P, T, Q_r, K_d, K_r images, e_C, the
    // decayed k Gram (and rq, rk above); forward workspace: U, then room for the
    // saved tensors when the caller keeps none; backward workspace: the reverse
    // scan's images, the q / k partials, the tensor-core pass's products
    size_t Delta, W, P, Tinv, qimg, kimg, krimg, ecd, gram, U, fwd_saved;
    size_t dSck, Dbar, kdb, qrb, wb, pbm, m1, ecb;
    size_t saved_total, fwd_total, bwd_total;
};
gdn_status kc_layout(const gdn_shape* shape, gdn::Dims* d, KcLayout* L) {
    gdn_status st = validate_shape(shape, d);
    if (st != GDN_OK) return st;
    *L = KcLayout{};
    if (gdn::kc_chunked_supported(*d)) {
        L->chunked = true;
        const size_t BH = (size_t)d->B * d->Hv, C = gdn::kChunk;
        const size_t img = BH * d->NC * d->Dk * d->Dv * 2;
        const size_t rowsk = BH * d->Tp * d->Dk, rowsv = BH * d->Tp * d->Dv;
        const size_t mat = BH * d->NC * C * C;
        size_t o = 0;
        L->ckpt = o; o = align_up(o + img);
        L->Delta = o; o = align_up(o + rowsv * 4);
        L->W = o; o = align_up(o + rowsk * 2);
        L->P = o; o = align_up(o + mat * 2);
        L->Tinv = o; o = align_up(o + mat * 2);
        L->qimg = o; o = align_up(o + rowsk * 2);
        L->kimg = o; o = align_up(o + rowsk * 2);
        L->krimg = o; o = align_up(o + rowsk * 2);
        L->ecd = o; o = align_up(o + BH * d->NC * d->Dk * 4);
        L->gram = o; o = align_up(o + mat * 4);
        L->rq = o; o = align_up(o + (size_t)d->B * d->Hk * d->Tp * 4);
        L->rk = o; o = align_up(o + (size_t)d->B * d->Hk * d->Tp * 4);
        L->saved_total = o;
        o = 0;
        L->U = o; o = align_up(o + rowsv * 4);
        L->fwd_saved = o; o = align_up(o + L->saved_total);
        L->fwd_total = o;
        o = 0;
        L->dSck = o; o = align_up(o + img);
        L->Dbar = o; o = align_up(o + rowsv * 2);
        L->dqh = o; o = align_up(o + rowsk * 4);
        L->dkh = o; o = align_up(o + rowsk * 4);
        L->kdb = o; o = align_up(o + rowsk * 4);
        L->qrb = o; o = align_up(o + rowsk * 4);
        L->wb = o; o = align_up(o + rowsk * 4);
        L->pbm = o; o = align_up(o + mat * 4);
        L->m1 = o; o = align_up(o + mat * 4);
        L->ecb = o; o = align_up(o + BH * d->NC * d->Dk * 4);
        L->bwd_total = o;
        return GDN_OK;
    }
    if (!gdn::kc_supported(*d)) return GDN_ERR_UNSUPPORTED_SHAPE;
    const size_t nt = (size_t)gdn::kc_tiles(*d);
    const size_t rows = (size_t)d->B * d->Hv * nt * d->Tp;  // per-tile partial rows
    L->ckpt = 0;
    L->saved_total = align_up((size_t)d->B * d->Hv * gdn::kc_segments(*d) * d->Dk * d->Dv * 4);
    size_t o = 0;
    L->rq = o; o = align_up(o + (size_t)d->B * d->Hk * d->Tp * 4);
    L->rk = o; o = align_up(o + (size_t)d->B * d->Hk * d->Tp * 4);
    L->fwd_total = o;
    L->dqh = o; o = align_up(o + rows * d->Dk * 4);
    L->dkh = o; o = align_up(o + rows * d->Dk * 4);
    L->gpart = o; o = align_up(o + rows * d->Dk * 4);
    L->bpart = o; o = align_up(o + rows * 4);
    L->bwd_total = o;
    return GDN_OK;
}

void carve_kc_saved(const KcLayout& L, void* saved, gdn::Ptrs* p) {
    char* s = static_cast<char*>(saved);
    p->ckpt = reinterpret_cast<float*>(s + L.ckpt);
    p->Delta = reinterpret_cast<float*>(s + L.Delta);
    p->W = s + L.W;
    p->P = s + L.P;
    p->Tinv = reinterpret_cast<float*>(s + L.Tinv);
    p->qimg = s + L.qimg;
    p->kimg = s + L.kimg;
    p->krimg = s + L.krimg;
    p->ecd = reinterpret_cast<float*>(s + L.ecd);
    p->gram = reinterpret_cast<float*>(s + L.gram);
    p->rq = reinterpret_cast<float*>(s + L.rq);
    p->rk = reinterpret_cast<float*>(s + L.rk);
}
}  // namespace

gdn_status gdn_kc_saved_bytes(const gdn_shape* shape, size_t* bytes) {
    gdn::Dims d;
    KcLayout L;
    gdn_status st = kc_layout(shape, &d, &L);
    if (st != GDN_OK) return st;
    if (bytes == nullptr) return GDN_ERR_INVALID_ARG;
    *bytes = L.saved_total;
    return GDN_OK;
}

gdn_status gdn_kc_workspace_bytes(const gdn_shape* shape, int pass, size_t* bytes) {
    gdn::Dims d;
    KcLayout L;
    gdn_status st = kc_layout(shape, &d, &L);
    if (st != GDN_OK) return st;
    if (bytes == nullptr || pass < 0 || pass > 1) return GDN_ERR_INVALID_ARG;
    *bytes = pass == 0 ? L.fwd_total : L.bwd_total;
    return GDN_OK;
}

gdn_status gdn_forward_kc(const gdn_shape* shape, const void* q, const void* k, const void* v,
                          const void* log_decay, const void* beta, const float* state0,
                          const uint8_t* mask, void* o, float* state_T, void* saved,
                          size_t saved_bytes, void* ws, size_t ws_bytes, void* stream) {
    gdn::Dims d;
    KcLayout L;
    gdn_status st = kc_layout(shape, &d, &L);
    if (st != GDN_OK) return st;
    if (!q || !k || !v || !log_decay || !beta || !o || !state_T || !ws) return GDN_ERR_INVALID_ARG;
    if (shape->has_mask && !mask) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, log_decay, beta, state0, mask, o, state_T, saved, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    if ((saved && saved_bytes < L.saved_total) || ws_bytes < L.fwd_total)
        return GDN_ERR_WORKSPACE_TOO_SMALL;
    gdn::Ptrs p{};
    p.q = q; p.k = k; p.v = v; p.state0 = state0;
    p.a = log_decay; p.b = beta;
    p.mask = shape->has_mask ? mask : nullptr;
    p.o = o; p.state_T = state_T;
    char* w = static_cast<char*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L.chunked) {
        carve_kc_saved(L, saved ? saved : w + L.fwd_saved, &p);
        p.U = reinterpret_cast<float*>(w + L.U);
        gdn::Tmaps maps;
        if (!make_tmaps(d, v, nullptr, o, p.U, &maps)) return tmap_error();
        p.tmaps = &maps;
        cudaError_t e = run_phase("prep", s, [&] { return gdn::launch_prep_norms(d, p, s); });
        if (e == cudaSuccess) e = run_phase("kc_chunk", s, [&] { return gdn::launch_kc_chunk(d, p, s); });
        if (e == cudaSuccess) e = run_phase("kc_scan", s, [&] { return gdn::launch_fwd_scan_kc(d, p, s); });
        return cuda_status(e);
    }
    p.rq = reinterpret_cast<float*>(w + L.rq);
    p.rk = reinterpret_cast<float*>(w + L.rk);
    cudaError_t e = run_phase("prep", s, [&] { return gdn::launch_prep_norms(d, p, s); });
    if (e == cudaSuccess)
        e = run_phase("kc_fwd", s, [&] {
            return gdn::launch_kc_forward(d, p, log_decay, beta, static_cast<float*>(saved), s);
        });
    return cuda_status(e);
}

gdn_status gdn_backward_kc(const gdn_shape* shape, const void* q, const void* k, const void* v,
                           const void* log_decay, const void* beta, const uint8_t* mask,
                           const void* saved, size_t saved_bytes, const void* d_o,
                           const float* d_state_T, void* dq, void* dk, void* dv,
                           void* d_log_decay, void* d_beta, float* dstate0, void* ws,
                           size_t ws_bytes, void* stream) {
    gdn::Dims d;
    KcLayout L;
    gdn_status st = kc_layout(shape, &d, &L);
    if (st != GDN_OK) return st;
    if (!q || !k || !v || !log_decay || !beta || !saved || !d_o || !dq || !dk || !dv ||
        !d_log_decay || !d_beta || !dstate0 || !ws)
        return GDN_ERR_INVALID_ARG;
    if (shape->has_mask && !mask) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, log_decay, beta, mask, saved, d_o, d_state_T, dq, dk, dv,
                          d_log_decay, d_beta, dstate0, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    if (saved_bytes < L.saved_total || ws_bytes < L.bwd_total) return GDN_ERR_WORKSPACE_TOO_SMALL;
    gdn::Ptrs p{};
    p.q = q; p.k = k; p.v = v;
    p.a = log_decay; p.b = beta;
    p.mask = shape->has_mask ? mask : nullptr;
    p.d_o = d_o; p.d_state_T = d_state_T;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dstate0 = dstate0;
    p.da = d_log_decay; p.db = d_beta;
    char* w = static_cast<char*>(ws);
    p.dqh = reinterpret_cast<float*>(w + L.dqh);
    p.dkh = reinterpret_cast<float*>(w + L.dkh);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L.chunked) {
        carve_kc_saved(L, const_cast<void*>(saved), &p);
        p.dSck = reinterpret_cast<float*>(w + L.dSck);
        p.Dbar = reinterpret_cast<float*>(w + L.Dbar);
        p.kdb = reinterpret_cast<float*>(w + L.kdb);
        p.qrb = reinterpret_cast<float*>(w + L.qrb);
        p.wb = reinterpret_cast<float*>(w + L.wb);
        p.pbm = reinterpret_cast<float*>(w + L.pbm);
        p.m1 = reinterpret_cast<float*>(w + L.m1);
        p.ecb = reinterpret_cast<float*>(w + L.ecb);
        gdn::Tmaps maps;
        if (!make_tmaps(d, v, d_o, nullptr, nullptr, &maps)) return tmap_error();
        p.tmaps = &maps;
        cudaError_t e = run_phase("kc_bwd_scan", s, [&] { return gdn::launch_bwd_scan_kc(d, p, s); });
        if (e == cudaSuccess) e = run_phase("kc_bwd_prod", s, [&] { return gdn::launch_kc_bwd_prod(d, p, s); });
        if (e == cudaSuccess) e = run_phase("kc_bwd_gate", s, [&] { return gdn::launch_kc_bwd_gate(d, p, s); });
        if (e == cudaSuccess) e = run_phase("kc_bwd_chan", s, [&] { return gdn::launch_kc_bwd_chan(d, p, s); });
        if (e == cudaSuccess) e = run_phase("bwd_reduce", s, [&] { return gdn::launch_qk_reduce(d, p, s); });
        return cuda_status(e);
    }
    p.rq = reinterpret_cast<float*>(w + L.rq);
    p.rk = reinterpret_cast<float*>(w + L.rk);
    cudaError_t e = run_phase("prep", s, [&] { return gdn::launch_prep_norms(d, p, s); });
    if (e == cudaSuccess)
        e = run_phase("kc_bwd", s, [&] {
            return gdn::launch_kc_backward(d, p, log_decay, beta, static_cast<const float*>(saved),
                                           reinterpret_cast<float*>(w + L.gpart),
                                           reinterpret_cast<float*>(w + L.bpart), d_log_decay,
                                           d_beta, s);
        });
    if (e == cudaSuccess) {
        // the tiles' partials as value heads of their own: G Dv / 16 per key head
        gdn::Dims d2 = d;
        d2.Hv = d.Hv * gdn::kc_tiles(d);
        d2.G = d.G * gdn::kc_tiles(d);
        e = run_phase("bwd_reduce", s, [&] { return gdn::launch_qk_reduce(d2, p, s); });
    }
    return cuda_status(e);
}

gdn_status gdn_causal_conv1d_update(int64_t B, int64_t C, int64_t S, int64_t K, int32_t dtype,
                                    const void* hidden, const void* conv_state,
                                    const void* weight, void* out, void* final_state,
                                    void* stream) {
    if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARG;
    if (B < 1 || C < 1 || S < 1 || K < 1 || K > gdn::kConvMaxK) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (B * C > (int64_t(1) << 40) || B * C * S > (int64_t(1) << 46)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!hidden || !conv_state || !weight || !out || !final_state) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {hidden, conv_state, weight, out, final_state};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(run_phase("conv1d", s, [&] {
        return gdn::launch_causal_conv1d_update(B, C, S, (int)K, dtype, hidden, conv_state, weight,
                                                out, final_state, s);
    }));
}

gdn_status gdn_decode_conv(const gdn_shape* shape, int32_t gates, int64_t K, const void* hidden,
                           const void* conv_state, const void* conv_weight,
                           void* final_conv_state, const void* a, const void* b,
                           const float* A_log, const float* dt_bias, const float* state0,
                           const uint8_t* mask, void* o, float* state_T, void* stream) {
    gdn::Dims d;
    gdn_status st = validate_shape(shape, &d);
    if (st != GDN_OK) return st;
    if (gates != 0 && gates != 1) return GDN_ERR_INVALID_ARG;
    d.gates = gates;
    if (d.T != 1 || K < 1 || K > gdn::kConvMaxK || !gdn::decode_supported(d.Dk, d.Dv))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!hidden || !conv_state || !conv_weight || !final_conv_state || !a || !b || !o || !state_T)
        return GDN_ERR_INVALID_ARG;
    if (gates == 0 && (!A_log || !dt_bias)) return GDN_ERR_INVALID_ARG;
    if (shape->has_mask && !mask) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {hidden, conv_state, conv_weight, final_conv_state, a, b, A_log,
                          dt_bias, state0, mask, o, state_T};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    const size_t es = d.dtype == GDN_DTYPE_BF16 ? 2 : 4;
    const size_t cs_bytes = (size_t)d.B * (2 * d.Hk * d.Dk + d.Hv * d.Dv) * K * es;
    const char* c0 = static_cast<const char*>(conv_state);
    const char* f0 = static_cast<const char*>(final_conv_state);
    if (f0 < c0 + cs_bytes && c0 < f0 + cs_bytes) return GDN_ERR_INVALID_ARG;  // overlap
    gdn::Ptrs p{};
    p.a = a; p.b = b; p.A_log = A_log; p.dt_bias = dt_bias; p.state0 = state0;
    p.mask = shape->has_mask ? mask : nullptr;
    p.o = o; p.state_T = state_T;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(run_phase("decode", s, [&] {
        return gdn::launch_decode_conv(d, p, hidden, conv_state, conv_weight, final_conv_state,
                                       (int)K, s);
    }));
}

uint64_t gdn_launch_count(void) { return g_launches.load(); }

gdn_status gdn_timing_begin(void) {
    for (auto& ev : g_events) {
        cudaEventDestroy(ev.start);
        cudaEventDestroy(ev.stop);
    }
    g_events.clear();
    g_timing = true;
    return GDN_OK;
}

gdn_status gdn_timing_end(gdn_phase_time* out, int max, int* count) {
    g_timing = false;
    if (count == nullptr || (out == nullptr && max > 0)) return GDN_ERR_INVALID_ARG;
    int n = 0;
    cudaError_t err = cudaSuccess;
    for (auto& ev : g_events) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(ev.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev.start, ev.stop);
        if (e != cudaSuccess) err = e;
        int i = 0;
        while (i < n && std::strcmp(out[i].name, ev.name) != 0) ++i;
        if (i == n && n < max) {
            out[n].name = ev.name;
            out[n].launches = 0;
            out[n].total_ms = 0.0;
            ++n;
        }
        if (i < n) {
            out[i].launches += 1;
            out[i].total_ms += ms;
        }
        cudaEventDestroy(ev.start);
        cudaEventDestroy(ev.stop);
    }
    g_events.clear();
    *count = n;
    return cuda_status(err);
}

}  // extern "C"
