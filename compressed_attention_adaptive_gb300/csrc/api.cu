// C ABI of libmita: argument validation, workspace carving and the order of
// launches for each entry point (declared in include/mita.h).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mita.h"
#include "internal.h"

namespace mita {

static thread_local std::string g_last_error;

// ---------------------------------------------------------------- profiling
// While a profile is open, every prof_mark() records a CUDA event on the
// launching stream; mita_profile_end() sums the time between consecutive
// marks per phase name.
static std::atomic<long long> g_launches{0};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<std::pair<std::string, cudaEvent_t>> g_prof_marks;
static std::vector<cudaEvent_t> g_prof_pool;

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

void prof_mark(cudaStream_t st, const char* phase) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on || g_prof_marks.size() >= g_prof_pool.size()) return;
    cudaEvent_t ev = g_prof_pool[g_prof_marks.size()];
    if (cudaEventRecord(ev, st) == cudaSuccess) g_prof_marks.emplace_back(phase, ev);
}

static mita_status fail(mita_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

static mita_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MITA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MITA_CUDA(call, what)                              \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

// Validates p and fills D. Returns MITA_OK or the error (with detail).
static mita_status resolve(const mita_params* p, Dims* D) {
    if (!p) return fail(MITA_ERR_INVALID_ARG, "params is NULL");
    if (p->B < 1 || p->H < 1 || p->N < 1) return fail(MITA_ERR_INVALID_ARG, "B, H, N must be >= 1");
    if (p->d < 8 || p->d > 256 || p->d % 8) return fail(MITA_ERR_INVALID_ARG, "d must be a multiple of 8 in [8, 256]");
    if (p->m < 1 || p->m > p->N) return fail(MITA_ERR_INVALID_ARG, "m must be in [1, N]");
    if (p->k < 1 || p->k > p->N) return fail(MITA_ERR_INVALID_ARG, "k must be in [1, N]");
    if (p->s < 1 || p->s > p->m) return fail(MITA_ERR_INVALID_ARG, "s must be in [1, m]");
    if (p->s > kMaxS) return fail(MITA_ERR_UNSUPPORTED, "s > %d is not supported", kMaxS);
    if (p->dtype != MITA_DTYPE_F32 && p->dtype != MITA_DTYPE_BF16) return fail(MITA_ERR_INVALID_ARG, "bad dtype");
    if (p->flags & ~(unsigned)(MITA_FLAG_NO_SHARED | MITA_FLAG_SIMT | MITA_FLAG_CAUSAL | MITA_TESTFLAG_STALL_PRODUCER))
        return fail(MITA_ERR_INVALID_ARG, "unknown flag");
    if ((p->flags & MITA_FLAG_CAUSAL) && p->grid_h != 0)
        return fail(MITA_ERR_INVALID_ARG, "the causal variant needs 1-D pooling (grid_h == 0)");
    if (!(p->scale >= 0.0f) || isinf(p->scale)) return fail(MITA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    if ((long long)p->B * p->H > 65535) return fail(MITA_ERR_UNSUPPORTED, "B*H must be <= 65535");
    if ((long long)p->B * p->H * p->N >= (1LL << 31)) return fail(MITA_ERR_UNSUPPORTED, "B*H*N must be < 2^31");
    D->B = p->B; D->H = p->H; D->BH = p->B * p->H; D->N = p->N; D->d = p->d;
    D->m = p->m; D->k = p->k; D->s = p->s;
    if (p->grid_h == 0) {
        D->gh = 1; D->gw = p->N; D->lh = 1; D->lw = p->m;
    } else {
        if (p->grid_h < 1 || p->grid_w < 1 || (long long)p->grid_h * p->grid_w != p->N)
            return fail(MITA_ERR_INVALID_ARG, "grid_h * grid_w must equal N");
        if (p->lm_h < 1 || p->lm_w < 1 || p->lm_h * p->lm_w != p->m)
            return fail(MITA_ERR_INVALID_ARG, "lm_h * lm_w must equal m");
        if (p->lm_h > p->grid_h || p->lm_w > p->grid_w)
            return fail(MITA_ERR_INVALID_ARG, "landmark grid larger than token grid");
        D->gh = p->grid_h; D->gw = p->grid_w; D->lh = p->lm_h; D->lw = p->lm_w;
    }
    D->scale = p->scale > 0.0f ? p->scale : 1.0f / sqrtf((float)p->d);
    D->flags = p->flags;
    D->dtype = p->dtype;
    D->shared = !(p->flags & MITA_FLAG_NO_SHARED);
    D->causal = (p->flags & MITA_FLAG_CAUSAL) != 0;
    if (D->causal && !(p->flags & MITA_FLAG_SIMT) && tc_supported(*D) && !tc_plan(*D).resident)
        return fail(MITA_ERR_UNSUPPORTED,
                    "the causal variant runs on the tensor-core path only for m <= 128, k <= 256 with the shared "
                    "slots on (MITA_FLAG_SIMT runs it on CUDA cores)");
    if (out_simt_smem(*D) > 200 * 1024) return fail(MITA_ERR_UNSUPPORTED, "m + s*k too large for this library");
    return MITA_OK;
}

static size_t elem_size(const Dims& D) { return D.dtype == MITA_DTYPE_F32 ? 4 : 2; }
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Sequential carving of one workspace allocation into 1 KiB-aligned buffers.
struct Carver {
    char* base;
    size_t off = 0;
    explicit Carver(void* b) : base((char*)b) {}
    template <typename T> T* take(size_t count) {
        off = align_up(off, 1024);
        T* p = base ? (T*)(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

static bool use_tc(const Dims& D) { return !(D.flags & MITA_FLAG_SIMT) && tc_supported(D); }

struct Work {
    int* status;
    float* Qt;
    float* Vt;
    int32_t* I;
    int32_t* E;
    // CUDA-core path
    float2* stats;
    float* S;
    float* R;
    // tensor-core path
    TcPlan plan;
    TcWork tc;
};

static Work carve(const Dims& D, void* ws, size_t* bytes) {
    Carver c(ws);
    Work w{};
    const size_t BH = D.BH;
    w.status = c.take<int>(64);
    w.Qt = c.take<float>(BH * D.m * D.d);
    w.Vt = c.take<float>(BH * D.m * D.d);
    w.I = c.take<int32_t>(BH * D.m * D.k);
    w.E = c.take<int32_t>(BH * D.N * D.s);
    if (!use_tc(D)) {
        w.stats = c.take<float2>(BH * D.m);
        w.S = c.take<float>(BH * D.m * D.N);
        w.R = c.take<float>(BH * D.N * D.m);
    } else {
        const TcPlan P = tc_plan(D);
        w.plan = P;
        TcWork& t = w.tc;
        t.Qhi = c.take<__nv_bfloat16>(BH * P.m_pad * D.d);
        t.Qlo = c.take<__nv_bfloat16>(BH * P.m_pad * D.d);
        t.Vtb = c.take<__nv_bfloat16>(BH * P.m_pad * D.d);
        t.Opart = c.take<float>(BH * P.splits * P.m_pad * D.d);
        t.ML = c.take<float2>(BH * P.splits * P.m_pad);
        t.Ssamp = c.take<float>(BH * D.m * (size_t)P.n_samp);
        t.thr = c.take<float>(BH * D.m);
        t.cand = c.take<int2>(BH * P.m_pad * (size_t)P.splits * (size_t)P.cand_cap);
        t.ccount = c.take<int>(BH * P.m_pad * (size_t)P.splits * 2);
        t.counts = c.take<int>(BH * D.m * 2);
        t.tile_ctr = c.take<int>(3);
        t.zero_begin = t.counts;
        t.zero_bytes = t.counts ? (size_t)((char*)(t.tile_ctr + 3) - (char*)t.counts) : 0;
        t.cursors = c.take<int>(BH * D.m * 2);
        t.toff = c.take<int>(BH * D.m);
        t.tiles = c.take<int4>((size_t)P.max_tiles);
        t.xtl = c.take<int2>(BH * D.m);
        t.perm = c.take<int32_t>(BH * D.N * D.s);
        t.part = c.take<__nv_bfloat16>(BH * D.N * D.s * P.nsub * D.d);
        t.lse = c.take<float>(BH * D.N * D.s * P.nsub);
        if (P.nsh) {
            t.sh_part = c.take<__nv_bfloat16>(BH * D.N * P.nsh * D.d);
            t.sh_lse = c.take<float>(BH * D.N * P.nsh);
        }
    }
    *bytes = align_up(c.off, 1024);
    return w;
}

static mita_status check_ws(const Dims& D, void* ws, size_t ws_bytes, Work* w) {
    size_t need;
    carve(D, nullptr, &need);
    if (!ws) return fail(MITA_ERR_WORKSPACE, "workspace is NULL");
    if ((uintptr_t)ws % 256) return fail(MITA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need) return fail(MITA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    *w = carve(D, ws, &need);
    return MITA_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

static mita_status run(const mita_params* p, const void* Q, const void* K, const void* V, void* O, float* Qt_out,
                       int32_t* idx_out, int32_t* route_out, float* Vt_out, void* ws, size_t ws_bytes,
                       void* stream, int upto, bool keep_status = false) {
    Dims D;
    mita_status st = resolve(p, &D);
    if (st) return st;
    if (keep_status) D.flags |= kFlagKeepStatus;
    if (!Q || !aligned16(Q)) return fail(MITA_ERR_INVALID_ARG, "Q must be a 16-byte aligned device pointer");
    if (upto >= 1 && (!K || !aligned16(K))) return fail(MITA_ERR_INVALID_ARG, "K must be a 16-byte aligned device pointer");
    if (upto >= 2 && (!V || !aligned16(V))) return fail(MITA_ERR_INVALID_ARG, "V must be a 16-byte aligned device pointer");
    if (upto >= 2 && (!O || !aligned16(O))) return fail(MITA_ERR_INVALID_ARG, "O must be a 16-byte aligned device pointer");
    Work w;
    st = check_ws(D, ws, ws_bytes, &w);
    if (st) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* Qt = Qt_out ? Qt_out : w.Qt;
    int32_t* I = idx_out ? idx_out : w.I;
    int32_t* E = route_out ? route_out : w.E;
    float* Vt = Vt_out ? Vt_out : w.Vt;

    prof_mark(s, "pool");
    if (use_tc(D)) {
        MITA_CUDA(launch_pool(D, Q, Qt, w.tc.Qhi, w.tc.Qlo, w.plan.m_pad, w.status, s), "landmark pooling");
        if (upto > 0)
            MITA_CUDA(launch_forward_tc(D, w.plan, w.tc, Q, K, V, O, Vt, I, (upto == 1 && !route_out) ? nullptr : E,
                                        w.status, upto, s),
                      "tensor-core forward");
        prof_mark(s, "");
        return MITA_OK;
    }
    MITA_CUDA(launch_pool(D, Q, Qt, nullptr, nullptr, 0, w.status, s), "landmark pooling");
    if (upto > 0) {
        prof_mark(s, "select");
        MITA_CUDA(launch_select_simt(D, Q, K, Qt, w.S, w.R, I, (upto == 1 && !route_out) ? nullptr : E, s),
                  "expert selection");
    }
    if (upto > 1) {
        prof_mark(s, "shared");
        MITA_CUDA(launch_shared_simt(D, V, w.S, w.stats, Vt, s), "shared expert");
        prof_mark(s, "output");
        MITA_CUDA(launch_out_simt(D, Q, K, V, Qt, Vt, I, E, O, w.status, s), "expert attention");
    }
    prof_mark(s, "");
    return MITA_OK;
}

// For other translation units of the library: argument check, error report
// and the whole forward pass on a given workspace.
mita_status validate(const mita_params* p) {
    Dims D;
    return resolve(p, &D);
}

mita_status report_error(mita_status st, const char* msg) { return fail(st, "%s", msg); }

void clear_error() { g_last_error.clear(); }

mita_status forward_on_workspace(const mita_params* p, const void* Q, const void* K, const void* V, void* O,
                                 void* ws, size_t ws_bytes, void* stream) {
    return run(p, Q, K, V, O, nullptr, nullptr, nullptr, nullptr, ws, ws_bytes, stream, 2);
}

// ---------------------------------------------------------------- backward

static mita_status resolve_bwd(const mita_params* p, Dims* D) {
    mita_status st = resolve(p, D);
    if (st) return st;
    if (D->causal) return fail(MITA_ERR_UNSUPPORTED, "the backward pass has no causal variant");
    if (D->gh != 1) return fail(MITA_ERR_UNSUPPORTED, "the backward pass supports 1-D pooling only");
    if (bwd_query_smem(*D) > 200 * 1024) return fail(MITA_ERR_UNSUPPORTED, "m + s*k too large for the backward pass");
    if (D->d != 64 && D->d != 128) return fail(MITA_ERR_UNSUPPORTED, "the backward pass supports d = 64 or 128");
    return MITA_OK;
}

// Carving of the backward workspace (status word first, like the forward's).
static BwdWork carve_bwd(const Dims& D, void* ws, size_t* bytes, int** status) {
    Carver c(ws);
    BwdWork w{};
    const size_t BH = D.BH, N = D.N, d = D.d, m = D.m;
    *status = c.take<int>(64);
    w.Qt = c.take<float>(BH * m * d);
    w.Vt = c.take<float>(BH * m * d);
    w.stats = c.take<float2>(BH * m);
    w.S = c.take<float>(BH * m * N);
    w.dA = c.take<float>(BH * m * N);
    w.Psh = c.take<float>(BH * N * m);
    w.dZsh = c.take<float>(BH * N * m);
    w.dQt = c.take<float>(BH * m * d);
    w.dVt = c.take<float>(BH * m * d);
    w.delta = c.take<float>(BH * m);
    w.dQacc = c.take<float>(BH * N * d);
    w.dKacc = c.take<float>(BH * N * d);
    w.dVacc = c.take<float>(BH * N * d);
    w.Pr = c.take<float>(BH * N * D.s * (size_t)D.k);
    w.dZr = c.take<float>(BH * N * D.s * (size_t)D.k);
    w.counts = c.take<int>(BH * m);
    w.cursors = c.take<int>(BH * m);
    w.offs = c.take<int>(BH * (m + 1));
    w.rows = c.take<int>(BH * N * D.s);
    *bytes = align_up(c.off, 1024);
    return w;
}

}  // namespace mita

using namespace mita;

extern "C" {

size_t mita_workspace_size(const mita_params* p) {
    Dims D;
    if (resolve(p, &D)) return 0;
    size_t bytes;
    carve(D, nullptr, &bytes);
    return bytes;
}

mita_status mita_landmarks(const mita_params* p, const void* Q, float* Qt, void* ws, size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (!Qt) return fail(MITA_ERR_INVALID_ARG, "Qt is NULL");
    return run(p, Q, nullptr, nullptr, nullptr, Qt, nullptr, nullptr, nullptr, ws, ws_bytes, stream, 0);
}

mita_status mita_select(const mita_params* p, const void* Q, const void* K, int32_t* idx, int32_t* route, void* ws,
                        size_t ws_bytes, void* stream) {
    g_last_error.clear();
    return run(p, Q, K, nullptr, nullptr, nullptr, idx, route, nullptr, ws, ws_bytes, stream, 1);
}

mita_status mita_forward(const mita_params* p, const void* Q, const void* K, const void* V, void* O,
                         int32_t* idx_out, int32_t* route_out, float* Vt_out, void* ws, size_t ws_bytes,
                         void* stream) {
    g_last_error.clear();
    return run(p, Q, K, V, O, nullptr, idx_out, route_out, Vt_out, ws, ws_bytes, stream, 2);
}

size_t mita_host_buffer_size(const mita_params* p) {
    Dims D;
    if (resolve(p, &D)) return 0;
    const size_t t = align_up((size_t)D.BH * D.N * D.d * elem_size(D), 1024);
    return 4 * t + mita_workspace_size(p);
}

// Copy streams and events of mita_forward_host, created once per device and
// kept for the process (creating them on every call costs host time in the
// middle of a pipelined sequence of calls). g_host_mu serializes the enqueue
// sequences, so that no two calls record the same event concurrently.
constexpr int kHostGroups = 8;
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[2 * (kHostGroups + 1) + 2] = {};
};
static std::mutex g_host_mu;
static HostPipe g_host_pipe[64];

static cudaError_t host_pipe(HostPipe** hp) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    HostPipe& h = g_host_pipe[dev];
    if (!h.in) {
        if ((e = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (cudaEvent_t& x : h.ev)
            if ((e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *hp = &h;
    return cudaSuccess;
}

mita_status mita_forward_host(const mita_params* p, const void* Q, const void* K, const void* V, void* O, void* dev,
                              size_t dev_bytes, void* stream) {
    g_last_error.clear();
    Dims D;
    mita_status st = resolve(p, &D);
    if (st) return st;
    if (!Q || !K || !V || !O) return fail(MITA_ERR_INVALID_ARG, "host buffers must not be NULL");
    const size_t need = mita_host_buffer_size(p);
    if (!dev || (uintptr_t)dev % 256) return fail(MITA_ERR_WORKSPACE, "device buffer NULL or not 256-byte aligned");
    if (dev_bytes < need) return fail(MITA_ERR_WORKSPACE, "device buffer too small: %zu < %zu bytes", dev_bytes, need);
    const size_t head = (size_t)D.N * D.d * elem_size(D);  // bytes of one head of Q, K, V or O
    const size_t t = align_up((size_t)D.BH * head, 1024);
    char* b = (char*)dev;
    const char *hq = (const char*)Q, *hk = (const char*)K, *hv = (const char*)V;
    char* ho = (char*)O;
    cudaStream_t s = (cudaStream_t)stream;
    // Heads are independent and contiguous in [B, H, N, d]: in groups of heads,
    // group g + 1's inputs go in and group g - 1's output comes out (two copy
    // streams) while group g computes on `stream`; the copy streams wait for
    // earlier work on `stream` and join it at the end, so the call stays
    // ordered on it. Groups of ceil(BH / 8) heads, the last one in two halves:
    // what runs after the last copy in (the last group's forward pass and copy
    // out) is then short, while no group is so small that the fixed latency of
    // its forward pass outlasts its copy in.
    int gsz[kHostGroups + 1];
    int G = 0;
    if (head % 256) {
        gsz[G++] = D.BH;  // offsets of later heads would break the copies' alignment
    } else {
        const int hb = (D.BH + kHostGroups - 1) / kHostGroups;
        for (int h = 0; h < D.BH; h += hb) gsz[G++] = std::min(hb, D.BH - h);
        if (gsz[G - 1] >= 2) {
            const int a = gsz[G - 1];
            gsz[G - 1] = a - a / 2;
            gsz[G++] = a / 2;
        }
    }
    std::lock_guard<std::mutex> lk(g_host_mu);
    HostPipe* hp = nullptr;
    MITA_CUDA(host_pipe(&hp), "create copy streams");
    cudaEvent_t* ev = hp->ev;
    MITA_CUDA(cudaEventRecord(ev[0], s), "record event");  // earlier work on `stream` first
    MITA_CUDA(cudaStreamWaitEvent(hp->in, ev[0], 0), "order copies");
    MITA_CUDA(cudaStreamWaitEvent(hp->out, ev[0], 0), "order copies");
    for (int g = 0, h0 = 0; g < G; h0 += gsz[g], ++g) {
        const int nh = gsz[g];
        const size_t off = (size_t)h0 * head, len = (size_t)nh * head;
        cudaEvent_t ein = ev[1 + 2 * g], erun = ev[2 + 2 * g];
        MITA_CUDA(cudaMemcpyAsync(b + off, hq + off, len, cudaMemcpyHostToDevice, hp->in), "copy Q to device");
        MITA_CUDA(cudaMemcpyAsync(b + t + off, hk + off, len, cudaMemcpyHostToDevice, hp->in), "copy K to device");
        MITA_CUDA(cudaMemcpyAsync(b + 2 * t + off, hv + off, len, cudaMemcpyHostToDevice, hp->in), "copy V to device");
        MITA_CUDA(cudaEventRecord(ein, hp->in), "record event");
        MITA_CUDA(cudaStreamWaitEvent(s, ein, 0), "order compute after copies");
        mita_params pg = *p;  // heads h0 .. h0 + nh - 1 as one batch of nh heads
        pg.B = 1;
        pg.H = nh;
        st = run(&pg, b + off, b + t + off, b + 2 * t + off, b + 3 * t + off, nullptr, nullptr, nullptr, nullptr,
                 b + 4 * t, dev_bytes - 4 * t, stream, 2, g > 0);
        if (st) return st;
        MITA_CUDA(cudaEventRecord(erun, s), "record event");
        MITA_CUDA(cudaStreamWaitEvent(hp->out, erun, 0), "order copy after compute");
        MITA_CUDA(cudaMemcpyAsync(ho + off, b + 3 * t + off, len, cudaMemcpyDeviceToHost, hp->out), "copy O to host");
    }
    MITA_CUDA(cudaEventRecord(ev[2 * (kHostGroups + 1) + 1], hp->out), "record event");
    MITA_CUDA(cudaStreamWaitEvent(s, ev[2 * (kHostGroups + 1) + 1], 0), "join copy stream");
    return MITA_OK;
}

mita_status mita_device_status(void* ws, void* stream) {
    g_last_error.clear();
    if (!ws) return fail(MITA_ERR_WORKSPACE, "workspace is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    MITA_CUDA(cudaStreamSynchronize(s), "stream synchronize");
    int v = 0;
    MITA_CUDA(cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost), "read device status");
    const int zero = 0;
    MITA_CUDA(cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice), "clear device status");
    if (v == kStTimeout) return fail(MITA_ERR_TIMEOUT, "a bounded device wait ran out");
    if (v == kStBounds) return fail(MITA_ERR_BOUNDS, "a device index was out of range");
    if (v != 0) return fail(MITA_ERR_CUDA, "unexpected device status %d", v);
    return MITA_OK;
}

const char* mita_status_string(mita_status s) {
    switch (s) {
        case MITA_OK: return "ok";
        case MITA_ERR_INVALID_ARG: return "invalid argument";
        case MITA_ERR_UNSUPPORTED: return "unsupported parameters";
        case MITA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MITA_ERR_CUDA: return "CUDA error";
        case MITA_ERR_TIMEOUT: return "device wait timed out";
        case MITA_ERR_BOUNDS: return "device index out of range";
    }
    return "unknown status";
}

const char* mita_last_error(void) { return g_last_error.c_str(); }

long long mita_launch_count(void) { return g_launches.load(); }


mita_status mita_profile_begin(int max_marks) {
    g_last_error.clear();
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) return fail(MITA_ERR_INVALID_ARG, "a profile is already open");
    if (max_marks < 2) return fail(MITA_ERR_INVALID_ARG, "max_marks must be >= 2");
    while ((int)g_prof_pool.size() < max_marks) {
        cudaEvent_t ev;
        MITA_CUDA(cudaEventCreate(&ev), "create profiling event");
        g_prof_pool.push_back(ev);
    }
    g_prof_marks.clear();
    g_prof_on = true;
    return MITA_OK;
}

int mita_profile_end(char* names, size_t names_bytes, double* ms, int max_phases) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = false;
    std::vector<std::string> order;
    std::vector<double> sum;
    if (!g_prof_marks.empty() && cudaEventSynchronize(g_prof_marks.back().second) != cudaSuccess) return -1;
    for (size_t i = 0; i + 1 < g_prof_marks.size(); ++i) {
        const std::string& nm = g_prof_marks[i].first;
        if (nm.empty()) continue;  // end-of-call marker
        float t = 0.0f;
        if (cudaEventElapsedTime(&t, g_prof_marks[i].second, g_prof_marks[i + 1].second) != cudaSuccess) return -1;
        size_t j = 0;
        while (j < order.size() && order[j] != nm) ++j;
        if (j == order.size()) { order.push_back(nm); sum.push_back(0.0); }
        sum[j] += t;
    }
    g_prof_marks.clear();
    std::string joined;
    int n = 0;
    for (size_t j = 0; j < order.size() && n < max_phases; ++j, ++n) {
        if (ms) ms[n] = sum[j];
        joined += order[j];
        joined += '\n';
    }
    if (names && names_bytes) {
        size_t c = joined.size() < names_bytes - 1 ? joined.size() : names_bytes - 1;
        memcpy(names, joined.data(), c);
        names[c] = 0;
    }
    return n;
}

size_t mita_backward_workspace_size(const mita_params* p) {
    Dims D;
    if (resolve_bwd(p, &D)) return 0;
    size_t bytes;
    int* st;
    carve_bwd(D, nullptr, &bytes, &st);
    return bytes;
}

mita_status mita_backward(const mita_params* p, const void* Q, const void* K, const void* V, const void* dO,
                          const int32_t* idx, const int32_t* route, void* dQ, void* dK, void* dV, void* ws,
                          size_t ws_bytes, void* stream) {
    g_last_error.clear();
    Dims D;
    mita_status st = resolve_bwd(p, &D);
    if (st) return st;
    const void* ptrs[] = {Q, K, V, dO, idx, route, dQ, dK, dV};
    for (const void* x : ptrs)
        if (!x || ((uintptr_t)x & 15))
            return fail(MITA_ERR_INVALID_ARG, "tensors must be 16-byte aligned device pointers");
    size_t need;
    int* status;
    carve_bwd(D, nullptr, &need, &status);
    if (!ws) return fail(MITA_ERR_WORKSPACE, "workspace is NULL");
    if ((uintptr_t)ws % 256) return fail(MITA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need) return fail(MITA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    const BwdWork w = carve_bwd(D, ws, &need, &status);
    cudaStream_t s = (cudaStream_t)stream;
    MITA_CUDA(cudaMemsetAsync(status, 0, sizeof(int), s), "clear the device status word");
    MITA_CUDA(launch_backward(D, w, Q, K, V, dO, idx, route, dQ, dK, dV, status, s), "backward pass");
    prof_mark(s, "");
    return MITA_OK;
}

int mita_uses_tensor_cores(const mita_params* p) {
    Dims D;
    if (resolve(p, &D)) return -1;
    return use_tc(D) ? 1 : 0;
}

}  // extern "C"
