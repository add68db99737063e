// Host side of the C ABI declared in include/lola.h: argument validation, the state and
// workspace layouts, and the stream-ordered sequence of kernels of each call.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {

int select_cluster_size(int lam);

namespace {
thread_local char g_cuda_error[256] = "";
}  // namespace

int32_t cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", where, cudaGetErrorString(e));
    return LOLA_ERR_CUDA;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int32_t to_dims(const lola_config* c, Dims* d) {
    if (!c) return LOLA_ERR_INVALID_ARG;
    if (c->B < 1 || c->Hh < 1 || c->d_k < 1 || c->d_v < 1 || c->D < 2 || (c->D & 1) || c->eta < 0 ||
        c->lambda < 0 || c->chunk < 1 || (c->dtype != LOLA_F32 && c->dtype != LOLA_BF16))
        return LOLA_ERR_INVALID_ARG;
    if (c->read_mask < 0 || c->read_mask > 3 || (c->read_mask != 0 && c->eta < 1)) return LOLA_ERR_INVALID_ARG;
    if (c->alloc != LOLA_ALLOC_TOKEN && c->alloc != LOLA_ALLOC_CHUNK) return LOLA_ERR_INVALID_ARG;
    if (c->score < LOLA_SCORE_SRE || c->score > LOLA_SCORE_ATTENTION) return LOLA_ERR_INVALID_ARG;
    if (c->score != LOLA_SCORE_SRE && (c->eta < 1 || c->alloc != LOLA_ALLOC_TOKEN)) return LOLA_ERR_INVALID_ARG;
    if (c->alloc == LOLA_ALLOC_CHUNK &&
        (c->chunk < 1 || c->eta < c->chunk || c->eta % c->chunk != 0 || c->read_mask != 0))
        return LOLA_ERR_INVALID_ARG;
    if ((int64_t)c->B * c->Hh > (1 << 24)) return LOLA_ERR_UNSUPPORTED;
    const bool dims_ok = (c->d_k == 128 && c->d_v == 128 && c->D == 128) || (c->d_k == 64 && c->d_v == 64 && c->D == 64);
    if (!dims_ok) return LOLA_ERR_UNSUPPORTED;
    if (c->lambda > 1024 || c->eta > 8192) return LOLA_ERR_UNSUPPORTED;
    if (c->chunk < 16 || c->chunk > 256 || (c->chunk & (c->chunk - 1))) return LOLA_ERR_UNSUPPORTED;
    d->B = c->B;
    d->Hh = c->Hh;
    d->BH = c->B * c->Hh;
    d->dk = c->d_k;
    d->dv = c->d_v;
    d->D = c->D;
    d->eta = c->eta;
    d->lam = c->lambda;
    d->chunk = c->chunk;
    d->dtype = c->dtype;
    d->read_mask = c->read_mask;
    d->alloc = c->alloc;
    d->score = c->score;
    if (d->alloc == LOLA_ALLOC_CHUNK && !chunk_mode_fits(*d)) return LOLA_ERR_UNSUPPORTED;
    return LOLA_OK;
}

__global__ void state_init_kernel(char* state, Layout L, int eta, int lam) {
    char* rec = state + (int64_t)blockIdx.x * L.head_bytes;
    int32_t* wp = reinterpret_cast<int32_t*>(rec + L.win_pos);
    int32_t* cp = reinterpret_cast<int32_t*>(rec + L.c_pos);
    for (int i = threadIdx.x; i < eta; i += blockDim.x) wp[i] = -1;
    for (int i = threadIdx.x; i < lam; i += blockDim.x) cp[i] = -1;
}

// ---- tracing: CUDA events around each launch ----
struct TimedLaunch {
    int id;
    cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TimedLaunch> g_pending;
double g_total_ms[LOLA_KERNEL_COUNT];
int64_t g_launches[LOLA_KERNEL_COUNT];

// Runs `launch` (returning cudaError_t) bracketed by events when tracing is on.
template <typename F>
cudaError_t traced(int id, cudaStream_t st, F&& launch) {
    bool on;
    {
        std::lock_guard<std::mutex> g(g_trace_mu);
        on = g_trace_on;
    }
    if (!on) return launch();
    TimedLaunch r{id, nullptr, nullptr};
    cudaError_t e = cudaEventCreate(&r.start);
    if (e == cudaSuccess) e = cudaEventCreate(&r.stop);
    if (e == cudaSuccess) e = cudaEventRecord(r.start, st);
    if (e != cudaSuccess) return e;
    e = launch();
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(r.stop, st);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(g_trace_mu);
    g_pending.push_back(r);
    return cudaSuccess;
}

// ---- a lower-priority side stream per device: the feature map of the queries runs on it
// while the selection chain (one CTA per head: 128 of the 152 SMs at 4 x 32 heads) runs on
// the caller's stream, then the caller's stream waits for it before the output pass ----
struct SideStream {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_side_mu;   // held from the fork to the join of one call (host side only)
SideStream g_side[kMaxDevices];

cudaError_t side_stream_locked(SideStream** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    SideStream& s = g_side[dev];
    if (!s.st) {
        int least = 0, greatest = 0;
        e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&s.st, cudaStreamNonBlocking, least);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    *out = &s;
    return cudaSuccess;
}

void drain_pending(int id) {
    std::vector<TimedLaunch> keep;
    for (auto& r : g_pending) {
        if (id >= 0 && r.id != id) {
            keep.push_back(r);
            continue;
        }
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) == cudaSuccess && cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
            g_total_ms[r.id] += ms;
            g_launches[r.id] += 1;
        }
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_pending.swap(keep);
}

// lola_selftest_bounded_wait: one thread waits on an mbarrier that nothing completes, with
// the wait the kernels use (tc::mbar_wait: bounded by %globaltimer); [0] = 1 if it returned
// without giving up, [1] = the nanoseconds it waited
__device__ int64_t g_selftest[2];
__global__ void bounded_wait_kernel(int64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    tc::mbar_init(b, 1);
    const uint64_t t0 = tc::globaltimer_ns();
    const bool done = tc::mbar_wait(b, 0, (uint64_t)limit_ns);
    g_selftest[0] = done ? 1 : 0;
    g_selftest[1] = (int64_t)(tc::globaltimer_ns() - t0);
}

}  // namespace

Workspace carve_workspace(const Dims& d, int n, void* base) {
    Workspace w;
    char* p = static_cast<char*>(base);
    int64_t o = 0;
    const int64_t BH = d.BH;
    w.snap_interval = d.chunk < 128 ? 128 : d.chunk;
    w.nck = (n + w.snap_interval - 1) / w.snap_interval;
    auto take = [&](int64_t bytes) {
        char* r = p ? p + o : nullptr;
        o = align256(o + bytes);
        return r;
    };
    // The tensor-core output path reads phi(Q), phi(K) and the H snapshots in bf16 only;
    // the float32 path reads float32 copies.  phi(K) in float32 is always kept (selection).
    const bool tc = output_tc_supported(d);
    const bool fixed = d.score != LOLA_SCORE_SRE;   // the query-dependent scores read phi(Q) in float32
    w.phiK = reinterpret_cast<float*>(take(4 * BH * n * d.D));
    w.phiQ = reinterpret_cast<float*>(tc && !fixed ? nullptr : take(4 * BH * n * d.D));
    w.phiKb = reinterpret_cast<__nv_bfloat16*>(tc ? take(2 * BH * n * d.D) : nullptr);
    w.phiQb = reinterpret_cast<__nv_bfloat16*>(tc ? take(2 * BH * n * d.D) : nullptr);
    w.wstep = reinterpret_cast<int32_t*>(take(4 * BH * n));
    w.wpos = reinterpret_cast<int32_t*>(take(4 * BH * n));
    w.snapH = reinterpret_cast<float*>(tc ? nullptr : take(4 * BH * w.nck * d.D * d.dv));
    w.snapHb = reinterpret_cast<__nv_bfloat16*>(tc ? take(2 * BH * w.nck * d.D * d.dv) : nullptr);
    w.snapS = reinterpret_cast<float*>(take(4 * BH * w.nck * d.D));
    w.snapC = reinterpret_cast<int32_t*>(take(4 * BH * w.nck * (int64_t)(d.lam > 0 ? d.lam : 1)));
    w.slotpos = reinterpret_cast<int32_t*>(take(4 * BH * (int64_t)(d.lam > 0 ? d.lam : 1)));
    w.score = reinterpret_cast<float*>(fixed ? take(4 * BH * n) : nullptr);
    w.dH = reinterpret_cast<float*>(fixed ? take(4 * BH * w.nck * d.D * d.dv) : nullptr);
    w.dS = reinterpret_cast<float*>(fixed ? take(4 * BH * w.nck * d.D) : nullptr);
    w.abort_flag = reinterpret_cast<int*>(take(4));
    w.bytes = (size_t)o;
    return w;
}

cudaError_t launch_state_init(const Dims& d, char* state, const Layout& L, cudaStream_t st) {
    return traced(LOLA_KERNEL_STATE_INIT, st, [&]() {
        cudaError_t e = cudaMemsetAsync(state, 0, (size_t)L.head_bytes * d.BH, st);
        if (e != cudaSuccess) return e;
        state_init_kernel<<<d.BH, 256, 0, st>>>(state, L, d.eta, d.lam);
        return cudaGetLastError();
    });
}

// ---- the write-magnitude cache layer: shapes and workspace ----
namespace {
struct HolaDims {
    int B, Hh, BH, w, chunk, nck;
};
struct HolaWs {
    uint8_t* xtile;       // [BH][ceil(n / 64)][64 KB] unit rows, split, in the state path's tiles
    __nv_bfloat16* qt;    // [BH][n][d_k] RMS-scaled rows (cache path)
    __nv_bfloat16* kt;
    float* ystate;        // [BH][n][d_v]
    float* scores;        // [BH][n]
    int32_t* cache;       // [BH][nck][w]
    int32_t* status;      // [BH][4], word 3 the status bits
    int* abort_flag;
    size_t bytes;
};
constexpr int kHolaD = 128;

int32_t hola_dims(const lola_hola_config* c, int n, HolaDims* d) {
    if (!c || n < 1) return LOLA_ERR_INVALID_ARG;
    if (c->B < 1 || c->Hh < 1 || c->d_k < 1 || c->d_v < 1 || c->w < 0 || c->chunk < 1 ||
        (c->dtype != LOLA_F32 && c->dtype != LOLA_BF16))
        return LOLA_ERR_INVALID_ARG;
    if (c->d_k != kHolaD || c->d_v != kHolaD || c->dtype != LOLA_BF16) return LOLA_ERR_UNSUPPORTED;
    if (c->w > hola_max_cache() || c->chunk % 128 != 0 || c->chunk > 1024) return LOLA_ERR_UNSUPPORTED;
    if ((int64_t)c->B * c->Hh > (1 << 24) || (int64_t)n * c->B * c->Hh * kHolaD > ((int64_t)1 << 40))
        return LOLA_ERR_UNSUPPORTED;
    d->B = c->B;
    d->Hh = c->Hh;
    d->BH = c->B * c->Hh;
    d->w = c->w;
    d->chunk = c->chunk;
    d->nck = (n + c->chunk - 1) / c->chunk;
    return LOLA_OK;
}

HolaWs hola_carve(const HolaDims& d, int n, void* base) {
    HolaWs w;
    char* p = static_cast<char*>(base);
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        char* r = p ? p + o : nullptr;
        o = align256(o + bytes);
        return r;
    };
    const int64_t rows = (int64_t)d.BH * n;
    w.xtile = reinterpret_cast<uint8_t*>(take((int64_t)d.BH * ((n + 63) / 64) * kHolaXTile));
    w.qt = reinterpret_cast<__nv_bfloat16*>(take(2 * rows * kHolaD));
    w.kt = reinterpret_cast<__nv_bfloat16*>(take(2 * rows * kHolaD));
    w.ystate = reinterpret_cast<float*>(take(4 * rows * kHolaD));
    w.scores = reinterpret_cast<float*>(take(4 * rows));
    w.cache = reinterpret_cast<int32_t*>(take(4 * (int64_t)d.BH * d.nck * (d.w > 0 ? d.w : 1)));
    w.status = reinterpret_cast<int32_t*>(take(16 * (int64_t)d.BH));
    w.abort_flag = reinterpret_cast<int*>(take(4));
    w.bytes = (size_t)o;
    return w;
}
}  // namespace

}  // namespace lola

using namespace lola;

extern "C" {

int32_t lola_version(void) { return 100; }

const char* lola_status_string(int32_t s) {
    switch (s) {
        case LOLA_OK: return "ok";
        case LOLA_ERR_INVALID_ARG: return "invalid argument";
        case LOLA_ERR_UNSUPPORTED: return "unsupported configuration";
        case LOLA_ERR_WORKSPACE: return "workspace too small";
        case LOLA_ERR_CUDA: return "CUDA runtime error";
        case LOLA_ERR_DEVICE: return "device-side error reported in the state";
        default: return "unknown status";
    }
}

const char* lola_last_cuda_error(void) { return g_cuda_error; }

int32_t lola_check_config(const lola_config* cfg) {
    Dims d;
    return to_dims(cfg, &d);
}

int32_t lola_state_layout_of(const lola_config* cfg, lola_state_layout* out) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (!out) return LOLA_ERR_INVALID_ARG;
    Layout L = make_layout(d);
    out->head_bytes = L.head_bytes;
    out->H = L.H;
    out->s = L.s;
    out->win_pos = L.win_pos;
    out->win_k = L.win_k;
    out->win_v = L.win_v;
    out->win_phi = L.win_phi;
    out->c_pos = L.c_pos;
    out->c_k = L.c_k;
    out->c_v = L.c_v;
    out->c_phi = L.c_phi;
    out->c_N = L.c_N;
    out->c_z = L.c_z;
    out->ev = L.ev;
    out->tok_phi = L.tok_phi;
    return LOLA_OK;
}

size_t lola_state_bytes(const lola_config* cfg) {
    Dims d;
    if (to_dims(cfg, &d) != LOLA_OK) return 0;
    return (size_t)make_layout(d).head_bytes * d.BH;
}

size_t lola_prefill_workspace_bytes(const lola_config* cfg, int32_t n) {
    Dims d;
    if (to_dims(cfg, &d) != LOLA_OK || n < 1) return 0;
    return carve_workspace(d, n, nullptr).bytes;
}

int32_t lola_state_init(const lola_config* cfg, void* state, void* stream) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (!state || !aligned16(state)) return LOLA_ERR_INVALID_ARG;
    cudaError_t e = launch_state_init(d, static_cast<char*>(state), make_layout(d), (cudaStream_t)stream);
    return e == cudaSuccess ? LOLA_OK : cuda_fail(e, "lola_state_init");
}

int32_t lola_prefill(const lola_config* cfg, int32_t n, const void* Q, const void* K, const void* V, const float* W,
                     int64_t w_head_stride, void* Y, void* state, int32_t* write_pos, void* workspace,
                     size_t workspace_bytes, void* stream) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (n < 1) return LOLA_ERR_INVALID_ARG;
    if ((int64_t)n * d.BH * d.D > ((int64_t)1 << 40)) return LOLA_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !W || !Y || !state || !workspace) return LOLA_ERR_INVALID_ARG;
    if (w_head_stride < 0 || w_head_stride % 4 != 0) return LOLA_ERR_INVALID_ARG;
    const void* ptrs[] = {Q, K, V, W, Y, state, workspace};
    for (const void* p : ptrs)
        if (!aligned16(p)) return LOLA_ERR_INVALID_ARG;
    if (write_pos && (reinterpret_cast<uintptr_t>(write_pos) & 3)) return LOLA_ERR_INVALID_ARG;
    Workspace ws = carve_workspace(d, n, workspace);
    if (workspace_bytes < ws.bytes) return LOLA_ERR_WORKSPACE;
    if (write_pos) ws.wpos = write_pos;
    const Layout L = make_layout(d);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_state_init(d, static_cast<char*>(state), L, st);
    if (e != cudaSuccess) return cuda_fail(e, "state init");
    e = cudaMemsetAsync(ws.abort_flag, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "workspace flag");
    e = traced(LOLA_KERNEL_PHI, st,
               [&]() { return launch_phi(d, n, K, W, w_head_stride, ws.phiK, ws.phiKb, static_cast<char*>(state), L.head_bytes, ws.abort_flag, st); });
    if (e != cudaSuccess) return cuda_fail(e, "phi(K)");
    if (d.score != LOLA_SCORE_SRE) {
        // query-dependent scores: phi(Q) first (the scores read it in float32), then the
        // chain-free allocation
        e = traced(LOLA_KERNEL_PHI_Q, st,
                   [&]() { return launch_phi(d, n, Q, W, w_head_stride, ws.phiQ, ws.phiQb, static_cast<char*>(state), L.head_bytes, ws.abort_flag, st); });
        if (e != cudaSuccess) return cuda_fail(e, "phi(Q)");
        e = traced(LOLA_KERNEL_SELECT, st, [&]() {
            return launch_fixed_select(d, n, ws, Q, K, V, static_cast<char*>(state), L, st);
        });
        if (e != cudaSuccess) return cuda_fail(e, "selection (query-dependent score)");
    } else {
        // the selection on the caller's stream, phi(Q) beside it on the side stream (launched
        // second, at lower priority, so the chain's CTAs are placed first)
        std::lock_guard<std::mutex> g(g_side_mu);
        SideStream* side = nullptr;
        e = side_stream_locked(&side);
        if (e != cudaSuccess) return cuda_fail(e, "side stream");
        e = cudaEventRecord(side->fork, st);
        if (e != cudaSuccess) return cuda_fail(e, "fork");
        e = traced(LOLA_KERNEL_SELECT, st, [&]() {
            return d.alloc == LOLA_ALLOC_CHUNK ? launch_chunk_select(d, n, ws, K, V, static_cast<char*>(state), L, st)
                                               : launch_select(d, n, ws, K, V, static_cast<char*>(state), L, st);
        });
        if (e != cudaSuccess) return cuda_fail(e, "selection");
        e = cudaStreamWaitEvent(side->st, side->fork, 0);
        if (e != cudaSuccess) return cuda_fail(e, "fork wait");
        e = traced(LOLA_KERNEL_PHI_Q, side->st,
                   [&]() { return launch_phi(d, n, Q, W, w_head_stride, ws.phiQ, ws.phiQb, static_cast<char*>(state), L.head_bytes, ws.abort_flag, side->st); });
        if (e != cudaSuccess) return cuda_fail(e, "phi(Q)");
        e = cudaEventRecord(side->join, side->st);
        if (e != cudaSuccess) return cuda_fail(e, "join");
        e = cudaStreamWaitEvent(st, side->join, 0);
        if (e != cudaSuccess) return cuda_fail(e, "join wait");
    }
    e = traced(LOLA_KERNEL_OUTPUT, st, [&]() {
        return output_tc_supported(d)
                   ? launch_output_tc(d, n, ws, Q, K, V, Y, static_cast<char*>(state), L.head_bytes, st)
                   : launch_output(d, n, ws, Q, K, V, Y, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "output");
    return LOLA_OK;
}

int32_t lola_decode_step(const lola_config* cfg, void* state, const float* W, int64_t w_head_stride, const void* q,
                         const void* k, const void* v, void* y, int32_t* written_pos, void* stream) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (!state || !W || !q || !k || !v || !y || w_head_stride < 0 || w_head_stride % 4 != 0)
        return LOLA_ERR_INVALID_ARG;
    if (d.alloc == LOLA_ALLOC_CHUNK) return LOLA_ERR_UNSUPPORTED;   // the decode step is per token
    if (d.score != LOLA_SCORE_SRE) return LOLA_ERR_UNSUPPORTED;     // the state keeps no window scores
    const void* ptrs[] = {state, W, q, k, v, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return LOLA_ERR_INVALID_ARG;
    if (written_pos && (reinterpret_cast<uintptr_t>(written_pos) & 3)) return LOLA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const Layout L = make_layout(d);
    if (decode_uses_tok_phi(d, w_head_stride)) {
        const cudaError_t e = traced(LOLA_KERNEL_PHI, st, [&]() {
            return launch_tok_phi(d, static_cast<char*>(state), L, W, w_head_stride, q, k, st);
        });
        if (e != cudaSuccess) return cuda_fail(e, "decode step feature map");
    }
    cudaError_t e = traced(LOLA_KERNEL_DECODE, st, [&]() {
        return launch_decode(d, static_cast<char*>(state), L, W, w_head_stride, q, k, v, y, written_pos, st);
    });
    return e == cudaSuccess ? LOLA_OK : cuda_fail(e, "decode step");
}

int32_t lola_read_status(const lola_config* cfg, const void* state, int32_t* host_status, void* stream) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (!state) return LOLA_ERR_INVALID_ARG;
    const Layout L = make_layout(d);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "lola_read_status sync");
    int32_t bad = 0;
    for (int i = 0; i < d.BH; ++i) {
        int32_t w = 0;
        e = cudaMemcpy(&w, static_cast<const char*>(state) + (int64_t)i * L.head_bytes + 4 * HDR_STATUS, 4,
                       cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "lola_read_status copy");
        if (host_status) host_status[i] = w;
        bad |= w;
    }
    return bad ? LOLA_ERR_DEVICE : LOLA_OK;
}

int32_t lola_kernel_timing(int32_t enable) {
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (enable) {
        drain_pending(-1);
        for (int i = 0; i < LOLA_KERNEL_COUNT; ++i) {
            g_total_ms[i] = 0.0;
            g_launches[i] = 0;
        }
    }
    g_trace_on = enable != 0;
    return LOLA_OK;
}

int32_t lola_kernel_time(int32_t id, double* total_ms, int64_t* launches) {
    if (id < 0 || id >= LOLA_KERNEL_COUNT) return LOLA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(g_trace_mu);
    drain_pending(id);
    if (total_ms) *total_ms = g_total_ms[id];
    if (launches) *launches = g_launches[id];
    return LOLA_OK;
}

const char* lola_kernel_name(int32_t id) {
    static const char* names[LOLA_KERNEL_COUNT] = {"state_init", "phi",        "select",     "output",     "decode",
                                                        "phi_q",      "hola_prep",  "hola_state", "hola_cache", "hola_read"};
    return (id >= 0 && id < LOLA_KERNEL_COUNT) ? names[id] : "";
}

int32_t lola_sre_map(const lola_config* cfg, int32_t n, const void* V, const void* workspace, size_t workspace_bytes,
                     float* out, void* stream) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (n < 1 || !V || !workspace || !out) return LOLA_ERR_INVALID_ARG;
    if (!aligned16(V) || !aligned16(workspace) || !aligned16(out)) return LOLA_ERR_INVALID_ARG;
    if ((int64_t)n * d.BH * d.D > ((int64_t)1 << 40)) return LOLA_ERR_UNSUPPORTED;
    const Workspace ws = carve_workspace(d, n, const_cast<void*>(workspace));
    if (workspace_bytes < ws.bytes) return LOLA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = launch_sre_map(d, n, ws, V, out, st);
    return e == cudaSuccess ? LOLA_OK : cuda_fail(e, "sre map");
}

int32_t lola_sre_map_relative(const lola_config* cfg, int32_t n, const void* V, const void* workspace,
                              size_t workspace_bytes, float* out, float* base, void* stream) {
    Dims d;
    int32_t s = to_dims(cfg, &d);
    if (s != LOLA_OK) return s;
    if (n < 1 || !V || !workspace || !out || !base) return LOLA_ERR_INVALID_ARG;
    if (!aligned16(V) || !aligned16(workspace) || !aligned16(out) || !aligned16(base)) return LOLA_ERR_INVALID_ARG;
    if ((int64_t)n * d.BH * d.D > ((int64_t)1 << 40)) return LOLA_ERR_UNSUPPORTED;
    const Workspace ws = carve_workspace(d, n, const_cast<void*>(workspace));
    if (workspace_bytes < ws.bytes) return LOLA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = launch_sre_map_relative(d, n, ws, V, out, base, st);
    return e == cudaSuccess ? LOLA_OK : cuda_fail(e, "relative sre map");
}

int32_t lola_selftest_bounded_wait(int64_t limit_ns, int64_t* host_elapsed_ns, void* stream) {
    if (limit_ns < 1 || limit_ns > 1000000000ll) return LOLA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    bounded_wait_kernel<<<1, 32, 0, st>>>(limit_ns);
    cudaError_t e = cudaGetLastError();
    int64_t out[2] = {0, 0};
    if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(out, g_selftest, sizeof(out), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "lola_selftest_bounded_wait");
    if (host_elapsed_ns) *host_elapsed_ns = out[1];
    return out[0] ? LOLA_OK : LOLA_ERR_DEVICE;
}

int64_t lola_hola_workspace_bytes(const lola_hola_config* cfg, int32_t n) {
    HolaDims d;
    const int32_t s = hola_dims(cfg, n, &d);
    if (s != LOLA_OK) return s;
    return (int64_t)hola_carve(d, n, nullptr).bytes;
}

int32_t lola_hola_prefill(const lola_hola_config* cfg, int32_t n, const void* Q, const void* K, const void* V,
                          const float* alpha, const float* beta, const float* gamma_q, const float* gamma_k,
                          const float* sink, const float* gate, void* Y, float* S_out, float* scores,
                          int32_t* cache, void* workspace, size_t workspace_bytes, void* stream) {
    HolaDims d;
    const int32_t s = hola_dims(cfg, n, &d);
    if (s != LOLA_OK) return s;
    const void* need[] = {Q, K, V, alpha, beta, gamma_q, gamma_k, sink, gate, Y, workspace};
    for (const void* p : need)
        if (!p || !aligned16(p)) return LOLA_ERR_INVALID_ARG;
    const void* opt[] = {S_out, scores, cache};
    for (const void* p : opt)
        if (p && !aligned16(p)) return LOLA_ERR_INVALID_ARG;
    HolaWs ws = hola_carve(d, n, workspace);
    if (workspace_bytes < ws.bytes) return LOLA_ERR_WORKSPACE;
    float* sc = scores ? scores : ws.scores;
    int32_t* cl = cache ? cache : ws.cache;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(ws.status, 0, 16 * (size_t)d.BH, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws.abort_flag, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "workspace status");
    e = traced(LOLA_KERNEL_HOLA_PREP, st, [&]() {
        return launch_hola_prep(d.BH, n, Q, K, gamma_q, gamma_k, ws.xtile, ws.qt, ws.kt, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "rows");
    e = traced(LOLA_KERNEL_HOLA_STATE, st, [&]() {
        return launch_hola_state_tc(d.BH, n, ws.xtile, V, alpha, beta, ws.ystate, sc, S_out, ws.status, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "delta-rule state");
    e = traced(LOLA_KERNEL_HOLA_CACHE, st, [&]() { return launch_hola_cache(d.BH, n, d.w, d.chunk, d.nck, sc, cl, st); });
    if (e != cudaSuccess) return cuda_fail(e, "persistent cache");
    e = traced(LOLA_KERNEL_HOLA_READ, st, [&]() {
        return launch_output_tc_hola(d.BH, d.Hh, n, d.w, d.chunk, ws.qt, ws.kt, V, Y, cl, d.nck, ws.ystate, sink, gate,
                                     ws.status, ws.abort_flag, st);
    });
    return e == cudaSuccess ? LOLA_OK : cuda_fail(e, "cache read");
}

int32_t lola_hola_status(const lola_hola_config* cfg, int32_t n, const void* workspace, int32_t* host_status,
                         void* stream) {
    HolaDims d;
    const int32_t s = hola_dims(cfg, n, &d);
    if (s != LOLA_OK) return s;
    if (!workspace) return LOLA_ERR_INVALID_ARG;
    const HolaWs ws = hola_carve(d, n, const_cast<void*>(workspace));
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "lola_hola_status sync");
    std::vector<int32_t> words(4 * (size_t)d.BH);
    e = cudaMemcpy(words.data(), ws.status, 16 * (size_t)d.BH, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "lola_hola_status copy");
    int32_t bad = 0;
    for (int i = 0; i < d.BH; ++i) {
        if (host_status) host_status[i] = words[4 * (size_t)i + HDR_STATUS];
        bad |= words[4 * (size_t)i + HDR_STATUS];
    }
    return bad ? LOLA_ERR_DEVICE : LOLA_OK;
}

}  // extern "C"
