// Prefill with a query-dependent cache score in place of the SRE: the scoring ablation of
// the LoLA reading notes (section 4.4, Table 4; appendix F names the scores, whose formulas
// the notes do not reproduce).  Reading taken (the oracle's lola_run_fixed_score): with
// e = exp(q_t . k_j / sqrt(d_k)), the softmax branch's weight, and l = phi(q_t) . phi(k_j),
// the linear branch's, key j's score sums over the eta queries of the steps it spends in
// the window (t = j .. j + eta - 1):
//   kernel squared error (e - l)^2, kernel absolute error |e - l|, ratio l / e, attention e.
// The score is complete when the key leaves the window and never changes after, so nothing
// is rescored: at every eviction the candidates are the cache and the evictee, and when
// they exceed lambda the lowest (score, position) is written -- the cache is always the
// lambda highest-scored evicted keys.  That makes the allocation chain-free: key j is
// written at step max(j, p) + eta, p the position of the lambda-th key (in position order)
// that outranks it (a higher score, or an equal score and a later position), or never if
// that step is past the sequence.  The kernels:
//   fixed_score_kernel   score[j] over its eta window queries (64 keys per CTA; the band of
//                        queries staged 32 at a time);
//   fixed_wstep_kernel   the closed-form write step of every key, and the per-step log;
//   fixed_delta_kernel   per snapshot interval [cP, cP + P): the sum of phi(k) v^T and
//                        phi(k) over the keys written in it, in step order;
//   fixed_prefix_kernel  snapshots H_c, s_c as prefix sums of those deltas (the memory
//                        before step cP) and the final H, s;
//   fixed_export_kernel  the cache before every snapshot (the evicted keys not yet written,
//                        in position order), the final cache and window into the state.
// The output kernels then read the write steps and snapshots exactly as for the SRE rule
// (key j exact for query t iff j <= t < w_j; linear iff w_j <= t).
#include "lola_internal.cuh"

namespace lola {
namespace {

constexpr int kFkKeys = 64;      // keys per score CTA
constexpr int kFkQ = 32;         // queries staged at a time
constexpr int kFkThreads = 256;  // 4 query lanes per key

struct FixedArgs {
    int n, eta, lam, kind, snap, nck;
    const void* Q;           // io [BH][n][DK]
    const void* K;
    const void* V;           // io [BH][n][DV]
    const float* phiQ;       // [BH][n][D] float32
    const float* phiK;
    float* score;            // [BH][n]
    int32_t* wstep;          // [BH][n]
    int32_t* wpos;           // [BH][n] (-1 filled before fixed_wstep_kernel)
    float* dH;               // [BH][nck][D*DV]
    float* dS;               // [BH][nck][D]
    float* snapH;            // [BH][nck][D*DV] float32, or
    __nv_bfloat16* snapHb;   // the same in bf16 (exactly one of the two is set)
    float* snapS;            // [BH][nck][D]
    int32_t* snapC;          // [BH][nck][lam]
    char* state;
    Layout L;
};

// CTA (key block, head): keys j0 .. j0 + 63 with their rows (k widened, phi(k)) in shared
// memory; the queries of steps j0 .. j0 + 63 + eta - 1 pass through kFkQ at a time.  Thread
// (j = tid % 64, u = tid / 64) takes the staged queries r = u, u + 4, ... and adds f(e, l)
// for those inside j's window steps; the four partials of j are added in u order.
template <int DK, int D, typename T>
__global__ void __launch_bounds__(kFkThreads) fixed_score_kernel(const FixedArgs a) {
    extern __shared__ __align__(16) float fsm[];
    float* Ks = fsm;                                  // [64][DK + 1]
    float* Ps = Ks + kFkKeys * (DK + 1);              // [64][D + 1]
    float* Qs = Ps + kFkKeys * (D + 1);               // [kFkQ][DK + 1]
    float* PQs = Qs + kFkQ * (DK + 1);                // [kFkQ][D + 1]
    float* part = PQs + kFkQ * (D + 1);               // [4][64]
    const int tid = threadIdx.x, bh = blockIdx.y, n = a.n;
    const int j0 = blockIdx.x * kFkKeys;
    const int64_t row0 = (int64_t)bh * n;
    const T* Kin = static_cast<const T*>(a.K) + row0 * DK;
    const T* Qin = static_cast<const T*>(a.Q) + row0 * DK;
    for (int i = tid; i < kFkKeys * DK; i += kFkThreads) {
        const int r = i / DK, c = i % DK;
        Ks[r * (DK + 1) + c] = j0 + r < n ? IO<T>::ld(Kin, (int64_t)(j0 + r) * DK + c) : 0.f;
    }
    for (int i = tid; i < kFkKeys * D; i += kFkThreads) {
        const int r = i / D, c = i % D;
        Ps[r * (D + 1) + c] = j0 + r < n ? a.phiK[(row0 + j0 + r) * D + c] : 0.f;
    }
    const int jl = tid % kFkKeys, u = tid / kFkKeys, j = j0 + jl;
    const float scale = rsqrtf((float)DK);
    float acc = 0.f;
    const int tend = min(n, j0 + kFkKeys + a.eta - 1);
    for (int q0 = j0; q0 < tend; q0 += kFkQ) {
        __syncthreads();   // key rows staged / the previous query tile consumed
        for (int i = tid; i < kFkQ * DK; i += kFkThreads) {
            const int r = i / DK, c = i % DK;
            Qs[r * (DK + 1) + c] = q0 + r < n ? IO<T>::ld(Qin, (int64_t)(q0 + r) * DK + c) : 0.f;
        }
        for (int i = tid; i < kFkQ * D; i += kFkThreads) {
            const int r = i / D, c = i % D;
            PQs[r * (D + 1) + c] = q0 + r < n ? a.phiQ[(row0 + q0 + r) * D + c] : 0.f;
        }
        __syncthreads();
        for (int r = u; r < kFkQ; r += kFkThreads / kFkKeys) {
            const int t = q0 + r;
            if (t >= n || t < j || t >= j + a.eta || j >= n) continue;
            float dot = 0.f, lin = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) dot = fmaf(Ks[jl * (DK + 1) + c], Qs[r * (DK + 1) + c], dot);
#pragma unroll 8
            for (int c = 0; c < D; ++c) lin = fmaf(Ps[jl * (D + 1) + c], PQs[r * (D + 1) + c], lin);
            const float e = expf(dot * scale);
            float f;
            switch (a.kind) {
                case LOLA_SCORE_KERNEL_SQ: f = (e - lin) * (e - lin); break;
                case LOLA_SCORE_KERNEL_ABS: f = fabsf(e - lin); break;
                case LOLA_SCORE_KERNEL_RATIO: f = lin / e; break;
                default: f = e; break;
            }
            acc += f;
        }
    }
    part[u * kFkKeys + jl] = acc;
    __syncthreads();
    if (tid < kFkKeys && j0 + tid < n) {
        float s = 0.f;
#pragma unroll
        for (int v = 0; v < kFkThreads / kFkKeys; ++v) s += part[v * kFkKeys + tid];
        a.score[row0 + j0 + tid] = s;
    }
}

// One thread per key: the keys that outrank j (a higher score, or an equal score and a later
// position) are counted in position order until lambda of them are found at position p; j is
// written at max(j, p) + eta when that step exists (lambda = 0: at j + eta).
__global__ void fixed_wstep_kernel(const FixedArgs a) {
    const int bh = blockIdx.y, n = a.n;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const int64_t row0 = (int64_t)bh * n;
    const float* sc = a.score + row0;
    const float sj = sc[j];
    int p = -1;
    if (a.lam == 0) {
        p = j;
    } else {
        int cnt = 0;
        for (int i = 0; i < n; ++i) {
            const float si = sc[i];
            if (si > sj || (si == sj && i > j)) {
                if (++cnt == a.lam) {
                    p = i;
                    break;
                }
            }
        }
    }
    int w = -1;
    if (p >= 0) {
        const int64_t t = (int64_t)max(j, p) + a.eta;
        if (t <= n - 1) w = (int)t;
    }
    a.wstep[row0 + j] = w;
    if (w >= 0) a.wpos[row0 + w] = j;   // the closed form writes at most one key per step
}

// CTA (interval c, head), 512 threads, thread (warp w, lane l) owning H rows w * (D/16) ..
// and columns l * (DV/32) ..: the keys written at steps [cP, cP + P), in step order.
template <int D, int DV, typename T>
__global__ void __launch_bounds__(512) fixed_delta_kernel(const FixedArgs a) {
    constexpr int HR = D / 16, HC = DV / 32;
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int c = blockIdx.x, bh = blockIdx.y, n = a.n;
    const int64_t row0 = (int64_t)bh * n;
    const T* Vin = static_cast<const T*>(a.V) + row0 * DV;
    float h[HR * HC];
#pragma unroll
    for (int i = 0; i < HR * HC; ++i) h[i] = 0.f;
    float s = 0.f;
    const int t1 = min(n, (c + 1) * a.snap);
    for (int t = c * a.snap; t < t1; ++t) {
        const int j = a.wpos[row0 + t];   // uniform across the CTA
        if (j < 0) continue;
        const float* ph = a.phiK + (row0 + j) * D;
        float vv[HC];
#pragma unroll
        for (int q = 0; q < HC; ++q) vv[q] = IO<T>::ld(Vin, (int64_t)j * DV + lane * HC + q);
#pragma unroll
        for (int r = 0; r < HR; ++r) {
            const float f = ph[warp * HR + r];
#pragma unroll
            for (int q = 0; q < HC; ++q) h[r * HC + q] = fmaf(f, vv[q], h[r * HC + q]);
        }
        if (tid < D) s += ph[tid];
    }
    float* dH = a.dH + ((int64_t)bh * a.nck + c) * D * DV;
#pragma unroll
    for (int r = 0; r < HR; ++r)
#pragma unroll
        for (int q = 0; q < HC; ++q) dH[(warp * HR + r) * DV + lane * HC + q] = h[r * HC + q];
    if (tid < D) a.dS[((int64_t)bh * a.nck + c) * D + tid] = s;
}

// Thread per element of H (and of s): the snapshots are the prefix sums of the interval
// deltas (snapshot c = the memory before step cP), the final sum goes to the state.
template <int D, int DV>
__global__ void fixed_prefix_kernel(const FixedArgs a) {
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= D * DV + D) return;
    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    float acc = 0.f;
    if (e < D * DV) {
        for (int c = 0; c < a.nck; ++c) {
            const int64_t sc = (int64_t)bh * a.nck + c;
            if (a.snapHb) a.snapHb[sc * D * DV + e] = __float2bfloat16_rn(acc);
            else a.snapH[sc * D * DV + e] = acc;
            acc += a.dH[sc * D * DV + e];
        }
        reinterpret_cast<float*>(rec + a.L.H)[e] = acc;
    } else {
        const int r = e - D * DV;
        for (int c = 0; c < a.nck; ++c) {
            const int64_t sc = (int64_t)bh * a.nck + c;
            a.snapS[sc * D + r] = acc;
            acc += a.dS[sc * D + r];
        }
        reinterpret_cast<float*>(rec + a.L.s)[r] = acc;
    }
}

// CTA per head: the cache before each snapshot -- the evicted keys not yet written,
// i + eta <= cP - 1 and (w_i < 0 or w_i >= cP), at most lambda in position order, -1 after --
// one warp per list; the final cache (c == nck), its rows, the header and the window ring.
template <int D, int DV, typename T>
__global__ void __launch_bounds__(512) fixed_export_kernel(const FixedArgs a) {
    const int tid = threadIdx.x, bh = blockIdx.x, n = a.n;
    const int64_t row0 = (int64_t)bh * n;
    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    const int32_t* ws = a.wstep + row0;
    const int warp = tid / kWarp, lane = tid % kWarp, nwarps = blockDim.x / kWarp;
    for (int c = warp; c <= a.nck; c += nwarps) {
        const int tb = c < a.nck ? c * a.snap : n;        // "before step tb"
        int32_t* out = c < a.nck ? a.snapC + ((int64_t)bh * a.nck + c) * a.lam
                                 : reinterpret_cast<int32_t*>(rec + a.L.c_pos);
        int cnt = 0;
        const int ilast = tb - 1 - a.eta;                  // evicted before step tb: i <= ilast
        for (int i0 = 0; i0 <= ilast; i0 += kWarp) {
            const int i = i0 + lane;
            const bool in = i <= ilast && (ws[i] < 0 || ws[i] >= tb);
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (in) {
                const int slot = cnt + __popc(m & ((1u << lane) - 1u));
                if (slot < a.lam) out[slot] = i;
            }
            cnt += __popc(m);
        }
        for (int sl = cnt + lane; sl < a.lam; sl += kWarp) out[sl] = -1;
        if (c == a.nck && lane == 0) {
            int32_t* hdr = reinterpret_cast<int32_t*>(rec);
            if (cnt > a.lam) atomicOr(&hdr[HDR_STATUS], (int)ST_BAD_STATE);   // the closed form broke capacity
            int nw = 0;
            for (int i = 0; i < n; ++i) nw += ws[i] >= 0;
            hdr[HDR_T] = n;
            hdr[HDR_NCACHE] = min(cnt, a.lam);
            hdr[HDR_NWRITTEN] = nw;
        }
    }
    __syncthreads();
    const T* Kin = static_cast<const T*>(a.K) + row0 * D;
    const T* Vin = static_cast<const T*>(a.V) + row0 * DV;
    const int32_t* cp = reinterpret_cast<const int32_t*>(rec + a.L.c_pos);
    T* ck = reinterpret_cast<T*>(rec + a.L.c_k);
    T* cv = reinterpret_cast<T*>(rec + a.L.c_v);
    float* cph = reinterpret_cast<float*>(rec + a.L.c_phi);
    for (int i = tid; i < a.lam * D; i += blockDim.x) {
        const int sl = i / D, r = i % D, p = cp[sl];
        if (p < 0) continue;
        ck[(int64_t)sl * D + r] = Kin[(int64_t)p * D + r];
        cph[(int64_t)sl * D + r] = a.phiK[(row0 + p) * D + r];
    }
    for (int i = tid; i < a.lam * DV; i += blockDim.x) {
        const int sl = i / DV, q = i % DV, p = cp[sl];
        if (p >= 0) cv[(int64_t)sl * DV + q] = Vin[(int64_t)p * DV + q];
    }
    int32_t* wp = reinterpret_cast<int32_t*>(rec + a.L.win_pos);
    T* wk = reinterpret_cast<T*>(rec + a.L.win_k);
    T* wv = reinterpret_cast<T*>(rec + a.L.win_v);
    float* wph = reinterpret_cast<float*>(rec + a.L.win_phi);
    for (int p = max(0, n - a.eta) + tid; p < n; p += blockDim.x) {
        const int e = p % a.eta;
        wp[e] = p;
        for (int r = 0; r < D; ++r) {
            wk[(int64_t)e * D + r] = Kin[(int64_t)p * D + r];
            wph[(int64_t)e * D + r] = a.phiK[(row0 + p) * D + r];
        }
        for (int q = 0; q < DV; ++q) wv[(int64_t)e * DV + q] = Vin[(int64_t)p * DV + q];
    }
}

template <int D, int DV, typename T>
cudaError_t launch_fixed_t(const Dims& d, const FixedArgs& a, cudaStream_t st) {
    const int n = a.n;
    const size_t smem = sizeof(float) * ((size_t)kFkKeys * (D + 1) * 2 + (size_t)kFkQ * (D + 1) * 2 + 4 * kFkKeys);
    auto ks = fixed_score_kernel<D, D, T>;
    cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ks<<<dim3((n + kFkKeys - 1) / kFkKeys, d.BH), kFkThreads, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = cudaMemsetAsync(a.wpos, 0xff, sizeof(int32_t) * (size_t)d.BH * n, st);
    if (e != cudaSuccess) return e;
    fixed_wstep_kernel<<<dim3((n + 255) / 256, d.BH), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fixed_delta_kernel<D, DV, T><<<dim3(a.nck, d.BH), 512, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fixed_prefix_kernel<D, DV><<<dim3((D * DV + D + 255) / 256, d.BH), 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fixed_export_kernel<D, DV, T><<<d.BH, 512, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fixed_select(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K,
                                const void* V, char* state, const Layout& L, cudaStream_t st) {
    FixedArgs a;
    a.n = n;
    a.eta = d.eta;
    a.lam = d.lam;
    a.kind = d.score;
    a.snap = ws.snap_interval;
    a.nck = ws.nck;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.phiQ = ws.phiQ;
    a.phiK = ws.phiK;
    a.score = ws.score;
    a.wstep = ws.wstep;
    a.wpos = ws.wpos;
    a.dH = ws.dH;
    a.dS = ws.dS;
    a.snapH = ws.snapH;
    a.snapHb = ws.snapHb;
    a.snapS = ws.snapS;
    a.snapC = ws.snapC;
    a.state = state;
    a.L = L;
    if (!a.phiQ || !a.score || !a.dH || !a.dS || d.eta < 1) return cudaErrorInvalidValue;
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128 && d.dk == 128)
        return bf ? launch_fixed_t<128, 128, __nv_bfloat16>(d, a, st) : launch_fixed_t<128, 128, float>(d, a, st);
    if (d.D == 64 && d.dv == 64 && d.dk == 64)
        return bf ? launch_fixed_t<64, 64, __nv_bfloat16>(d, a, st) : launch_fixed_t<64, 64, float>(d, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
