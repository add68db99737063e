// K3: co-normalised LoLA output for every query, in parallel over (head, chunk).
//
// LoLA reading notes (arXiv 2505.23666v3), section 2.5, Eq. 14:
//   y_t = (H_t^T phi(q_t) + sum_{j in G_t ∪ W_t} a_tj v_j) / (phi(q_t)^T s_t + sum a_tj),
//   a_tj = exp(q_t . k_j / sqrt(d_k)).
// With w_j the step at which key j was written (none: never), key j is exact for
// query t iff j <= t < w_j, and in the linear memory iff w_j <= t.  From the chunk-start
// snapshot (H_c, s_c, cache positions) taken before step c0, every query t of the chunk
// [c0, c0 + C) reads
//   exact:  the cache before c0 ∪ the window range [c0 - eta, t], masked by t < w_j;
//   linear: H_c^T phi(q_t) + sum_{c0 <= w_j <= t} (phi(q_t) . phi(k_j)) v_j over the same
//           pool (the keys written inside the chunk), with s_c and the same weights;
// the softmax part uses an online maximum m; the linear part is kept unscaled and
// joined at the end as (O_soft + e^{-m} O_lin) / (l_soft + e^{-m} l_lin), which is
// Eq. 14 for every m and stays finite when no key is exact.
//
// This version is CUDA-core float32: 8 warps per CTA, 8 query rows per warp, pool keys
// staged 32 at a time in shared memory.
#include "lola_internal.cuh"

namespace lola {
namespace {

constexpr int kOutThreads = 256;
constexpr int kOutWarps = kOutThreads / kWarp;
constexpr int kRowsPerWarp = 8;
constexpr int kSubRows = kOutWarps * kRowsPerWarp;   // 64 query rows per pass
constexpr int kKeyTile = 32;

struct OutArgs {
    int n, eta, lam, chunk, nck, read_mask;
    const void* Q;
    const void* K;
    const void* V;
    void* Y;
    const float* phiQ;     // [BH][n][D]
    const float* phiK;     // [BH][n][D]
    const int32_t* wstep;  // [BH][n]
    const float* snapH;    // [BH][nck][D*DV]
    const float* snapS;    // [BH][nck][D]
    const int32_t* snapC;  // [BH][nck][lam]
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kOutThreads, 1) output_kernel(const OutArgs a) {
    constexpr int DK = D;
    constexpr int NI = DV / 32;
    extern __shared__ __align__(16) float sm[];
    float* Hs = sm;                              // [D][DV]
    float* sS = Hs + D * DV;                     // [D]
    float* qs = sS + D;                          // [kSubRows][DK]
    float* pq = qs + kSubRows * DK;              // [kSubRows][D]
    float* Kt = pq + kSubRows * D;               // [kKeyTile][DK + 1]
    float* Vt = Kt + kKeyTile * (DK + 1);        // [kKeyTile][DV]
    float* Pk = Vt + kKeyTile * DV;              // [kKeyTile][D + 1]
    float* pw = Pk + kKeyTile * (D + 1);         // [warps][kRowsPerWarp][kKeyTile] softmax weights
    float* lw = pw + kOutWarps * kRowsPerWarp * kKeyTile;  // linear weights
    int* kpos = reinterpret_cast<int*>(lw + kOutWarps * kRowsPerWarp * kKeyTile);
    int* kw = kpos + kKeyTile;

    const int c = blockIdx.x, bh = blockIdx.y;
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int n = a.n;
    const int c0 = c * a.chunk, c1 = min(n, c0 + a.chunk);
    const int wlo = max(0, c0 - a.eta);
    const int P = a.lam + (c1 - wlo);
    const float scale = 1.0f / sqrtf((float)DK);
    const T* Q = static_cast<const T*>(a.Q);
    const T* K = static_cast<const T*>(a.K);
    const T* V = static_cast<const T*>(a.V);
    const int64_t row0 = (int64_t)bh * n;
    const int32_t* wst = a.wstep + row0;
    const int32_t* cpos = a.snapC + ((int64_t)bh * a.nck + c) * a.lam;

    {
        const float* sh = a.snapH + ((int64_t)bh * a.nck + c) * D * DV;
        for (int i = tid; i < D * DV; i += kOutThreads) Hs[i] = sh[i];
        for (int i = tid; i < D; i += kOutThreads) sS[i] = a.snapS[((int64_t)bh * a.nck + c) * D + i];
    }

    for (int t0 = c0; t0 < c1; t0 += kSubRows) {
        __syncthreads();
        for (int i = tid; i < kSubRows * DK; i += kOutThreads) {
            const int r = i / DK, t = t0 + r;
            qs[i] = t < c1 ? IO<T>::ld(Q, (row0 + t) * DK + (i % DK)) : 0.f;
        }
        for (int i = tid; i < kSubRows * D; i += kOutThreads) {
            const int r = i / D, t = t0 + r;
            pq[i] = t < c1 ? a.phiQ[(row0 + t) * D + (i % D)] : 0.f;
        }
        __syncthreads();

        float accs[kRowsPerWarp][NI], accl[kRowsPerWarp][NI], mrow[kRowsPerWarp], lsr[kRowsPerWarp],
            llr[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float* pr = pq + (warp * kRowsPerWarp + i) * D;
            float lin = 0.f;
#pragma unroll
            for (int m = 0; m < D / 32; ++m) lin = fmaf(pr[lane + 32 * m], sS[lane + 32 * m], lin);
            llr[i] = warp_sum(lin);
#pragma unroll
            for (int q = 0; q < NI; ++q) {
                float acc = 0.f;
                for (int k = 0; k < D; ++k) acc = fmaf(pr[k], Hs[k * DV + lane + 32 * q], acc);
                accl[i][q] = acc;
                accs[i][q] = 0.f;
            }
            mrow[i] = -INFINITY;
            lsr[i] = 0.f;
        }

        for (int u0 = 0; u0 < P; u0 += kKeyTile) {
            __syncthreads();
            if (tid < kKeyTile) {
                const int u = u0 + tid;
                int p = -1;
                if (u < P) p = u < a.lam ? cpos[u] : wlo + (u - a.lam);
                kpos[tid] = p;
                kw[tid] = p >= 0 ? wst[p] : -1;
            }
            __syncthreads();
            for (int i = tid; i < kKeyTile * DK; i += kOutThreads) {
                const int j = i / DK, cc = i % DK;
                const int p = kpos[j];
                Kt[j * (DK + 1) + cc] = p >= 0 ? IO<T>::ld(K, (row0 + p) * DK + cc) : 0.f;
            }
            for (int i = tid; i < kKeyTile * DV; i += kOutThreads) {
                const int j = i / DV, cc = i % DV;
                const int p = kpos[j];
                Vt[j * DV + cc] = p >= 0 ? IO<T>::ld(V, (row0 + p) * DV + cc) : 0.f;
            }
            for (int i = tid; i < kKeyTile * D; i += kOutThreads) {
                const int j = i / D, cc = i % D;
                const int p = kpos[j];
                Pk[j * (D + 1) + cc] = p >= 0 ? a.phiK[(row0 + p) * D + cc] : 0.f;
            }
            __syncthreads();

            const int p = kpos[lane];
            const int w = kw[lane];
            float* pws = pw + warp * kRowsPerWarp * kKeyTile;
            float* lws = lw + warp * kRowsPerWarp * kKeyTile;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const int r = warp * kRowsPerWarp + i;
                const int t = t0 + r;
                const bool row_ok = t < c1;
                // (the read mask's HIDE_CACHE keeps only the window: t - eta < p)
                const bool vs = row_ok && p >= 0 && p <= t && (w < 0 || w > t) &&
                                (!(a.read_mask & LOLA_READ_HIDE_CACHE) || p > t - a.eta);
                const bool vl = row_ok && p >= 0 && w >= c0 && w <= t;
                float sc = -INFINITY;
                if (vs) {
                    const float* qr = qs + r * DK;
                    const float* kr = Kt + lane * (DK + 1);
                    float acc = 0.f;
#pragma unroll 8
                    for (int cc = 0; cc < DK; ++cc) acc = fmaf(qr[cc], kr[cc], acc);
                    sc = acc * scale;
                }
                float lv = 0.f;
                if (vl) {
                    const float* pr = pq + r * D;
                    const float* kr = Pk + lane * (D + 1);
#pragma unroll 8
                    for (int cc = 0; cc < D; ++cc) lv = fmaf(pr[cc], kr[cc], lv);
                }
                const float mt = warp_max(sc);
                const float mnew = fmaxf(mrow[i], mt);
                if (mnew > mrow[i]) {
                    const float f = mrow[i] == -INFINITY ? 0.f : expf(mrow[i] - mnew);
#pragma unroll
                    for (int q = 0; q < NI; ++q) accs[i][q] *= f;
                    lsr[i] *= f;
                    mrow[i] = mnew;
                }
                const float pv = vs ? expf(sc - mrow[i]) : 0.f;
                lsr[i] += warp_sum(pv);
                llr[i] += warp_sum(lv);
                pws[i * kKeyTile + lane] = pv;
                lws[i * kKeyTile + lane] = lv;
            }
            __syncwarp();
            for (int j = 0; j < kKeyTile; ++j) {
                float vj[NI];
#pragma unroll
                for (int q = 0; q < NI; ++q) vj[q] = Vt[j * DV + lane + 32 * q];
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    const float ps = pws[i * kKeyTile + j];
                    const float pl = lws[i * kKeyTile + j];
#pragma unroll
                    for (int q = 0; q < NI; ++q) {
                        accs[i][q] = fmaf(ps, vj[q], accs[i][q]);
                        accl[i][q] = fmaf(pl, vj[q], accl[i][q]);
                    }
                }
            }
            __syncwarp();
        }

        T* Y = static_cast<T*>(a.Y);
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int t = t0 + warp * kRowsPerWarp + i;
            if (t >= c1) continue;
            const bool any = mrow[i] != -INFINITY;
            const float em = any ? expf(-mrow[i]) : 1.f;
            // HIDE_STATE: the linear terms stay out of the read (then the window's current
            // token makes any true)
            const float el = (a.read_mask & LOLA_READ_HIDE_STATE) ? 0.f : em;
            const float den = any ? fmaf(el, llr[i], lsr[i]) : llr[i];
            const float inv = 1.0f / den;
#pragma unroll
            for (int q = 0; q < NI; ++q) {
                const float num = any ? fmaf(el, accl[i][q], accs[i][q]) : accl[i][q];
                IO<T>::st(Y, (row0 + t) * DV + lane + 32 * q, num * inv);
            }
        }
    }
}

template <int D, int DV, typename T>
cudaError_t launch_output_t(const Dims& d, const OutArgs& a, cudaStream_t st) {
    constexpr int DK = D;
    const size_t smem = sizeof(float) * (D * DV + D + kSubRows * DK + kSubRows * D + kKeyTile * (DK + 1) +
                                         kKeyTile * DV + kKeyTile * (D + 1) +
                                         2 * kOutWarps * kRowsPerWarp * kKeyTile) +
                        sizeof(int) * 2 * kKeyTile;
    auto kern = output_kernel<D, DV, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.nck, d.BH), kOutThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_output(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K, const void* V,
                          void* Y, cudaStream_t st) {
    OutArgs a;
    a.n = n;
    a.eta = d.eta;
    a.lam = d.lam;
    a.chunk = ws.snap_interval;
    a.nck = ws.nck;
    a.read_mask = d.read_mask;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.Y = Y;
    a.phiQ = ws.phiQ;
    a.phiK = ws.phiK;
    a.wstep = ws.wstep;
    a.snapH = ws.snapH;
    a.snapS = ws.snapS;
    a.snapC = ws.snapC;
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_output_t<128, 128, __nv_bfloat16>(d, a, st) : launch_output_t<128, 128, float>(d, a, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_output_t<64, 64, __nv_bfloat16>(d, a, st) : launch_output_t<64, 64, float>(d, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
