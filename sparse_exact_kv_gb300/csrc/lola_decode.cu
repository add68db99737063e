// K4: one LoLA decode step for every head, state updated in place.
//
// LoLA reading notes (arXiv 2505.23666v3), sections 2.3-2.5 (Eqs. 10-14): the new token
// enters the window; the token leaving it joins the cache as a candidate; if the
// candidates exceed lambda the smallest-SRE one (ties: older) is written into (H, s);
// y is the co-normalised read after the write.  Appendix B's bounded state is what each
// head streams: H (D x d_v float32, read and written), s, the eta + lambda exact KV, and
// the per-slot bookkeeping c_phi, c_N = H^T phi(k), c_z = s^T phi(k) that lets the step
// score the cache without recomputing H^T phi(k) for every slot.
//
// One CTA of 512 threads per head.  The arithmetic that decides which candidate is
// written (phi, the evictee's H^T phi, the slot SREs and their updates) uses the same
// thread mapping and operation order as the prefill selection kernel, so a decode step
// continues a prefill bit for bit.
#include <climits>

#include "lola_internal.cuh"

namespace lola {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / kWarp;
constexpr int kSG = 8;
constexpr int kSlotsPerPass = kDecThreads / kSG;   // 64

struct DecArgs {
    char* state;
    Layout L;
    int eta, lam, Hh;
    const float* W;
    int64_t w_head_stride;
    const void* q;
    const void* k;
    const void* v;
    void* y;
    int32_t* written_pos;
};

__device__ __forceinline__ int slot_dim(int sub, int i) { return 4 * sub + 32 * (i >> 2) + (i & 3); }

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const DecArgs a) {
    constexpr int DK = D;
    constexpr int PD = D / kSG, PV = DV / kSG;
    constexpr int NRG = kDecThreads / DV;
    constexpr int HR = D / NRG;
    extern __shared__ __align__(16) float sm[];
    float* Ws = sm;                              // [D/2][DK+1]
    float* xq = Ws + (D / 2) * (DK + 1);         // [DK]
    float* xk = xq + DK;                         // [DK]  new key
    float* xv = xk + DK;                         // [DV]  new value
    float* ek = xv + DV;                         // [DK]  evictee key
    float* evv = ek + DK;                        // [DV]  evictee value
    float* phq = evv + DV;                       // [D]
    float* phe = phq + D;                        // [D]
    float* wphi = phe + D;                       // [D]   written phi
    float* wv = wphi + D;                        // [DV]  written v
    float* s_sm = wv + DV;                       // [D]
    float* red = s_sm + D;                       // [NRG][DV]
    float* Ne = red + NRG * DV;                  // [DV]
    float* sre = Ne + DV;                        // [lam]   slot SRE^2, then softmax weights
    float* sc = sre + a.lam;                     // [eta + lam] scores
    float* misc = sc + a.eta + a.lam;            // ze, vve, ese, ...
    int* imisc = reinterpret_cast<int*>(misc + 8);

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x, h = bh % a.Hh;
    const int eta = a.eta, lam = a.lam;
    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    int32_t* hdr = reinterpret_cast<int32_t*>(rec);
    const int t = hdr[HDR_T];
    const int nc = hdr[HDR_NCACHE];
    float* Hg = reinterpret_cast<float*>(rec + a.L.H);
    float* sg = reinterpret_cast<float*>(rec + a.L.s);
    int32_t* winpos = reinterpret_cast<int32_t*>(rec + a.L.win_pos);
    T* wk = reinterpret_cast<T*>(rec + a.L.win_k);
    T* wvv = reinterpret_cast<T*>(rec + a.L.win_v);
    int32_t* cpos = reinterpret_cast<int32_t*>(rec + a.L.c_pos);
    T* ck = reinterpret_cast<T*>(rec + a.L.c_k);
    T* cv = reinterpret_cast<T*>(rec + a.L.c_v);
    float* cphi = reinterpret_cast<float*>(rec + a.L.c_phi);
    float* cN = reinterpret_cast<float*>(rec + a.L.c_N);
    float* cz = reinterpret_cast<float*>(rec + a.L.c_z);
    const T* qin = static_cast<const T*>(a.q) + (int64_t)bh * DK;
    const T* kin = static_cast<const T*>(a.k) + (int64_t)bh * DK;
    const T* vin = static_cast<const T*>(a.v) + (int64_t)bh * DV;

    const bool ev = t >= eta;
    const int e = t - eta;
    const int ring = eta > 0 ? t % eta : 0;

    // ---- 1. load W, the new token, the evictee, H and s ----
    const float* Wh = a.W + (int64_t)h * a.w_head_stride;
    for (int i = tid; i < (D / 2) * DK; i += kDecThreads) Ws[(i / DK) * (DK + 1) + (i % DK)] = Wh[i];
    if (tid < DK) {
        xq[tid] = IO<T>::ld(qin, tid);
        xk[tid] = IO<T>::ld(kin, tid);
        if (ev) ek[tid] = eta > 0 ? IO<T>::ld(wk, (int64_t)ring * DK + tid) : IO<T>::ld(kin, tid);
    }
    if (tid < DV) {
        xv[tid] = IO<T>::ld(vin, tid);
        if (ev) evv[tid] = eta > 0 ? IO<T>::ld(wvv, (int64_t)ring * DV + tid) : IO<T>::ld(vin, tid);
    }
    const int hj = tid % DV, hrg = tid / DV;
    float hreg[HR];
#pragma unroll
    for (int r = 0; r < HR; ++r) hreg[r] = Hg[(hrg + NRG * r) * DV + hj];
    if (tid < D) s_sm[tid] = sg[tid];
    __syncthreads();
    if (eta > 0 && ev && tid == 0 && winpos[ring] != e) atomicOr(&hdr[HDR_STATUS], (int)ST_BAD_STATE);

    // ---- 2. phi(q), phi(k_e) ----
    if (warp == 0) {
        float ph[D / 32];
        phi_warp<DK, D>(xq, Ws, lane, ph);
#pragma unroll
        for (int m = 0; m < D / 32; ++m) phq[lane + 32 * m] = ph[m];
    } else if (warp == 1 && ev) {
        float ph[D / 32];
        phi_warp<DK, D>(ek, Ws, lane, ph);
#pragma unroll
        for (int m = 0; m < D / 32; ++m) phe[lane + 32 * m] = ph[m];
    }
    __syncthreads();

    // ---- 3. evictee partial H^T phi_e; slot SREs ----
    if (ev) {
        float pj = 0.f;
#pragma unroll
        for (int r = 0; r < HR; ++r) pj = fmaf(phe[hrg + NRG * r], hreg[r], pj);
        red[hrg * DV + hj] = pj;
    }
    const int sl = tid / kSG, sub = tid % kSG;
    for (int base = 0; base < nc; base += kSlotsPerPass) {
        const int i = base + sl;
        float ss = 0.f, vv = 0.f, z = 0.f;
        if (i < nc) {
            z = cz[i];
#pragma unroll
            for (int q = 0; q < PV; ++q) {
                const int dd = slot_dim(sub, q);
                const float vq = IO<T>::ld(cv, (int64_t)i * DV + dd);
                const float dlt = fmaf(-z, vq, cN[(int64_t)i * DV + dd]);
                ss = fmaf(dlt, dlt, ss);
                vv = fmaf(vq, vq, vv);
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        vv += __shfl_xor_sync(0xffffffffu, vv, 1);
        vv += __shfl_xor_sync(0xffffffffu, vv, 2);
        vv += __shfl_xor_sync(0xffffffffu, vv, 4);
        if (i < nc && sub == 0) sre[i] = z == 0.f ? vv : ss / (z * z);
    }
    __syncthreads();

    // ---- 4. decision (warp 0) ----
    const bool write = ev && (nc + 1 > lam);
    if (warp == 0) {
        float es = INFINITY;
        if (ev) {
            float Nv[DV / 32], ze = 0.f, sse = 0.f, vve = 0.f;
#pragma unroll
            for (int i = 0; i < DV / 32; ++i) {
                float acc = 0.f;
#pragma unroll
                for (int r = 0; r < NRG; ++r) acc += red[r * DV + lane + 32 * i];
                Nv[i] = acc;
                Ne[lane + 32 * i] = acc;
            }
#pragma unroll
            for (int i = 0; i < D / 32; ++i) ze = fmaf(s_sm[lane + 32 * i], phe[lane + 32 * i], ze);
            ze = warp_sum(ze);
#pragma unroll
            for (int i = 0; i < DV / 32; ++i) {
                const float vq = evv[lane + 32 * i];
                const float dlt = fmaf(-ze, vq, Nv[i]);
                sse = fmaf(dlt, dlt, sse);
                vve = fmaf(vq, vq, vve);
            }
            sse = warp_sum(sse);
            vve = warp_sum(vve);
            es = ze == 0.f ? vve : sse / (ze * ze);
            if (lane == 0) misc[0] = ze;
        }
        float bs = INFINITY;
        int bp = INT_MAX, bi = -2;
        for (int i = lane; i < nc; i += kWarp) {
            const int p = cpos[i];
            if (key_less(sre[i], p, bs, bp)) { bs = sre[i]; bp = p; bi = i; }
        }
        if (ev && lane == 0 && key_less(es, e, bs, bp)) { bs = es; bp = e; bi = -1; }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int op = __shfl_xor_sync(0xffffffffu, bp, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (key_less(os, op, bs, bp)) { bs = os; bp = op; bi = oi; }
        }
        if (lane == 0) {
            imisc[0] = write ? bi : -2;     // -1: evictee written; >= 0: slot written
            imisc[1] = write ? bp : -1;
        }
    }
    __syncthreads();
    const int wsel = imisc[0];
    const int wposn = imisc[1];
    const float ze = misc[0];

    // ---- 5. write: phi_w, v_w; H, s, slots ----
    if (write) {
        if (tid < D) wphi[tid] = wsel < 0 ? phe[tid] : cphi[(int64_t)wsel * D + tid];
        if (tid < DV) wv[tid] = wsel < 0 ? evv[tid] : IO<T>::ld(cv, (int64_t)wsel * DV + tid);
        __syncthreads();
        const float wvj = wv[hj];
#pragma unroll
        for (int r = 0; r < HR; ++r) hreg[r] = fmaf(wphi[hrg + NRG * r], wvj, hreg[r]);
        if (tid < D) s_sm[tid] += wphi[tid];
        // every cached slot (and the surviving evictee) absorbs the write
        for (int base = 0; base < nc; base += kSlotsPerPass) {
            const int i = base + sl;
            const bool live = i < nc && i != wsel;
            float g = 0.f;
            if (live) {
#pragma unroll
                for (int q = 0; q < PD; ++q) {
                    const int dd = slot_dim(sub, q);
                    g = fmaf(wphi[dd], cphi[(int64_t)i * D + dd], g);
                }
            }
            g += __shfl_xor_sync(0xffffffffu, g, 1);
            g += __shfl_xor_sync(0xffffffffu, g, 2);
            g += __shfl_xor_sync(0xffffffffu, g, 4);
            if (live) {
#pragma unroll
                for (int q = 0; q < PV; ++q) {
                    const int dd = slot_dim(sub, q);
                    float* p = cN + (int64_t)i * DV + dd;
                    *p = fmaf(g, wv[dd], *p);
                }
                if (sub == 0) cz[i] += g;
            }
        }
        if (wsel >= 0 && warp == kDecWarps - 1) {
            // the evictee survives and takes the written slot, after absorbing the write
            float g = 0.f;
            if (sub < kSG && lane < kSG) {
#pragma unroll
                for (int q = 0; q < PD; ++q) {
                    const int dd = slot_dim(lane, q);
                    g = fmaf(wphi[dd], phe[dd], g);
                }
            }
            g += __shfl_xor_sync(0xffffffffu, g, 1);
            g += __shfl_xor_sync(0xffffffffu, g, 2);
            g += __shfl_xor_sync(0xffffffffu, g, 4);
            if (lane < kSG) {
#pragma unroll
                for (int q = 0; q < PV; ++q) {
                    const int dd = slot_dim(lane, q);
                    cN[(int64_t)wsel * DV + dd] = fmaf(g, wv[dd], Ne[dd]);
                }
                if (lane == 0) cz[wsel] = ze + g;
            }
        }
    }
    int nc_after = nc;
    int slot_new = -1;
    if (ev && !write) { slot_new = nc; nc_after = nc + 1; }
    if (write && wsel >= 0) slot_new = wsel;
    if (slot_new >= 0) {
        if (!write) {
            if (tid < DV) cN[(int64_t)slot_new * DV + tid] = Ne[tid];
            if (tid == 0) cz[slot_new] = ze;
        }
        if (tid < D) cphi[(int64_t)slot_new * D + tid] = phe[tid];
        if (tid < DK) IO<T>::st(ck, (int64_t)slot_new * DK + tid, ek[tid]);
        if (tid < DV) IO<T>::st(cv, (int64_t)slot_new * DV + tid, evv[tid]);
        if (tid == 0) cpos[slot_new] = e;
    }
    // the new token enters the window ring (its previous occupant was the evictee)
    if (eta > 0) {
        if (tid < DK) IO<T>::st(wk, (int64_t)ring * DK + tid, xk[tid]);
        if (tid < DV) IO<T>::st(wvv, (int64_t)ring * DV + tid, xv[tid]);
        if (tid == 0) winpos[ring] = t;
    }
    __syncthreads();

    // ---- 6. output: softmax over window ∪ cache, linear read of (H, s) ----
    const float scale = 1.0f / sqrtf((float)DK);
    const int nwin = min(t + 1, eta);
    const int nkeys = nwin + nc_after;
    // scores: 8 lanes per key
    for (int base = 0; base < nkeys; base += kSlotsPerPass) {
        const int i = base + sl;
        float acc = 0.f;
        if (i < nkeys) {
            const T* kr;
            if (i < nwin) {
                const int p = t - i;                      // window positions t, t-1, ...
                kr = wk + (int64_t)(p % eta) * DK;
            } else {
                kr = ck + (int64_t)(i - nwin) * DK;
            }
#pragma unroll
            for (int q = 0; q < PD; ++q) {
                const int dd = slot_dim(sub, q);
                acc = fmaf(xq[dd], IO<T>::ld(kr, dd), acc);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (i < nkeys && sub == 0) sc[i] = acc * scale;
    }
    // linear read partials
    {
        float pj = 0.f;
#pragma unroll
        for (int r = 0; r < HR; ++r) pj = fmaf(phq[hrg + NRG * r], hreg[r], pj);
        red[hrg * DV + hj] = pj;
    }
    __syncthreads();
    if (warp == 0) {
        float m = -INFINITY;
        for (int i = lane; i < nkeys; i += kWarp) m = fmaxf(m, sc[i]);
        m = warp_max(m);
        float l = 0.f;
        for (int i = lane; i < nkeys; i += kWarp) {
            const float p = expf(sc[i] - m);
            sc[i] = p;
            l += p;
        }
        l = warp_sum(l);
        float dl = 0.f;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) dl = fmaf(phq[lane + 32 * i], s_sm[lane + 32 * i], dl);
        dl = warp_sum(dl);
        if (lane == 0) {
            const bool any = nkeys > 0;
            misc[1] = any ? expf(-m) : 1.f;
            misc[2] = any ? fmaf(misc[1], dl, l) : dl;
        }
    }
    __syncthreads();
    // y_j = (sum_i p_i v_i[j] + e^{-m} (H^T phi_q)_j) / den ; keys split over NRG groups
    {
        float acc = 0.f;
        for (int i = hrg; i < nkeys; i += NRG) {
            const T* vr = i < nwin ? wvv + (int64_t)((t - i) % eta) * DV : cv + (int64_t)(i - nwin) * DV;
            acc = fmaf(sc[i], IO<T>::ld(vr, hj), acc);
        }
        __syncthreads();
        float lin = 0.f;
        if (hrg == 0) {
#pragma unroll
            for (int r = 0; r < NRG; ++r) lin += red[r * DV + hj];
        }
        __syncthreads();
        red[hrg * DV + hj] = acc;
        if (hrg == 0) Ne[hj] = lin;
        __syncthreads();
        if (tid < DV) {
            float num = 0.f;
#pragma unroll
            for (int r = 0; r < NRG; ++r) num += red[r * DV + tid];
            num = fmaf(misc[1], Ne[tid], num);
            IO<T>::st(static_cast<T*>(a.y), (int64_t)bh * DV + tid, num / misc[2]);
        }
    }

    // ---- 7. write back H, s, header ----
#pragma unroll
    for (int r = 0; r < HR; ++r) Hg[(hrg + NRG * r) * DV + hj] = hreg[r];
    if (tid < D) sg[tid] = s_sm[tid];
    if (tid == 0) {
        hdr[HDR_T] = t + 1;
        hdr[HDR_NCACHE] = nc_after;
        if (write) hdr[HDR_NWRITTEN] += 1;
        if (a.written_pos) a.written_pos[bh] = write ? wposn : -1;
    }
}

template <int D, int DV, typename T>
cudaError_t launch_decode_t(const Dims& d, const DecArgs& a, cudaStream_t st) {
    constexpr int DK = D;
    const int NRG = kDecThreads / DV;
    const size_t smem = sizeof(float) * ((D / 2) * (DK + 1) + 3 * DK + 2 * DV + 3 * D + DV + D + NRG * DV + DV +
                                         d.lam + d.eta + d.lam + 16);
    auto kern = decode_kernel<D, DV, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<d.BH, kDecThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Dims& d, char* state, const Layout& L, const float* W, int64_t w_head_stride,
                          const void* q, const void* k, const void* v, void* y, int32_t* written_pos,
                          cudaStream_t st) {
    DecArgs a;
    a.state = state;
    a.L = L;
    a.eta = d.eta;
    a.lam = d.lam;
    a.Hh = d.Hh;
    a.W = W;
    a.w_head_stride = w_head_stride;
    a.q = q;
    a.k = k;
    a.v = v;
    a.y = y;
    a.written_pos = written_pos;
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_decode_t<128, 128, __nv_bfloat16>(d, a, st) : launch_decode_t<128, 128, float>(d, a, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_decode_t<64, 64, __nv_bfloat16>(d, a, st) : launch_decode_t<64, 64, float>(d, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
