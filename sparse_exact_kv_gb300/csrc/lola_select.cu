// K2: the allocation chain of LoLA prefill -- window eviction, SRE scoring of the
// candidates, the top-lambda keep / write-the-rest decision and the (H, s) write.
//
// LoLA reading notes (arXiv 2505.23666v3): section 2.3, Eq. 10 (SRE), section 2.4,
// Eqs. 11-13 (candidates = cache ∪ evictee, scored against the memory before the write,
// the lambda largest stay, the rest are written once), section 2.2, Eqs. 3-5 (H, s).
// Per token at most one candidate is written, so "keep the top lambda of lambda + 1"
// is "write the argmin" (smaller SRE^2, then the older position).
//
// The chain is sequential in t, so one CTA -- or a thread-block cluster of CL CTAs when
// lambda > 64 -- owns one head for the whole sequence:
//   * cache slots live in registers: 8 lanes per slot, 4 slots per warp, 64 per CTA;
//     each lane holds D/8 entries of phi(k) and d_v/8 entries of v and N = H^T phi(k);
//     every slot keeps z = s^T phi(k) current, so a write w only costs each slot
//     g = phi_w . phi_i, N += g v_w, z += g (exact: H changes by a rank-1 term);
//   * each CTA holds a replica of H (D x d_v float32) in registers, 32 (or 8) entries
//     per thread, for the evictee's N_e = H^T phi(k_e) and for the chunk snapshots;
//   * per step: apply the previous write, score the live slots, warp argmin, then
//     warp 0 finishes the evictee's SRE and the CTA argmin; with CL > 1 each CTA pushes
//     its best to every peer's shared memory (st.shared::cluster) and one cluster
//     barrier orders the exchange; the winner's phi/v are read back through DSMEM.
// At every chunk start it stores H, s and the cache positions, from which the parallel
// output kernel rebuilds every query's exact set and linear state.
#include <climits>

#include "lola_internal.cuh"

namespace lola {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / kWarp;
constexpr int kSG = 8;                     // lanes per slot
constexpr int kSPW = kWarp / kSG;          // slots per warp
constexpr int kSPC = kSelWarps * kSPW;     // slots per CTA
constexpr int kMaxCluster = 16;

struct SelArgs {
    int n, eta, lam, chunk, nck, CL, io_bf16;
    const float* phiK;   // [BH][n][D]
    const void* K;       // io [BH][n][D]
    const void* V;       // io [BH][n][DV]
    int32_t* wpos;       // [BH][n]
    int32_t* wstep;      // [BH][n]
    float* snapH;        // [BH][nck][D*DV]
    float* snapS;        // [BH][nck][D]
    int32_t* snapC;      // [BH][nck][lam]
    int32_t* slotpos;    // [BH][lam]
    char* state;
    Layout L;
};

struct Dec {
    int write;   // a candidate was written this step
    int is_ev;   // ... and it was the evictee
    int pos;     // written position
    int cta;     // owner CTA of the written slot
    int ws;      // warp * kSPW + slot of the written slot
    int ev;      // an evictee joined the candidates this step
    int fill;    // global slot the evictee fills when nothing was written
    int pad;
};

struct __align__(16) Best {
    float sre2;
    int pos;
    int ws;      // warp * kSPW + slot, or -1 for the evictee
    int pad;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, const Best& b) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(__float_as_int(b.sre2)),
                 "r"(b.pos), "r"(b.ws), "r"(b.pad)
                 : "memory");
}
__device__ __forceinline__ float4 ld_cluster(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// entry i (0..PD-1) of lane `sub` of a slot: float4 chunks interleaved across the 8 lanes
__device__ __forceinline__ int slot_dim(int sub, int i) { return 4 * sub + 32 * (i >> 2) + (i & 3); }

template <typename T>
__device__ __forceinline__ float ldio(const void* p, int64_t i) {
    return IO<T>::ld(static_cast<const T*>(p), i);
}

template <int D, int DV, bool CLUSTER, typename T>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(const SelArgs a) {
    constexpr int PD = D / kSG, PV = DV / kSG;     // per-lane phi / v entries of a slot
    constexpr int NRG = kSelThreads / DV;          // H row groups
    constexpr int HR = D / NRG;                    // H rows per thread
    constexpr int EW = D + DV;                     // phi and v of one candidate
    static_assert(PD % 4 == 0 && PV % 4 == 0 && kSelThreads % DV == 0 && D % NRG == 0, "shape");

    extern __shared__ __align__(16) float dyn_sm[];
    float (*xbuf)[kSelWarps][EW] = reinterpret_cast<float (*)[kSelWarps][EW]>(dyn_sm);  // [2] warp-best phi/v
    constexpr int PF = 4;                                   // evictee prefetch distance (steps)
    constexpr int NEB = 8;                                  // ring of evictee buffers, by step & 7
    constexpr int VCH = DV * (int)sizeof(T) / 16;           // 16-byte chunks of one value row
    __shared__ __align__(16) float ebuf[NEB][EW];           // evictee phi and v (float32)
    __shared__ __align__(16) T evraw[NEB][DV];              // value row as stored (cp.async target)
    __shared__ __align__(16) float wbuf[EW];                // winner phi/v copied from a peer
    __shared__ __align__(16) float red[NRG][DV];            // N_e partial sums
    __shared__ __align__(16) float s_sm[D];
    __shared__ __align__(16) float nbuf[2][DV];             // evictee N_e
    __shared__ float zbuf[2], vvbuf[2];
    __shared__ Best wb[kSelWarps];
    __shared__ Best exch[2][kMaxCluster];
    __shared__ Dec dec[2];

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int rank = CLUSTER ? (int)cluster_rank() : 0;
    const int CL = CLUSTER ? a.CL : 1;
    const int bh = blockIdx.x / CL;
    const int n = a.n, eta = a.eta, lam = a.lam;

    // slot role
    const int sl = lane / kSG, sub = lane % kSG;
    const int ls = warp * kSPW + sl;          // local slot
    const int gslot = ls * CL + rank;         // global slot (fill order)
    float sphi[PD], sv[PV], sN[PV], sz = 0.f, svv = 0.f;
    int spos = -1;
#pragma unroll
    for (int i = 0; i < PD; ++i) sphi[i] = 0.f;
#pragma unroll
    for (int i = 0; i < PV; ++i) { sv[i] = 0.f; sN[i] = 0.f; }

    // H role
    const int hj = tid % DV, hrg = tid / DV;
    float h[HR];
#pragma unroll
    for (int r = 0; r < HR; ++r) h[r] = 0.f;
    if (tid < D) s_sm[tid] = 0.f;

    const float* phiK = a.phiK + (int64_t)bh * n * D;
    const int64_t vrow0 = (int64_t)bh * n;
    int32_t* wpos = a.wpos + (int64_t)bh * n;
    int32_t* wstep = a.wstep + (int64_t)bh * n;

    if (rank == 0)
        for (int i = tid; i < n; i += kSelThreads) wstep[i] = -1;

    // Evictee rows arrive by cp.async PF steps ahead: threads [0, D/4) copy phi(k_e),
    // threads [D/4, D/4 + VCH) copy v_e; each step commits one group (possibly empty).
    auto prefetch = [&](int step) {
        const int e = step - eta;
        if (step < n && e >= 0) {
            if (tid < D / 4) cp_async16(&ebuf[step & (NEB - 1)][4 * tid], phiK + (int64_t)e * D + 4 * tid);
            else if (tid < D / 4 + VCH)
                cp_async16(reinterpret_cast<char*>(evraw[step & (NEB - 1)]) + 16 * (tid - D / 4),
                           reinterpret_cast<const char*>(static_cast<const T*>(a.V) + (vrow0 + e) * DV) +
                               16 * (tid - D / 4));
        }
        cp_async_commit();
    };
    // After this thread's copies for `step` have landed: widen its value chunk to float32.
    auto finish = [&](int step) {
        if (step < n && step - eta >= 0 && tid >= D / 4 && tid < D / 4 + VCH) {
            constexpr int PER = 16 / (int)sizeof(T);
            const int c = tid - D / 4;
            const T* src = &evraw[step & (NEB - 1)][c * PER];
            float* dst = &ebuf[step & (NEB - 1)][D + c * PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) dst[i] = IO<T>::ld(src, i);
        }
    };
    for (int st = 0; st < PF; ++st) prefetch(st);
    cp_async_wait<0>();
    finish(0);
    int n_cached = 0, n_written = 0;
    __syncthreads();

    // Applies the decision taken at step tp: the surviving evictee moves into its slot,
    // then every live slot, H and s absorb the write.
    auto apply = [&](int tp) {
        const Dec dc = dec[tp & 1];
        const float* wsrc = nullptr;
        if (dc.write) {
            if (dc.is_ev) {
                wsrc = ebuf[tp & (NEB - 1)];
            } else if (!CLUSTER || dc.cta == rank) {
                wsrc = xbuf[tp & 1][dc.ws / kSPW];
            } else {
                if (tid < EW / 4) {
                    const uint32_t src = map_rank(smem_addr(&xbuf[tp & 1][dc.ws / kSPW][4 * tid]), dc.cta);
                    reinterpret_cast<float4*>(wbuf)[tid] = ld_cluster(src);
                }
                __syncthreads();
                wsrc = wbuf;
            }
        }
        if (dc.ev && !(dc.write && dc.is_ev)) {
            const int tcta = dc.write ? dc.cta : dc.fill % CL;
            const int tls = dc.write ? dc.ws : dc.fill / CL;
            const bool mine = tcta == rank && tls == ls;
            const float* eb = ebuf[tp & (NEB - 1)];
            // ||v||^2 of the evictee with the slot's lane partition (the decode kernel's order)
            float vv = 0.f;
#pragma unroll
            for (int i = 0; i < PV; ++i) {
                const float x = eb[D + slot_dim(sub, i)];
                vv = fmaf(x, x, vv);
            }
            vv += __shfl_xor_sync(0xffffffffu, vv, 1);
            vv += __shfl_xor_sync(0xffffffffu, vv, 2);
            vv += __shfl_xor_sync(0xffffffffu, vv, 4);
            if (mine) {
#pragma unroll
                for (int i = 0; i < PD; ++i) sphi[i] = eb[slot_dim(sub, i)];
#pragma unroll
                for (int i = 0; i < PV; ++i) {
                    sv[i] = eb[D + slot_dim(sub, i)];
                    sN[i] = nbuf[tp & 1][slot_dim(sub, i)];
                }
                sz = zbuf[tp & 1];
                svv = vv;
                spos = tp - eta;
            }
        }
        if (dc.write) {
            float g = 0.f;
#pragma unroll
            for (int i = 0; i < PD; ++i) g = fmaf(wsrc[slot_dim(sub, i)], sphi[i], g);
            g += __shfl_xor_sync(0xffffffffu, g, 1);
            g += __shfl_xor_sync(0xffffffffu, g, 2);
            g += __shfl_xor_sync(0xffffffffu, g, 4);
            if (spos >= 0) {
#pragma unroll
                for (int i = 0; i < PV; ++i) sN[i] = fmaf(g, wsrc[D + slot_dim(sub, i)], sN[i]);
                sz += g;
            }
            const float wvj = wsrc[D + hj];
#pragma unroll
            for (int r = 0; r < HR; ++r) h[r] = fmaf(wsrc[hrg + NRG * r], wvj, h[r]);
            if (tid < D) s_sm[tid] += wsrc[tid];
        }
    };

    for (int t = 0; t < n; ++t) {
        if (t > 0) apply(t - 1);

        // chunk-start snapshot of the memory before step t
        if (t % a.chunk == 0) {
            const int c = t / a.chunk;
            if (rank == 0) {
                float* sh = a.snapH + ((int64_t)bh * a.nck + c) * D * DV;
#pragma unroll
                for (int r = 0; r < HR; ++r) sh[(hrg + NRG * r) * DV + hj] = h[r];
                if (tid < D) a.snapS[((int64_t)bh * a.nck + c) * D + tid] = s_sm[tid];
            }
            if (sub == 0 && gslot < lam) a.snapC[((int64_t)bh * a.nck + c) * lam + gslot] = spos;
        }

        // ---- score: evictee partial N_e, slot SREs, warp argmin ----
        const bool ev = t >= eta;
        const float* eb = ebuf[t & (NEB - 1)];
        if (ev) {
            float pj = 0.f;
#pragma unroll
            for (int r = 0; r < HR; ++r) pj = fmaf(eb[hrg + NRG * r], h[r], pj);
            red[hrg][hj] = pj;
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PV; ++i) {
            const float dlt = fmaf(-sz, sv[i], sN[i]);
            ss = fmaf(dlt, dlt, ss);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        float bs = spos < 0 ? INFINITY : (sz == 0.f ? svv : ss / (sz * sz));
        int bp = spos < 0 ? INT_MAX : spos;
        int bsl = sl;
#pragma unroll
        for (int o = kSG; o < kWarp; o <<= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int op = __shfl_xor_sync(0xffffffffu, bp, o);
            const int osl = __shfl_xor_sync(0xffffffffu, bsl, o);
            if (key_less(os, op, bs, bp)) { bs = os; bp = op; bsl = osl; }
        }
        if (lane == 0) wb[warp] = Best{bs, bp, warp * kSPW + bsl, 0};
        if (sl == bsl && bp != INT_MAX) {
            float* xb = xbuf[t & 1][warp];
#pragma unroll
            for (int i = 0; i < PD; ++i) xb[slot_dim(sub, i)] = sphi[i];
#pragma unroll
            for (int i = 0; i < PV; ++i) xb[D + slot_dim(sub, i)] = sv[i];
        }
        prefetch(t + PF);
        __syncthreads();

        // ---- decide: evictee SRE, CTA argmin, cluster exchange ----
        const bool write = ev && (n_cached + 1 > lam);
        if (warp == 0) {
            float es = INFINITY;
            if (ev) {
                float Ne[DV / 32], ze = 0.f, sse = 0.f, vve = 0.f;
#pragma unroll
                for (int i = 0; i < DV / 32; ++i) {
                    float acc = 0.f;
#pragma unroll
                    for (int r = 0; r < NRG; ++r) acc += red[r][lane + 32 * i];
                    Ne[i] = acc;
                    nbuf[t & 1][lane + 32 * i] = acc;
                }
#pragma unroll
                for (int i = 0; i < D / 32; ++i) ze = fmaf(s_sm[lane + 32 * i], eb[lane + 32 * i], ze);
                ze = warp_sum(ze);
#pragma unroll
                for (int i = 0; i < DV / 32; ++i) {
                    const float v = eb[D + lane + 32 * i];
                    const float dlt = fmaf(-ze, v, Ne[i]);
                    sse = fmaf(dlt, dlt, sse);
                    vve = fmaf(v, v, vve);
                }
                sse = warp_sum(sse);
                vve = warp_sum(vve);
                es = ze == 0.f ? vve : sse / (ze * ze);
                if (lane == 0) { zbuf[t & 1] = ze; vvbuf[t & 1] = vve; }
            }
            Best b = lane < kSelWarps ? wb[lane] : Best{INFINITY, INT_MAX, -2, 0};
            if (ev && lane == kSelWarps) b = Best{es, t - eta, -1, 0};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                Best c;
                c.sre2 = __shfl_xor_sync(0xffffffffu, b.sre2, o);
                c.pos = __shfl_xor_sync(0xffffffffu, b.pos, o);
                c.ws = __shfl_xor_sync(0xffffffffu, b.ws, o);
                if (key_less(c.sre2, c.pos, b.sre2, b.pos)) b = c;
            }
            if constexpr (CLUSTER) {
                if (lane < CL) st_cluster(map_rank(smem_addr(&exch[t & 1][rank]), lane), b);
            } else if (lane == 0) {
                exch[t & 1][0] = b;
            }
        }
        if constexpr (CLUSTER) cluster_barrier(); else __syncwarp();
        if (warp == 0) {
            Best b = exch[t & 1][0];
            int bc = 0;
            if constexpr (CLUSTER) {
                b = lane < CL ? exch[t & 1][lane] : Best{INFINITY, INT_MAX, -2, 0};
                bc = lane;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    Best c;
                    c.sre2 = __shfl_xor_sync(0xffffffffu, b.sre2, o);
                    c.pos = __shfl_xor_sync(0xffffffffu, b.pos, o);
                    c.ws = __shfl_xor_sync(0xffffffffu, b.ws, o);
                    const int cc = __shfl_xor_sync(0xffffffffu, bc, o);
                    if (key_less(c.sre2, c.pos, b.sre2, b.pos) || (c.sre2 == b.sre2 && c.pos == b.pos && cc < bc)) {
                        b = c;
                        bc = cc;
                    }
                }
            }
            if (lane == 0) {
                Dec d;
                d.write = write;
                d.is_ev = write && b.ws < 0;
                d.pos = write ? b.pos : -1;
                d.cta = bc;
                d.ws = b.ws;
                d.ev = ev;
                d.fill = n_cached;
                d.pad = 0;
                dec[t & 1] = d;
                if (rank == 0) {
                    wpos[t] = d.pos;
                    if (write) wstep[b.pos] = t;
                }
            }
        }
        cp_async_wait<PF - 1>();   // this thread's copies for step t + 1 have landed
        finish(t + 1);
        __syncthreads();
        if (ev && !write) ++n_cached;
        if (write) ++n_written;
    }
    if (n > 0) apply(n - 1);

    // ---- export the memory after token n-1 into the state record ----
    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    const T* Kin = static_cast<const T*>(a.K);
    const T* Vin = static_cast<const T*>(a.V);
    if (rank == 0) {
        int32_t* hdr = reinterpret_cast<int32_t*>(rec);
        if (tid == 0) {
            hdr[HDR_T] = n;
            hdr[HDR_NCACHE] = n_cached;
            hdr[HDR_NWRITTEN] = n_written;
            hdr[HDR_STATUS] = 0;
        }
        float* Hs = reinterpret_cast<float*>(rec + a.L.H);
#pragma unroll
        for (int r = 0; r < HR; ++r) Hs[(hrg + NRG * r) * DV + hj] = h[r];
        if (tid < D) reinterpret_cast<float*>(rec + a.L.s)[tid] = s_sm[tid];
        // window ring: entry e holds the newest position p <= n-1 with p % eta == e
        int32_t* wp = reinterpret_cast<int32_t*>(rec + a.L.win_pos);
        T* wk = reinterpret_cast<T*>(rec + a.L.win_k);
        T* wv = reinterpret_cast<T*>(rec + a.L.win_v);
        for (int i = tid; i < eta * (1 + D + DV); i += kSelThreads) {
            const int e = i % eta, part = i / eta;
            const int p = (n - 1) - ((((n - 1) - e) % eta) + eta) % eta;
            if (part == 0) wp[e] = p >= 0 ? p : -1;
            else if (p >= 0 && part <= D) wk[(int64_t)e * D + (part - 1)] = Kin[(vrow0 + p) * D + (part - 1)];
            else if (p >= 0) wv[(int64_t)e * DV + (part - 1 - D)] = Vin[(vrow0 + p) * DV + (part - 1 - D)];
        }
    }
    // cache: live slots first, sorted by position
    int32_t* sp = a.slotpos + (int64_t)bh * lam;
    if (sub == 0 && gslot < lam) sp[gslot] = spos;
    __threadfence();
    if constexpr (CLUSTER) cluster_barrier(); else __syncthreads();
    int cnt = 0;
    if (spos >= 0)
        for (int g = sub; g < lam; g += kSG) {
            const int p = sp[g];
            cnt += (p >= 0 && p < spos) ? 1 : 0;
        }
    cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, 4);
    if (spos >= 0 && gslot < lam) {
        const int r = cnt;
        float* cphi = reinterpret_cast<float*>(rec + a.L.c_phi) + (int64_t)r * D;
        float* cN = reinterpret_cast<float*>(rec + a.L.c_N) + (int64_t)r * DV;
        T* ck = reinterpret_cast<T*>(rec + a.L.c_k) + (int64_t)r * D;
        T* cv = reinterpret_cast<T*>(rec + a.L.c_v) + (int64_t)r * DV;
#pragma unroll
        for (int i = 0; i < PD; ++i) cphi[slot_dim(sub, i)] = sphi[i];
#pragma unroll
        for (int i = 0; i < PV; ++i) cN[slot_dim(sub, i)] = sN[i];
        for (int c = sub; c < D; c += kSG) ck[c] = Kin[(vrow0 + spos) * D + c];
        for (int c = sub; c < DV; c += kSG) cv[c] = Vin[(vrow0 + spos) * DV + c];
        if (sub == 0) {
            reinterpret_cast<int32_t*>(rec + a.L.c_pos)[r] = spos;
            reinterpret_cast<float*>(rec + a.L.c_z)[r] = sz;
        }
    }
    if (rank == 0)
        for (int r = n_cached + tid; r < lam; r += kSelThreads) reinterpret_cast<int32_t*>(rec + a.L.c_pos)[r] = -1;
}

template <int D, int DV>
constexpr size_t select_dyn_smem() { return sizeof(float) * 2 * kSelWarps * (D + DV); }

template <int D, int DV, typename T>
cudaError_t launch_select_single(const Dims& d, const SelArgs& a, cudaStream_t st) {
    auto kern = select_kernel<D, DV, false, T>;
    const size_t smem = select_dyn_smem<D, DV>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<d.BH, kSelThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int D, int DV, typename T>
cudaError_t launch_select_cluster(const Dims& d, const SelArgs& a, cudaStream_t st) {
    auto kern = select_kernel<D, DV, true, T>;
    const size_t smem = select_dyn_smem<D, DV>();
    {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (a.CL > 8) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.BH * a.CL);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&nclusters, (void*)kern, &cfg);
    if (e != cudaSuccess) return e;
    if (nclusters < 1) return cudaErrorInvalidConfiguration;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

// Number of CTAs per head: enough register slots for lambda cache entries (64 per CTA).
int select_cluster_size(int lam) {
    int need = (lam + kSPC - 1) / kSPC;
    int cl = 1;
    while (cl < need) cl <<= 1;
    return cl;
}

cudaError_t launch_select(const Dims& d, int n, const Workspace& ws, const void* K, const void* V, char* state,
                          const Layout& L, cudaStream_t st) {
    SelArgs a;
    a.n = n;
    a.eta = d.eta;
    a.lam = d.lam;
    a.chunk = d.chunk;
    a.nck = ws.nck;
    a.CL = select_cluster_size(d.lam);
    a.io_bf16 = d.dtype == LOLA_BF16;
    a.phiK = ws.phiK;
    a.K = K;
    a.V = V;
    a.wpos = ws.wpos;
    a.wstep = ws.wstep;
    a.snapH = ws.snapH;
    a.snapS = ws.snapS;
    a.snapC = ws.snapC;
    a.slotpos = ws.slotpos;
    a.state = state;
    a.L = L;
    if (a.CL > kMaxCluster) return cudaErrorInvalidValue;
    const bool bf = a.io_bf16;
    if (a.CL == 1) {
        if (d.D == 128 && d.dv == 128)
            return bf ? launch_select_single<128, 128, __nv_bfloat16>(d, a, st)
                      : launch_select_single<128, 128, float>(d, a, st);
        if (d.D == 64 && d.dv == 64)
            return bf ? launch_select_single<64, 64, __nv_bfloat16>(d, a, st)
                      : launch_select_single<64, 64, float>(d, a, st);
        return cudaErrorInvalidValue;
    }
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_select_cluster<128, 128, __nv_bfloat16>(d, a, st)
                  : launch_select_cluster<128, 128, float>(d, a, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_select_cluster<64, 64, __nv_bfloat16>(d, a, st)
                  : launch_select_cluster<64, 64, float>(d, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
