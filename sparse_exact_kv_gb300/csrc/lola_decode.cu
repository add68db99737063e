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
// One CTA of 512 threads per head, with the layouts and the arithmetic of the prefill
// chain (lola_chain.cuh): the evictee's N arrives from the state (computed one step
// ahead, against the memory before the previous write, then corrected by that write),
// and at the end of the step the next evictee's N is prepared the same way.  A decode
// step therefore continues a prefill bit for bit whenever eta > 0.  (With eta = 0 the
// evictee is the token itself, unknown one step ahead; its N is then taken directly
// against the current memory, equal in exact arithmetic.)
#include <climits>

#include "lola_chain.cuh"
#include "lola_phi_tc.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace chain;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kDecWarps = kThreads / kWarp;
constexpr int kSlotsPerPass = kThreads / kSG;   // 64

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
    int BH;
    int prefetch_ahead;   // heads ahead of this one whose state is prefetched into L2 (0: none)
    int read_mask;        // lola_read_flags: memories left out of the read (the update is unchanged)
    int tok_phi_ready;    // decode_kernel: phi(q), phi(k) of the token are in tok_phi already
};

// Ask L2 to fetch [p, p + bytes) with bulk prefetches of at most 16 KB each, issued by
// lane 0 of successive warps from warp first_warp on (p 16-byte aligned, bytes a multiple of
// 16): the CTA that processes that head about one wave later then finds its state in L2
// instead of DRAM.
constexpr int kPrefetchChunk = 16384;
__device__ __forceinline__ void prefetch_l2(const char* p, int64_t bytes, int tid, int nthreads, int first_warp = 0) {
    if (tid % kWarp != 0) return;
    const int nw = nthreads / kWarp;
    const int rank = (tid / kWarp - first_warp + nw) % nw;
    for (int64_t o = (int64_t)rank * kPrefetchChunk; o < bytes; o += (int64_t)nw * kPrefetchChunk) {
        const int64_t left = bytes - o;
        const uint32_t n = (uint32_t)(left < kPrefetchChunk ? left : kPrefetchChunk);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + o), "r"(n) : "memory");
    }
}

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecArgs a) {
    using S = Shape<D, DV>;
    constexpr int DK = D;
    constexpr int PD = S::PD, PV = S::PV, NRG = S::NRG, HR = S::HR, HC = S::HC;
    constexpr int KS = kThreads / DV;        // key splits of the output numerator
    constexpr int kEvWarp = kDecWarps - 1;   // holds s and finishes the evictee (slot layout)
    extern __shared__ __align__(16) float sm[];
    float* Ws = sm;                              // [D/2][DK+1]
    float* xq = Ws + (D / 2) * w_stride<DK>();   // [DK]  query
    float* xk = xq + DK;                         // [DK]  new key
    float* xv = xk + DK;                         // [DV]  new value
    float* ek = xv + DV;                         // [DK]  evictee key
    float* evv = ek + DK;                        // [DV]  evictee value
    float* nk = evv + DV;                        // [D]   phi(k_t) of the new token
    float* phq = nk + DK;                        // [D]
    float* phe = phq + D;                        // [D]   phi of the evictee
    float* phn = phe + D;                        // [D]   phi of the next evictee
    float* wphi = phn + D;                       // [D]   written phi
    float* wv = wphi + D;                        // [DV]  written v
    float* red = wv + DV;                        // [NRG][DV]
    float* Ne_s = red + NRG * DV;                // [DV]  evictee N (for the move into a slot)
    float* lin = Ne_s + DV;                      // [DV]  H^T phi(q)
    float* sc = lin + DV;                        // [eta + lam] scores, then weights
    uint2* wkey = reinterpret_cast<uint2*>(sc + a.eta + a.lam + (((a.eta + a.lam) & 1) ? 1 : 0));  // [16+1]
    float* misc = reinterpret_cast<float*>(wkey + kDecWarps + 2);
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
    float* evs = reinterpret_cast<float*>(rec + a.L.ev);
    float* wphg = reinterpret_cast<float*>(rec + a.L.win_phi);
    const T* qin = static_cast<const T*>(a.q) + (int64_t)bh * DK;
    const T* kin = static_cast<const T*>(a.k) + (int64_t)bh * DK;
    const T* vin = static_cast<const T*>(a.v) + (int64_t)bh * DV;

    const bool ev = t >= eta;
    const int e = t - eta;
    const int ring = eta > 0 ? t % eta : 0;
    const bool nxt = eta > 0 && t + 1 - eta >= 0;   // the next step has an evictee known now
    const int nring = eta > 0 ? (t + 1) % eta : 0;

    // ---- 1. loads: W, tokens, H (H role), s (evictee warp) ----
    const float* Wh = a.W + (int64_t)h * a.w_head_stride;
    if (!a.tok_phi_ready) stage_w<DK, D, kThreads>(Ws, Wh, tid);
    if (tid < DK) {
        xq[tid] = IO<T>::ld(qin, tid);
        xk[tid] = IO<T>::ld(kin, tid);
        if (ev) ek[tid] = eta > 0 ? IO<T>::ld(wk, (int64_t)ring * DK + tid) : IO<T>::ld(kin, tid);
    }
    if (tid < D && eta > 0) {
        if (ev) phe[tid] = wphg[(int64_t)ring * D + tid];
        if (nxt) phn[tid] = wphg[(int64_t)nring * D + tid];
    }
    if (tid < DV) {
        xv[tid] = IO<T>::ld(vin, tid);
        if (ev) evv[tid] = eta > 0 ? IO<T>::ld(wvv, (int64_t)ring * DV + tid) : IO<T>::ld(vin, tid);
    }
    float hreg[HR * HC];
    h_load<D, DV>(hreg, Hg, warp, lane);
    const int sl = tid / kSG, sub = tid % kSG;
    float s_reg[PD];                                      // s, held by the evictee warp
#pragma unroll
    for (int i = 0; i < PD; ++i) s_reg[i] = 0.f;
    if (warp == kEvWarp) slot_load<D>(sg, sub, s_reg);
    __syncthreads();
    if (ev && eta > 0 && tid == 0 && winpos[ring] != e) atomicOr(&hdr[HDR_STATUS], (int)ST_BAD_STATE);

    // ---- 2. phi(q), phi(k_e), phi(k_{e+1}) ----
    if (a.tok_phi_ready) {
        // mapped by the token feature-map kernel that ran before this one
        const float* tphi = reinterpret_cast<const float*>(rec + a.L.tok_phi);
        if (tid < D) {
            phq[tid] = tphi[tid];
            nk[tid] = tphi[D + tid];
            if (eta == 0) phe[tid] = tphi[D + tid];
        }
    } else if (warp == 0) {
        float ph[D / 32];
        phi_warp<DK, D>(xq, Ws, lane, ph);
#pragma unroll
        for (int m = 0; m < D / 32; ++m) phq[lane + 32 * m] = ph[m];
    } else if (warp == 1) {
        // phi(k_t): stored in the window ring; with eta = 0 it is also the evictee's phi
        float ph[D / 32];
        phi_warp<DK, D>(xk, Ws, lane, ph);
#pragma unroll
        for (int m = 0; m < D / 32; ++m) {
            nk[lane + 32 * m] = ph[m];
            if (eta == 0) phe[lane + 32 * m] = ph[m];
        }
    }
    __syncthreads();

    // ---- 3. partials against the memory before this step's write: the next evictee's
    //         (or, with eta = 0, this step's own evictee) H^T phi ----
    const float* pvec = eta > 0 ? phn : phe;
    const bool want_partials = eta > 0 ? nxt : ev;
    if (want_partials) h_partial_store<D, DV>(red, pvec, hreg, warp, lane);
    __syncthreads();

    // ---- 4. the evictee's N, z and SRE; the next evictee's N', z' (evictee warp) ----
    float Nn[PV], zn = 0.f;
#pragma unroll
    for (int i = 0; i < PV; ++i) Nn[i] = 0.f;
    if (warp == kEvWarp) {
        uint32_t ehi = kNoKey, elo = kNoKey;
        if (ev) {
            // the evictee's SRE in the warp layout (DV/32 consecutive entries per lane), the
            // arithmetic of the prefill chain's evictee warp
            constexpr int EV = DV / kWarp;
            float ze;
            if (eta > 0) {
                if (tid - kEvWarp * kWarp < DV / 4)
                    reinterpret_cast<float4*>(Ne_s)[tid - kEvWarp * kWarp] = reinterpret_cast<const float4*>(evs)[tid - kEvWarp * kWarp];
                ze = evs[DV];
            } else {
                float Ne[PV];
                slot_reduce_partials<D, DV>(red, sub, Ne);
                if (lane < kSG) slot_store<DV>(Ne_s, sub, Ne);
                ze = slot_gram<D>(phe, s_reg, sub);
            }
            __syncwarp();
            float ve[PV], Nw[EV], vw[EV];
            slot_load<DV>(evv, sub, ve);
            h_vec_load<EV>(Ne_s + lane * EV, Nw);
            h_vec_load<EV>(evv + lane * EV, vw);
            const float es = warp_sre2<DV>(Nw, ze, vw, slot_vv<DV>(ve));
            if (lane == 0) misc[0] = ze;
            ehi = key_hi(es);
            elo = key_lo(e, kEvCode);
        }
        if (lane == 0) wkey[kDecWarps] = make_uint2(ehi, elo);
        if (nxt) {
            slot_reduce_partials<D, DV>(red, sub, Nn);
            zn = warp_dot<D>(phn, sg, lane);   // s before this step's write
        }
    }
    // slot SREs, pass by pass; each warp keeps its minimum over all passes
    uint32_t bhi = kNoKey, blo = kNoKey;
    for (int base = 0; base < nc; base += kSlotsPerPass) {
        const int i = base + sl;
        float sN[PV], sv[PV], z = 0.f;
#pragma unroll
        for (int q = 0; q < PV; ++q) { sN[q] = 0.f; sv[q] = 0.f; }
        if (i < nc) {
            z = cz[i];
#pragma unroll
            for (int q = 0; q < PV; ++q) {
                const int dd = slot_dim(sub, q);
                sv[q] = IO<T>::ld(cv, (int64_t)i * DV + dd);
                sN[q] = cN[(int64_t)i * DV + dd];
            }
        }
        const float svv = slot_vv<DV>(sv);
        const float sre = slot_sre2<DV>(sN, z, sv, svv);
        uint32_t khi = i < nc ? key_hi(sre) : kNoKey;
        uint32_t klo = i < nc ? key_lo(cpos[i], 0) : kNoKey;
        warp_min_key(khi, klo);
        if (khi < bhi || (khi == bhi && klo < blo)) { bhi = khi; blo = klo; }
    }
    if (lane == 0) wkey[warp] = make_uint2(bhi, blo);
    __syncthreads();

    // ---- 5. decision ----
    const bool write = ev && (nc + 1 > lam);
    if (warp == 0) {
        uint2 k = lane <= kDecWarps ? wkey[lane] : make_uint2(kNoKey, kNoKey);
        warp_min_key(k.x, k.y);
        if (lane == 0) {
            int wsel = -2, wpos = -1;
            if (write) {
                wpos = (int)(k.y >> 7);
                wsel = ((k.y & 127u) == (uint32_t)kEvCode) ? -1 : -3;   // -3: a slot, found below
            }
            imisc[0] = wsel;
            imisc[1] = wpos;
        }
    }
    __syncthreads();
    int wsel = imisc[0];
    const int wposn = imisc[1];
    if (wsel == -3) {
        // the written slot: the one holding position wposn
        for (int i = tid; i < nc; i += kThreads)
            if (cpos[i] == wposn) imisc[2] = i;
        __syncthreads();
        wsel = imisc[2];
    }
    const float ze = misc[0];

    // ---- 6. write: phi_w, v_w; H, s, slots; the surviving evictee; next evictee ----
    if (write) {
        if (tid < D) wphi[tid] = wsel < 0 ? phe[tid] : cphi[(int64_t)wsel * D + tid];
        if (tid < DV) wv[tid] = wsel < 0 ? evv[tid] : IO<T>::ld(cv, (int64_t)wsel * DV + tid);
        __syncthreads();
        float vh[HC];
        h_vec_load<HC>(wv + lane * HC, vh);
        h_update<D, DV>(hreg, wphi, vh, warp);
        if (warp == kEvWarp) {
            float wp[PD];
            slot_load<D>(wphi, sub, wp);
#pragma unroll
            for (int i = 0; i < PD; ++i) s_reg[i] += wp[i];
        }
        for (int base = 0; base < nc; base += kSlotsPerPass) {
            const int i = base + sl;
            float sphi[PD], sN[PV];
            const bool live = i < nc;
            // the written slot takes the evictee, which absorbs the write like the others
            const bool moved = live && i == wsel;
#pragma unroll
            for (int q = 0; q < PD; ++q) {
                const int dd = slot_dim(sub, q);
                sphi[q] = live ? (moved ? phe[dd] : cphi[(int64_t)i * D + dd]) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < PV; ++q) {
                const int dd = slot_dim(sub, q);
                sN[q] = live ? (moved ? Ne_s[dd] : cN[(int64_t)i * DV + dd]) : 0.f;
            }
            const float g = slot_gram<D>(wphi, sphi, sub);
            if (live) {
                slot_axpy<DV>(sN, g, wv, sub);
#pragma unroll
                for (int q = 0; q < PV; ++q) cN[(int64_t)i * DV + slot_dim(sub, q)] = sN[q];
                if (sub == 0) cz[i] = (moved ? ze : cz[i]) + g;
            }
        }
        if (warp == kEvWarp && nxt) {
            const float g = warp_dot<D>(wphi, phn, lane);
            slot_axpy<DV>(Nn, g, wv, sub);
            zn += g;
        }
    }
    int nc_after = nc;
    int slot_new = -1;
    if (ev && !write) {
        slot_new = nc;
        nc_after = nc + 1;
        if (tid < DV) cN[(int64_t)slot_new * DV + tid] = Ne_s[tid];
        if (tid == 0) cz[slot_new] = ze;
    }
    if (write && wsel >= 0) slot_new = wsel;
    if (slot_new >= 0) {
        if (tid < D) cphi[(int64_t)slot_new * D + tid] = phe[tid];
        if (tid < DK) IO<T>::st(ck, (int64_t)slot_new * DK + tid, ek[tid]);
        if (tid < DV) IO<T>::st(cv, (int64_t)slot_new * DV + tid, evv[tid]);
        if (tid == 0) cpos[slot_new] = e;
    }
    if (warp == kEvWarp && nxt) {
        if (lane < kSG) slot_store<DV>(evs, sub, Nn);
        if (lane == 0) evs[DV] = zn;
    }
    // the new token enters the window ring (its previous occupant was the evictee)
    if (eta > 0) {
        if (tid < DK) IO<T>::st(wk, (int64_t)ring * DK + tid, xk[tid]);
        if (tid < DV) IO<T>::st(wvv, (int64_t)ring * DV + tid, xv[tid]);
        if (tid < D) wphg[(int64_t)ring * D + tid] = nk[tid];
        if (tid == 0) winpos[ring] = t;
    }
    __syncthreads();

    // ---- 7. output: softmax over window ∪ cache, linear read of (H, s) after the write ----
    const float scale = 1.0f / sqrtf((float)DK);
    const int nwin = min(t + 1, eta);
    const int nkeys = (a.read_mask & LOLA_READ_HIDE_CACHE) ? nwin : nwin + nc_after;   // window first
    for (int base = 0; base < nkeys; base += kSlotsPerPass) {
        const int i = base + sl;
        float acc = 0.f;
        if (i < nkeys) {
            const T* kr = i < nwin ? wk + (int64_t)((t - i) % eta) * DK : ck + (int64_t)(i - nwin) * DK;
#pragma unroll
            for (int q = 0; q < PD; ++q) {
                const int dd = slot_dim(sub, q);
                acc = fmaf(xq[dd], IO<T>::ld(kr, dd), acc);
            }
        }
        acc += __shfl_xor_sync(kFull, acc, 1);
        acc += __shfl_xor_sync(kFull, acc, 2);
        acc += __shfl_xor_sync(kFull, acc, 4);
        if (i < nkeys && sub == 0) sc[i] = acc * scale;
    }
    h_partial_store<D, DV>(red, phq, hreg, warp, lane);
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
        if (lane == 0) {
            const bool any = nkeys > 0;
            misc[1] = any ? expf(-m) : 1.f;
            misc[3] = l;
        }
    } else if (warp == kEvWarp) {
        const float dl = slot_gram<D>(phq, s_reg, sub);
        if (lane == 0) misc[4] = dl;
    } else if (warp == 1 && tid - 32 < DV / 4) {
        // H^T phi(q): sum the row-group partials
        const int j0 = 4 * (tid - 32);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            float acc = red[j0 + jj];
#pragma unroll
            for (int rg = 1; rg < NRG; ++rg) acc += red[rg * DV + j0 + jj];
            lin[j0 + jj] = acc;
        }
    }
    __syncthreads();
    {
        // numerator: keys split KS ways (thread: split ks, column kj), then combined
        const int ks = tid / DV, kj = tid % DV;
        float acc = 0.f;
        for (int i = ks; i < nkeys; i += KS) {
            const T* vr = i < nwin ? wvv + (int64_t)((t - i) % eta) * DV : cv + (int64_t)(i - nwin) * DV;
            acc = fmaf(sc[i], IO<T>::ld(vr, kj), acc);
        }
        red[ks * DV + kj] = acc;
        __syncthreads();
        if (tid < DV) {
            float num = 0.f;
#pragma unroll
            for (int r = 0; r < KS; ++r) num += red[r * DV + tid];
            const float el = (a.read_mask & LOLA_READ_HIDE_STATE) ? 0.f : misc[1];   // the state's weight
            num = fmaf(el, lin[tid], num);
            const float den = nkeys > 0 ? fmaf(el, misc[4], misc[3]) : misc[4];
            IO<T>::st(static_cast<T*>(a.y), (int64_t)bh * DV + tid, num / den);
        }
    }

    // ---- 8. write back H, s, header ----
    h_store<D, DV>(Hg, hreg, warp, lane);
    if (warp == kEvWarp && lane < kSG) slot_store<D>(sg, sub, s_reg);
    if (tid == 0) {
        hdr[HDR_T] = t + 1;
        hdr[HDR_NCACHE] = nc_after;
        if (write) hdr[HDR_NWRITTEN] += 1;
        if (a.written_pos) a.written_pos[bh] = write ? wposn : -1;
    }
}

// ---------------------------------------------------------------------------------
// Fast path (1 <= eta <= kFastEta, lambda <= 64): every byte of a head's step is requested
// in one burst at the start -- H and the slots' N, z in registers, the slots' phi and the
// exact KV of cache and window (plus the two evictees' phi) in shared memory by cp.async --
// because none of it depends on the decision.  The decision, the write and the output then
// run on chip and everything is written back at the end.  Same chain arithmetic.
// ---------------------------------------------------------------------------------
constexpr int kFastLam = 64;
constexpr int kFastEta = 128;
constexpr size_t kMaxSmemPerCta = 227 * 1024;   // opt-in dynamic shared memory of one sm_103 CTA

// values 2 kc and 2 kc + 1 of a value row (float32 or bfloat16, widened exactly)
template <typename T>
__device__ __forceinline__ void h_cols2(const T* v, int kc, float* out) {
    if constexpr (sizeof(T) == 4) {
        const float2 f = reinterpret_cast<const float2*>(v)[kc];
        out[0] = f.x;
        out[1] = f.y;
    } else {
        const uint32_t x = reinterpret_cast<const uint32_t*>(v)[kc];
        out[0] = bf16_lo(x);
        out[1] = bf16_hi(x);
    }
}

template <int D, int DV, typename T>
struct FastSmem {
    static constexpr int DK = D;
    static constexpr int NRG = Shape<D, DV>::NRG;   // H row groups (partials)
    static constexpr size_t a16(size_t x) { return (x + 15) / 16 * 16; }
    // byte offsets (16-byte aligned)
    static constexpr size_t HST = 0;                                        // [D][DV] f32 H, for its bulk store
    static constexpr size_t CPHI = HST + 4 * D * DV;                       // [64][D] f32; then the N rows' bulk store
    static constexpr size_t CV = CPHI + 4 * kFastLam * D;                  // [64][DV] T
    static constexpr size_t CK = CV + sizeof(T) * kFastLam * DV;           // [64][DK] T
    static constexpr size_t RK = CK + sizeof(T) * kFastLam * DK;           // [kFastEta][DK] T
    static constexpr size_t RV = RK + sizeof(T) * kFastEta * DK;           // [kFastEta][DV] T
    static constexpr size_t NV = RV + sizeof(T) * kFastEta * DV;           // [DV] T the new token's v
    static constexpr size_t PHE = a16(NV + sizeof(T) * DV);                // [D] f32 evictee phi
    static constexpr size_t PHN = PHE + 4 * D;                             // [D] f32 next evictee phi
    static constexpr size_t EVN = PHN + 4 * D;                             // [DV + 4] f32 evictee N, z
    static constexpr size_t SS = EVN + 4 * (DV + 4);                       // [D] f32 s
    static constexpr size_t XQ = SS + 4 * D;                               // [DK] f32
    static constexpr size_t XK = XQ + 4 * DK;                              // [DK] f32
    static constexpr size_t PHQ = XK + 4 * DK;                             // [D] f32
    static constexpr size_t RED = PHQ + 4 * D;                             // [NRG][DV] f32
    static constexpr size_t RED2 = RED + 4 * NRG * DV;                     // [NRG][DV] f32
    static constexpr size_t NPART = RED2 + 4 * NRG * DV;                   // [DV] f32 next evictee's summed partials
    static constexpr size_t LIN = NPART + 4 * DV;                          // [DV] f32
    static constexpr size_t SC = LIN + 4 * DV;                             // [kFastEta + 64] f32
    static constexpr size_t PB = SC + 4 * (kFastEta + kFastLam);           // [kFastEta + 64] f32 weights
    static constexpr size_t LPART = PB + 4 * (kFastEta + kFastLam);        // [16] f32 per-warp weight sums
    static constexpr size_t VOFF = LPART + 4 * kDecWarps;                  // [kFastEta + 64] i32 value-row offsets
    static constexpr size_t WKEY = VOFF + 4 * (kFastEta + kFastLam);       // [17] uint2
    static constexpr size_t MISC = WKEY + 8 * 18;                          // [8] f32
    static_assert(DV <= D, "the N rows are staged in the slot phi rows");
    static constexpr size_t MBAR = a16(MISC + 4 * 8);                      // u64 burst barrier
    static constexpr size_t TOTAL = MBAR + 8;
};

// bulk copies (TMA engine) of the burst, completing on an mbarrier
constexpr uint64_t kBurstWaitNs = 1000000000ull;   // a burst that has not landed in 1 s is an error
__device__ __forceinline__ void mbar_expect(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// [src, src + bytes) -> shared dst; both 16-byte aligned, bytes a nonzero multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
// shared [src, src + bytes) -> global dst (same rules), in this thread's current bulk group
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"((uint32_t)__cvta_generic_to_shared(src)), "r"(bytes)
                 : "memory");
}
// programmatic dependent launch: wait for the preceding grid (a no-op without it) / let the
// next grid start launching
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's bulk stores have been read
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's shared-memory writes become visible to the bulk copies (async proxy)
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads, 1) decode_fast_kernel(const DecArgs a) {
    using S = Shape<D, DV>;
    using M = FastSmem<D, DV, T>;
    constexpr int DK = D;
    constexpr int PD = S::PD, PV = S::PV, HR = S::HR, HC = S::HC;
    constexpr int kEvWarp = kDecWarps - 1;
    extern __shared__ __align__(16) uint8_t smb[];
    float* hst = reinterpret_cast<float*>(smb + M::HST);
    float* cphi_s = reinterpret_cast<float*>(smb + M::CPHI);
    T* cv_s = reinterpret_cast<T*>(smb + M::CV);
    T* ck_s = reinterpret_cast<T*>(smb + M::CK);
    T* rk_s = reinterpret_cast<T*>(smb + M::RK);
    T* rv_s = reinterpret_cast<T*>(smb + M::RV);
    T* nv_s = reinterpret_cast<T*>(smb + M::NV);
    float* phe = reinterpret_cast<float*>(smb + M::PHE);
    float* phn = reinterpret_cast<float*>(smb + M::PHN);
    float* evn = reinterpret_cast<float*>(smb + M::EVN);
    float* s_sm = reinterpret_cast<float*>(smb + M::SS);
    float* xq = reinterpret_cast<float*>(smb + M::XQ);
    float* xk = reinterpret_cast<float*>(smb + M::XK);
    float* phq = reinterpret_cast<float*>(smb + M::PHQ);
    float* red = reinterpret_cast<float*>(smb + M::RED);
    float* red2 = reinterpret_cast<float*>(smb + M::RED2);
    float* npart = reinterpret_cast<float*>(smb + M::NPART);
    float* lin = reinterpret_cast<float*>(smb + M::LIN);
    float* sc = reinterpret_cast<float*>(smb + M::SC);
    float* pb = reinterpret_cast<float*>(smb + M::PB);
    float* lpart = reinterpret_cast<float*>(smb + M::LPART);
    int* voff = reinterpret_cast<int*>(smb + M::VOFF);
    uint2* wkey = reinterpret_cast<uint2*>(smb + M::WKEY);
    float* misc = reinterpret_cast<float*>(smb + M::MISC);

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x;
    const int eta = a.eta, lam = a.lam;
    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    int32_t* hdr = reinterpret_cast<int32_t*>(rec);
    const int t = hdr[HDR_T];
    const int nc = hdr[HDR_NCACHE];
    const int nwr = hdr[HDR_NWRITTEN];
    float* Hg = reinterpret_cast<float*>(rec + a.L.H);
    float* sg = reinterpret_cast<float*>(rec + a.L.s);
    int32_t* winpos = reinterpret_cast<int32_t*>(rec + a.L.win_pos);
    T* wk = reinterpret_cast<T*>(rec + a.L.win_k);
    T* wvv = reinterpret_cast<T*>(rec + a.L.win_v);
    float* wphg = reinterpret_cast<float*>(rec + a.L.win_phi);
    int32_t* cpos = reinterpret_cast<int32_t*>(rec + a.L.c_pos);
    T* ck = reinterpret_cast<T*>(rec + a.L.c_k);
    T* cv = reinterpret_cast<T*>(rec + a.L.c_v);
    float* cphi = reinterpret_cast<float*>(rec + a.L.c_phi);
    float* cN = reinterpret_cast<float*>(rec + a.L.c_N);
    float* cz = reinterpret_cast<float*>(rec + a.L.c_z);
    float* evs = reinterpret_cast<float*>(rec + a.L.ev);

    const bool ev = t >= eta;
    const int e = t - eta;
    const int ring = t % eta;
    const bool nxt = t + 1 - eta >= 0;
    const int nring = (t + 1) % eta;
    const int wpr = (ev && tid == 0) ? winpos[ring] : e;   // checked once the burst is in

    // ---- 1. one burst of bulk copies issued by lanes of warp 0 (the TMA engine moves them
    //         while the threads load): the exact KV of cache and window, the slots' phi, the
    //         two evictees' phi, s and the evictee's N, z.  The new token, H and the slots'
    //         N, z, positions come by plain loads meanwhile ----
    const uint32_t bar = (uint32_t)__cvta_generic_to_shared(smb + M::MBAR);
    int* fail = reinterpret_cast<int*>(misc + 7);
    if (warp == 0) {
        constexpr uint32_t kPhiB = 4 * D, kKB = sizeof(T) * DK, kVB = sizeof(T) * DV;
        const uint32_t bytes = (uint32_t)nc * (kPhiB + kVB + kKB) + (uint32_t)eta * (kKB + kVB) +
                               (ev ? kPhiB + 4 * (DV + 4) : 0) + (nxt ? kPhiB : 0) + kPhiB;
        if (lane == 0) {
            *fail = 0;
            mbar_init(bar, 1);
            mbar_expect(bar, bytes);
        }
        __syncwarp();
        switch (lane) {
            case 0: if (nc > 0) bulk_g2s(cphi_s, cphi, nc * kPhiB, bar); break;
            case 1: bulk_g2s(rk_s, wk, eta * kKB, bar); break;
            case 2: if (nc > 0) bulk_g2s(cv_s, cv, nc * kVB, bar); break;
            case 3: bulk_g2s(rv_s, wvv, eta * kVB, bar); break;
            case 4: if (nc > 0) bulk_g2s(ck_s, ck, nc * kKB, bar); break;
            case 5: if (ev) bulk_g2s(phe, wphg + (size_t)ring * D, kPhiB, bar); break;
            case 6: if (nxt) bulk_g2s(phn, wphg + (size_t)nring * D, kPhiB, bar); break;
            case 7: bulk_g2s(s_sm, sg, kPhiB, bar); break;
            case 8: if (ev) bulk_g2s(evn, evs, 4 * (DV + 4), bar); break;
            default: break;
        }
    }
    if (tid < DK) {
        xq[tid] = IO<T>::ld(static_cast<const T*>(a.q) + (int64_t)bh * DK, tid);
        xk[tid] = IO<T>::ld(static_cast<const T*>(a.k) + (int64_t)bh * DK, tid);
    }
    if (tid < DV) nv_s[tid] = static_cast<const T*>(a.v)[(int64_t)bh * DV + tid];
    float hreg[HR * HC];
    h_load<D, DV>(hreg, Hg, warp, lane);
    // slot role (one pass: lambda <= 64)
    const int sl = tid / kSG, sub = tid % kSG;
    const bool live = sl < nc;
    float sN[PV], sz = 0.f;
    int spos = -1;
#pragma unroll
    for (int q = 0; q < PV; ++q) sN[q] = 0.f;
    if (live) {
        slot_load<DV>(cN + (size_t)sl * DV, sub, sN);
        sz = cz[sl];
        spos = cpos[sl];
    }
    __syncthreads();   // the new token staged, the barrier initialised; the burst may still be in flight
    if (!mbar_wait(bar, 0, kBurstWaitNs)) *fail = 1;
    __syncthreads();
    if (*fail) {
        // the burst did not land in time: flag the head and leave once its copies are done.
        // The second wait is long but finite (20 s): copies still in flight after it would
        // land in shared memory the CTA no longer owns, so the head's status word keeps
        // ST_TIMEOUT and nothing read after a timed-out step is trusted.
        if (tid == 0) {
            atomicOr(&hdr[HDR_STATUS], (int)ST_TIMEOUT);
            mbar_wait(bar, 0, 20ull * kBurstWaitNs);
        }
        return;
    }
    if (wpr != e) atomicOr(&hdr[HDR_STATUS], (int)ST_BAD_STATE);
    // the state of the head one wave ahead, into L2 (all heads step together, so its window
    // ring rows for this step are ring and nring as here); the window phi ring is skipped
    // but for those two rows
    if (a.prefetch_ahead > 0 && bh + a.prefetch_ahead < a.BH) {
        const char* nr = a.state + (int64_t)(bh + a.prefetch_ahead) * a.L.head_bytes;
        // (spread over warps 1 .. 14: warp 0 has just issued the burst, warp 15 scores the
        // evictee next)
        prefetch_l2(nr, a.L.win_phi, tid, kThreads, 1);
        prefetch_l2(nr + a.L.win_phi + (int64_t)ring * D * 4, D * 4, tid, kThreads, 2);
        prefetch_l2(nr + a.L.win_phi + (int64_t)nring * D * 4, D * 4, tid, kThreads, 3);
        prefetch_l2(nr + a.L.c_pos, a.L.head_bytes - a.L.c_pos, tid, kThreads, 8);
    }

    // ---- 2b. next evictee's partials; evictee and slot SREs ----
    if (nxt) h_partial_store<D, DV>(red, phn, hreg, warp, lane);
    float zn_prev = 0.f;
    if (warp == kEvWarp) {
        uint32_t ehi = kNoKey, elo = kNoKey;
        if (ev) {
            // the evictee's SRE in the warp layout (DV/32 consecutive entries per lane), the
            // arithmetic of the prefill chain's evictee warp
            constexpr int EV = DV / kWarp;
            float ve[PV], Nw[EV], vw[EV];
            slot_load_io<DV, T>(rv_s + (size_t)ring * DV, sub, ve);
            h_vec_load<EV>(evn + lane * EV, Nw);
            h_cols<DV, T>(rv_s + (size_t)ring * DV, lane, vw);
            const float es = warp_sre2<DV>(Nw, evn[DV], vw, slot_vv<DV>(ve));
            ehi = key_hi(es);
            elo = key_lo(e, kEvCode);
        }
        if (lane == 0) wkey[kDecWarps] = make_uint2(ehi, elo);
        // z' of the next evictee against s before this step's write
        if (nxt) zn_prev = warp_dot<D>(phn, s_sm, lane);
    }
    {
        float sv[PV];
        slot_load_io<DV, T>(cv_s + (size_t)(live ? sl : 0) * DV, sub, sv);
        const float sre = slot_sre2<DV>(sN, sz, sv, slot_vv<DV>(sv));
        uint32_t khi = live ? key_hi(sre) : kNoKey;
        uint32_t klo = live ? key_lo(spos, sl) : kNoKey;
        warp_min_key(khi, klo);
        if (lane == 0) wkey[warp] = make_uint2(khi, klo);
    }
    // ---- the scores q.k / sqrt(d) of every key the output may read, ahead of the decision:
    //      key 0 the new token, keys 1 .. nwin-1 the window (positions t-1, t-2, ...), key
    //      nwin + j cache slot j; the evictee's (its window row before the write) is kept
    //      aside (sc_e) and put in place once the decision says where it goes ----
    const float scale = 1.0f / sqrtf((float)DK);
    const int nwin = min(t + 1, eta);
    {
        float qs[PD];
        slot_load<DK>(xq, sub, qs);
        const int nk0 = nwin + nc;
        for (int base = 0; base < nk0; base += kThreads / kSG) {
            const int i = base + sl;
            float acc = 0.f;
            if (i < nk0) {
                int vo;
                float kv[PD];
                if (i == 0) {
                    slot_load<DK>(xk, sub, kv);
                    vo = (int)M::NV;
                } else {
                    const T* kr;
                    if (i < nwin) {
                        int r = ring - i;
                        r += r < 0 ? eta : 0;
                        kr = rk_s + (size_t)r * DK;
                        vo = (int)(M::RV + sizeof(T) * (size_t)r * DV);
                    } else {
                        const int j = i - nwin;
                        kr = ck_s + (size_t)j * DK;
                        vo = (int)(M::CV + sizeof(T) * (size_t)j * DV);
                    }
                    slot_load_io<DK, T>(kr, sub, kv);
                }
#pragma unroll
                for (int q = 0; q < PD; ++q) acc = fmaf(qs[q], kv[q], acc);
                if (sub == 0) voff[i] = vo;
            }
            acc += __shfl_xor_sync(kFull, acc, 1);
            acc += __shfl_xor_sync(kFull, acc, 2);
            acc += __shfl_xor_sync(kFull, acc, 4);
            if (i < nk0 && sub == 0) sc[i] = acc * scale;
        }
    }
    float sc_e = 0.f;   // the evictee's score (evictee warp)
    if (warp == kEvWarp && ev) {
        float qv[DK / kWarp], kv[DK / kWarp];
        h_vec_load<DK / kWarp>(xq + lane * (DK / kWarp), qv);
        h_cols<DK, T>(rk_s + (size_t)ring * DK, lane, kv);
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < DK / kWarp; ++q) acc = fmaf(qv[q], kv[q], acc);
        sc_e = warp_sum(acc) * scale;
    }
    __syncthreads();

    // ---- 3. decision (every warp) and write ----
    // phi(q), phi(k) of the token come from tok_phi_kernel, which may still be running when
    // this grid starts (programmatic dependent launch): wait for it, then fetch them into
    // registers (used at the write-back: each warp the phi(q) entries of its own H rows, the
    // first D threads the phi(k) row)
    grid_dep_wait();
    const float* tphi = reinterpret_cast<const float*>(rec + a.L.tok_phi);
    const float pq = lane < HR ? tphi[warp * HR + lane] : 0.f;
    const float pk = tid < D ? tphi[D + tid] : 0.f;
    const bool write = ev && (nc + 1 > lam);
    uint2 kk = lane <= kDecWarps ? wkey[lane] : make_uint2(kNoKey, kNoKey);
    warp_min_key(kk.x, kk.y);
    const int code = (int)(kk.y & 127u);
    const int wposn = write ? (int)(kk.y >> 7) : -1;
    const int wsel = !write ? -2 : (code == kEvCode ? -1 : code);   // -1: the evictee is written
    const float* wphi = wsel >= 0 ? cphi_s + (size_t)wsel * D : phe;
    const T* wvT = wsel >= 0 ? cv_s + (size_t)wsel * DV : rv_s + (size_t)ring * DV;
    // the moved evictee (written slot) and the appended one (no write)
    const int slot_new = (ev && !write) ? nc : (wsel >= 0 ? wsel : -1);
    const int nc_after = (ev && !write) ? nc + 1 : nc;
    if (write) {
        float vh[HC];
        h_cols<DV, T>(wvT, lane, vh);
        h_update<D, DV>(hreg, wphi, vh, warp);
        h_store<D, DV>(hst, hreg, warp, lane);   // staged for one bulk store (issued after the scores)
        if (warp == kEvWarp && lane < kSG) {
            float wp[PD], sr[PD];
            slot_load<D>(wphi, sub, wp);
            slot_load<D>(s_sm, sub, sr);
#pragma unroll
            for (int i = 0; i < PD; ++i) sr[i] += wp[i];
            slot_store<D>(s_sm, sub, sr);
        }
    }
    // slot update: every live slot absorbs the write; the written slot takes the evictee
    {
        const bool moved = live && sl == wsel;
        float sphi[PD];
        if (moved) {
            slot_load<D>(phe, sub, sphi);
            slot_load<DV>(evn, sub, sN);
            sz = evn[DV];
            spos = e;
        } else {
            slot_load<D>(cphi_s + (size_t)(live ? sl : 0) * D, sub, sphi);
        }
        if (write) {
            const float g = slot_gram<D>(wphi, sphi, sub);
            if (live) {
                slot_axpy_io<DV, T>(sN, g, wvT, sub);
                sz += g;
            }
        }
    }
    // ---- write back what is final now: H, s and every slot's N, z change only with a
    //      write (H and the N rows go out as bulk stores from shared memory once the scores
    //      are done; the moved slot's N row, whose phi row others still read, by plain
    //      stores); an append stores the evictee's own N, z; the new cache row; the new
    //      token into the window ring ----
    if (write) {
        if (warp == kEvWarp && lane < kSG) {
            float sr[PD];
            slot_load<D>(s_sm, sub, sr);
            slot_store<D>(sg, sub, sr);
        }
        if (live) {
            if (sl == wsel) slot_store<DV>(cN + (size_t)sl * DV, sub, sN);
            else slot_store<DV>(cphi_s + (size_t)sl * DV, sub, sN);
            if (sub == 0) {
                cz[sl] = sz;
                if (sl == wsel) cpos[sl] = e;
            }
        }
        fence_proxy_async();
    } else if (ev && sl == nc) {
        float Ne[PV];
        slot_load<DV>(evn, sub, Ne);
        slot_store<DV>(cN + (size_t)sl * DV, sub, Ne);
        if (sub == 0) {
            cz[sl] = evn[DV];
            cpos[sl] = e;
        }
    }
    if (slot_new >= 0) {
        if (tid < D) cphi[(size_t)slot_new * D + tid] = phe[tid];
        if (tid < DK) ck[(size_t)slot_new * DK + tid] = rk_s[(size_t)ring * DK + tid];
        if (tid < DV) cv[(size_t)slot_new * DV + tid] = rv_s[(size_t)ring * DV + tid];
    }
    if (tid < DK) IO<T>::st(wk, (int64_t)ring * DK + tid, xk[tid]);
    if (tid < DV) wvv[(int64_t)ring * DV + tid] = nv_s[tid];
    if (tid < D) wphg[(int64_t)ring * D + tid] = pk;
    if (lane < HR) phq[warp * HR + lane] = pq;   // this warp's rows (all of phq after the next barrier)
    // the next evictee: its partials summed in row-group order (column form); the gram of
    // this step's write with it (evictee warp; the correction is applied at the write-back)
    if (nxt && tid < DV) npart[tid] = reduce_partials_col<D, DV>(red, tid);
    float gn = 0.f, zn = zn_prev;
    if (warp == kEvWarp && nxt && write) {
        gn = warp_dot<D>(wphi, phn, lane);
        zn += gn;
    }
    __syncwarp();

    // ---- 4. output over window ∪ cache after the write: the evictee's score and value row
    //      where the decision put it (the slot it replaced, or appended as slot nc) ----
    // (the read mask's HIDE_CACHE reads the window keys only: they come first)
    const int nkeys = (a.read_mask & LOLA_READ_HIDE_CACHE) ? nwin : nwin + nc_after;
    if (warp == kEvWarp && lane == 0 && slot_new >= 0) {
        sc[nwin + slot_new] = sc_e;
        voff[nwin + slot_new] = (int)(M::RV + sizeof(T) * (size_t)ring * DV);
    }
    h_partial_store<D, DV>(red2, phq, hreg, warp, lane);
    __syncthreads();
    if (write && tid == 0) {
        // H, then the N rows but the moved slot's: they drain while the output is formed
        bulk_s2g(Hg, hst, 4 * D * DV);
        if (wsel > 0) bulk_s2g(cN, cphi_s, 4 * DV * wsel);
        const int r0 = wsel + 1;   // wsel = -1 (the evictee was written): every row
        if (r0 < nc) bulk_s2g(cN + (size_t)r0 * DV, cphi_s + (size_t)r0 * DV, 4 * DV * (nc - r0));
        bulk_commit();
    }
    // weights: every warp takes the maximum m over all scores (the order does not matter);
    // thread i < nkeys forms p_i = exp(score_i - m); the per-warp sums of p are added in warp
    // order at the end
    float mx = -INFINITY;
    for (int i = lane; i < nkeys; i += kWarp) mx = fmaxf(mx, sc[i]);
    mx = warp_max(mx);
    {
        const float p = tid < nkeys ? expf(sc[tid] - mx) : 0.f;
        if (tid < nkeys) pb[tid] = p;
        const float lw = warp_sum(p);
        if (lane == 0) lpart[warp] = lw;
    }
    if (warp == kEvWarp) {
        float sr[PD];
        slot_load<D>(s_sm, sub, sr);
        const float dl = slot_gram<D>(phq, sr, sub);
        if (lane == 0) misc[4] = dl;
    } else if (warp >= 1 && warp <= DV / kWarp) {
        // H^T phi(q): the row-group partials summed (column per thread)
        const int j = tid - kWarp;
        lin[j] = reduce_partials_col<D, DV>(red2, j);
    }
    __syncthreads();
    {
        // numerator: thread (split ks, column pair 2 kc, 2 kc + 1) over keys ks, ks + NS, ...;
        // the NS splits are then summed in order
        constexpr int NS = kThreads / (DV / 2);
        const int ks = tid / (DV / 2), kc = tid % (DV / 2);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        int i = ks;
        for (; i + NS < nkeys; i += 2 * NS) {
            float v0[2], v1[2];
            h_cols2<T>(reinterpret_cast<const T*>(smb + voff[i]), kc, v0);
            h_cols2<T>(reinterpret_cast<const T*>(smb + voff[i + NS]), kc, v1);
            const float p0 = pb[i], p1 = pb[i + NS];
            a0 = __ffma2_rn(make_float2(p0, p0), make_float2(v0[0], v0[1]), a0);
            a1 = __ffma2_rn(make_float2(p1, p1), make_float2(v1[0], v1[1]), a1);
        }
        if (i < nkeys) {
            float v0[2];
            h_cols2<T>(reinterpret_cast<const T*>(smb + voff[i]), kc, v0);
            const float p0 = pb[i];
            a0 = __ffma2_rn(make_float2(p0, p0), make_float2(v0[0], v0[1]), a0);
        }
        *reinterpret_cast<float2*>(red + ks * DV + 2 * kc) = make_float2(a0.x + a1.x, a0.y + a1.y);
    }
    __syncthreads();
    if (tid < DV) {
        constexpr int NS = kThreads / (DV / 2);
        float num = 0.f;
#pragma unroll
        for (int r = 0; r < NS; ++r) num += red[r * DV + tid];
        const float emx = expf(-mx);   // nkeys >= 1: the new token is always a key
        const float el = (a.read_mask & LOLA_READ_HIDE_STATE) ? 0.f : emx;   // the state's weight
        num = fmaf(el, lin[tid], num);
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) l += lpart[w];
        const float den = fmaf(el, misc[4], l);
        IO<T>::st(static_cast<T*>(a.y), (int64_t)bh * DV + tid, num / den);
    }

    // ---- 5. the next evictee's N, z; the header ----
    if (warp == kEvWarp && lane < kSG) {
        if (nxt) {
            // N of the next evictee: summed partials + this step's write (slot_axpy's order)
            float Nn[PV];
            slot_load<DV>(npart, sub, Nn);
            if (write) slot_axpy_io<DV, T>(Nn, gn, wvT, sub);
            slot_store<DV>(evs, sub, Nn);
            if (lane == 0) evs[DV] = zn;
        }
    }
    if (tid == 0) {
        winpos[ring] = t;
        hdr[HDR_T] = t + 1;
        hdr[HDR_NCACHE] = nc_after;
        if (write) hdr[HDR_NWRITTEN] = nwr + 1;
        if (a.written_pos) a.written_pos[bh] = wposn;
        bulk_wait_read();   // the bulk stores' shared-memory sources are read before the CTA ends
    }
}

// phi(q) and phi(k) of the token of every head into its tok_phi scratch, for
// decode_fast_kernel.  Head h has 2B rows to map (q then k of every batch row); CTA (h, g)
// stages W_h once and its kTokPhiWarps warps take kTokPhiRows consecutive rows each from
// row kTokPhiRowsPerCta * g on, with the arithmetic of the prefill's feature map (phi_rows:
// each row's result does not depend on how many rows a warp maps together).
constexpr int kTokPhiWarps = 4;
constexpr int kTokPhiRows = 8;
constexpr int kTokPhiRowsPerCta = kTokPhiWarps * kTokPhiRows;
template <int D, typename T>
__global__ void __launch_bounds__(kTokPhiWarps * kWarp) tok_phi_kernel(const DecArgs a, int B) {
    constexpr int DK = D;
    constexpr int NT = kTokPhiWarps * kWarp;
    extern __shared__ __align__(16) float smf[];
    float* Ws = smf;                                    // [D/2][DK+4]
    float* xs = smf + (D / 2) * w_stride<DK>();         // [kTokPhiWarps][kTokPhiRows][DK]
    grid_dep_launch();   // decode_fast_kernel may start its burst now; it waits for this grid
                         // before it reads tok_phi
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int h = blockIdx.x;
    const int j0 = blockIdx.y * kTokPhiRowsPerCta + warp * kTokPhiRows;   // this warp's first row
    const int t = reinterpret_cast<const int32_t*>(a.state)[HDR_T];   // all heads are at step t
    float* xw = xs + warp * kTokPhiRows * DK;
    // the rows first (their loads overlap W's), then W
    float xv[kTokPhiRows][DK / kWarp];
#pragma unroll
    for (int r = 0; r < kTokPhiRows; ++r) {
        const int j = j0 + r;
        const int b = j < B ? j : j - B;
        const T* src = static_cast<const T*>(j < B ? a.q : a.k) + ((int64_t)b * a.Hh + h) * DK;
#pragma unroll
        for (int c = 0; c < DK / kWarp; ++c) xv[r][c] = j < 2 * B ? IO<T>::ld(src, lane + kWarp * c) : 0.f;
    }
    stage_w<DK, D, NT>(Ws, a.W + (int64_t)h * a.w_head_stride, tid);
#pragma unroll
    for (int r = 0; r < kTokPhiRows; ++r)
#pragma unroll
        for (int c = 0; c < DK / kWarp; ++c) xw[r * DK + lane + kWarp * c] = xv[r][c];
    __syncthreads();
    // with this CTA's own loads in: the state of decode_fast_kernel's first wave (heads
    // 0 .. prefetch_ahead - 1) into L2, shared among this grid's CTAs (each later wave is
    // prefetched by the wave before it); of the window phi ring only the two rows the step
    // reads (the evictee's and the next one's)
    {
        const int ncta = gridDim.x * gridDim.y, cta = blockIdx.y * gridDim.x + blockIdx.x;
        const int wave = a.prefetch_ahead < a.BH ? a.prefetch_ahead : a.BH;
        const int64_t r0 = (int64_t)(t % a.eta) * 4 * D, r1 = (int64_t)((t + 1) % a.eta) * 4 * D;
        for (int hb = cta; hb < wave; hb += ncta) {
            const char* nr = a.state + (int64_t)hb * a.L.head_bytes;
            prefetch_l2(nr, a.L.win_phi, tid, NT);
            prefetch_l2(nr + a.L.c_pos, a.L.head_bytes - a.L.c_pos, tid, NT, 1);
            prefetch_l2(nr + a.L.win_phi + r0, 4 * D, tid, NT, 2);
            prefetch_l2(nr + a.L.win_phi + r1, 4 * D, tid, NT, 3);
        }
    }
    float ph[kTokPhiRows][D / 32];
    phi_rows<DK, D, kTokPhiRows>(xw, Ws, lane, ph);
#pragma unroll
    for (int r = 0; r < kTokPhiRows; ++r) {
        const int j = j0 + r;
        if (j >= 2 * B) break;
        const int b = j < B ? j : j - B;
        float* out = reinterpret_cast<float*>(a.state + ((int64_t)b * a.Hh + h) * a.L.head_bytes + a.L.tok_phi) +
                     (j < B ? 0 : D);
#pragma unroll
        for (int m = 0; m < D / 32; ++m) out[lane + 32 * m] = ph[r][m];
    }
}

// phi(q) and phi(k) of the token of every head on the tensor cores (phi_uses_tc: bf16,
// d_k = D = 128, one W for every head), with the arithmetic of the prefill's feature map
// (lola_phi_tc.cuh), so a decode step continues a prefill bit for bit.  The rows are q of
// heads 0 .. BH-1, then k of heads 0 .. BH-1; CTA g maps rows 128 g .. + 127: its threads
// gather the row tile and split W, one thread issues the 24 MMAs, and warp w forms half w / 4
// of the phi of rows 32 (w % 4) .. + 31 and writes it into each row's tok_phi scratch.
constexpr int kTokTcThreads = 256;
constexpr uint32_t kTokSW = 0;
constexpr uint32_t kTokSX = phitc::kWSplitBytes;
constexpr uint32_t kTokSEnd = kTokSX + phitc::kXBytes;
__global__ void __launch_bounds__(kTokTcThreads) tok_phi_tc_kernel(const DecArgs a) {
    using namespace tc;
    constexpr int D = phitc::kD;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    __shared__ __align__(8) uint64_t mbar;
    __shared__ uint32_t tmem_base;
    grid_dep_launch();   // decode_fast_kernel may start its burst now; it waits for this grid
                         // before it reads tok_phi
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int BH = a.BH;
    const int r0 = blockIdx.x * 128;
    if (tid == 0) mbar_init(smem_u32(&mbar), 1);
    if (warp == 0) tmem_alloc<phitc::kN>(smem_u32(&tmem_base));
    // the row tile: 16-byte chunks into the K-major swizzled layout, rows past 2 BH zero (all
    // of the thread's loads in flight before its first store; W's loads follow)
    constexpr int kXPer = 128 * 16 / kTokTcThreads;
    uint4 xv[kXPer];
#pragma unroll
    for (int u = 0; u < kXPer; ++u) {
        const int i = tid + u * kTokTcThreads;
        const int r = i >> 4, c16 = i & 15, j = r0 + r;
        xv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (j < 2 * BH) {
            const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(j < BH ? a.q : a.k) +
                                       (int64_t)(j < BH ? j : j - BH) * phitc::kDK + 8 * c16;
            xv[u] = *reinterpret_cast<const uint4*>(src);
        }
    }
    phitc::stage_w_split<kTokTcThreads>(sm + kTokSW, a.W, tid);
#pragma unroll
    for (int u = 0; u < kXPer; ++u) {
        const int i = tid + u * kTokTcThreads;
        const int r = i >> 4, c16 = i & 15;
        *reinterpret_cast<uint4*>(sm + kTokSX + (c16 >> 3) * phitc::kXAtom + kmaj_chunk(r, c16 & 7)) = xv[u];
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_base;
    if (tid == 0) {
        phitc::issue_mma(tb, sb + kTokSX, sb + kTokSW);
        mma_commit(smem_u32(&mbar));
    }
    // with this CTA's own loads in: the state of decode_fast_kernel's first wave (heads
    // 0 .. prefetch_ahead - 1) into L2, shared among this grid's CTAs; of the window phi ring
    // only the two rows the step reads (the evictee's and the next one's)
    if (a.prefetch_ahead > 0 && a.eta > 0) {
        const int t = reinterpret_cast<const int32_t*>(a.state)[HDR_T];   // all heads are at step t
        const int wave = a.prefetch_ahead < BH ? a.prefetch_ahead : BH;
        const int64_t p0 = (int64_t)(t % a.eta) * 4 * D, p1 = (int64_t)((t + 1) % a.eta) * 4 * D;
        for (int hb = blockIdx.x; hb < wave; hb += gridDim.x) {
            const char* nr = a.state + (int64_t)hb * a.L.head_bytes;
            prefetch_l2(nr, a.L.win_phi, tid, kTokTcThreads);
            prefetch_l2(nr + a.L.c_pos, a.L.head_bytes - a.L.c_pos, tid, kTokTcThreads, 1);
            prefetch_l2(nr + a.L.win_phi + p0, 4 * D, tid, kTokTcThreads, 2);
            prefetch_l2(nr + a.L.win_phi + p1, 4 * D, tid, kTokTcThreads, 3);
        }
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&mbar), 0, kBurstWaitNs));
    fence_after();
    const int quarter = warp & 3;
    const bool neg = warp >= 4;
    const int j = r0 + 32 * quarter + lane;
    const int hb = j < BH ? j : j - BH;
    if (ok) {
        float z[phitc::kN], e[phitc::kN];
        phitc::load_z(tb + ((uint32_t)(quarter * 32) << 16), z);
        phitc::half_phi(z, neg, e);
        if (j < 2 * BH) {
            float* out = reinterpret_cast<float*>(a.state + (int64_t)hb * a.L.head_bytes + a.L.tok_phi) +
                         (j < BH ? 0 : D) + (neg ? phitc::kN : 0);
#pragma unroll
            for (int c = 0; c < phitc::kN; c += 4)
                *reinterpret_cast<float4*>(out + c) = make_float4(e[c], e[c + 1], e[c + 2], e[c + 3]);
        }
    } else if (j < 2 * BH && !neg) {
        atomicOr(reinterpret_cast<int32_t*>(a.state + (int64_t)hb * a.L.head_bytes) + HDR_STATUS, (int)ST_TIMEOUT);
    }
    fence_before();
    __syncthreads();
    // TMEM is released only after the product has landed (a second, longer bounded wait when
    // the first one gave up)
    if (tid == 0 && !ok) mbar_wait(smem_u32(&mbar), 0, 20ull * kBurstWaitNs);
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc<phitc::kN>(tb);
}

// the fast path's limits (float32 KV at D = 128 does not fit one CTA's shared memory: the
// general kernel runs it)
template <int D, int DV, typename T>
bool fast_fits(const Dims& d) {
    return d.eta >= 1 && d.eta <= kFastEta && d.lam <= kFastLam && FastSmem<D, DV, T>::TOTAL <= kMaxSmemPerCta;
}

cudaError_t launch_tok_phi_tc(const Dims& d, const DecArgs& a, cudaStream_t st) {
    const size_t smem = kTokSEnd + 1024;
    cudaError_t e = cudaFuncSetAttribute(tok_phi_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tok_phi_tc_kernel<<<(2 * d.BH + 127) / 128, kTokTcThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_tok_phi_t(const Dims& d, const DecArgs& a, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((D / 2) * w_stride<D>() + kTokPhiRowsPerCta * D);
    auto kern = tok_phi_kernel<D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int B = d.BH / d.Hh;
    kern<<<dim3(d.Hh, (2 * B + kTokPhiRowsPerCta - 1) / kTokPhiRowsPerCta), kTokPhiWarps * kWarp, smem, st>>>(a, B);
    return cudaGetLastError();
}

template <int D, int DV, typename T>
bool launch_decode_fast(const Dims& d, const DecArgs& a, cudaStream_t st, cudaError_t* err) {
    if (!fast_fits<D, DV, T>(d)) return false;
    const size_t smem = FastSmem<D, DV, T>::TOTAL;
    auto kern = decode_fast_kernel<D, DV, T>;
    *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (*err != cudaSuccess) return true;
    // launched as a programmatic dependent of tok_phi_kernel (the launch before it on `st`)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.BH);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *err = cudaLaunchKernelEx(&cfg, kern, a);
    return true;
}

template <int D, int DV, typename T>
cudaError_t launch_decode_t(const Dims& d, const DecArgs& a, cudaStream_t st) {
    cudaError_t fe = cudaSuccess;
    if (launch_decode_fast<D, DV, T>(d, a, st, &fe)) return fe;
    constexpr int DK = D;
    constexpr int NRG = Shape<D, DV>::NRG;
    const size_t floats = (D / 2) * w_stride<DK>() + 4 * DK + 2 * DV + 4 * D + DV + NRG * DV + 2 * DV +
                          (d.eta + d.lam + 1) + 2 * (kDecWarps + 2) + 16;
    const size_t smem = sizeof(float) * floats + 64;
    auto kern = decode_kernel<D, DV, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<d.BH, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

namespace {
DecArgs make_args(const Dims& d, char* state, const Layout& L, const float* W, int64_t w_head_stride,
                  const void* q, const void* k, const void* v, void* y, int32_t* written_pos) {
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
    a.BH = d.BH;
    a.read_mask = d.read_mask;
    a.tok_phi_ready = 0;
    a.prefetch_ahead = 0;
    {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            a.prefetch_ahead = sms;   // one resident CTA per SM
    }
    return a;
}
}  // namespace

namespace {
bool decode_is_fast(const Dims& d) {
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128) return bf ? fast_fits<128, 128, __nv_bfloat16>(d) : fast_fits<128, 128, float>(d);
    if (d.D == 64 && d.dv == 64) return bf ? fast_fits<64, 64, __nv_bfloat16>(d) : fast_fits<64, 64, float>(d);
    return false;
}
}  // namespace

bool decode_uses_tok_phi(const Dims& d, int64_t w_head_stride) {
    return decode_is_fast(d) || phi_uses_tc(d, w_head_stride);
}

cudaError_t launch_tok_phi(const Dims& d, char* state, const Layout& L, const float* W, int64_t w_head_stride,
                           const void* q, const void* k, cudaStream_t st) {
    DecArgs a = make_args(d, state, L, W, w_head_stride, q, k, nullptr, nullptr, nullptr);
    if (!decode_is_fast(d)) a.prefetch_ahead = 0;   // the L2 prefetch serves the fast kernel's layout
    if (phi_uses_tc(d, w_head_stride)) return launch_tok_phi_tc(d, a, st);
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dk == 128)
        return bf ? launch_tok_phi_t<128, __nv_bfloat16>(d, a, st) : launch_tok_phi_t<128, float>(d, a, st);
    if (d.D == 64 && d.dk == 64)
        return bf ? launch_tok_phi_t<64, __nv_bfloat16>(d, a, st) : launch_tok_phi_t<64, float>(d, a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const Dims& d, char* state, const Layout& L, const float* W, int64_t w_head_stride,
                          const void* q, const void* k, const void* v, void* y, int32_t* written_pos,
                          cudaStream_t st) {
    DecArgs a = make_args(d, state, L, W, w_head_stride, q, k, v, y, written_pos);
    a.tok_phi_ready = phi_uses_tc(d, w_head_stride) ? 1 : 0;
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_decode_t<128, 128, __nv_bfloat16>(d, a, st) : launch_decode_t<128, 128, float>(d, a, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_decode_t<64, 64, __nv_bfloat16>(d, a, st) : launch_decode_t<64, 64, float>(d, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
