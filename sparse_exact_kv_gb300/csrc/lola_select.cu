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
// lambda > 64 -- owns one head for the whole sequence (layouts in lola_chain.cuh):
//   * cache slots live in registers, 8 lanes per slot, 4 slots per warp, 64 per CTA; a
//     write w costs each slot g = phi_w . phi_i, N += g v_w, z += g (exact: H changes by
//     a rank-1 term);
//   * each CTA holds a replica of H in registers (8 rows x 4 columns, or 4 x 2, per thread) to compute
//     the next evictee's H^T phi one step ahead and to emit the chunk snapshots;
//   * the evictee is finished in two parts: right after the previous decision the first
//     DV/32 warps sum the H^T phi partials and add the last write's correction, one column
//     per lane, and hand the vector to the last warp through a named barrier; the last
//     warp holds s and scores the evictee with the arithmetic of a slot;
//   * per step: apply the previous write; every warp scores its slots and takes its
//     packed-key minimum with two redux.sync; after the step's single barrier every warp
//     takes the CTA minimum itself and keeps the decision in registers; with CL > 1 each
//     CTA pushes its best key into every peer's shared memory with st.async, completing on
//     the peer's exchange mbarrier (one thread waits, bounded by 1 s, and a CTA barrier
//     hands the keys to the others); when the winner is a cached key, its owner CTA then
//     pushes its phi / v row the same way to every peer (the evictee, the usual winner, is
//     held by every CTA, so most steps move no row);
//   * evictee rows (phi(k_e), v_e) arrive by cp.async four steps ahead.
// At every chunk start it stores H, s and the cache positions, from which the parallel
// output kernel rebuilds every query's exact set and linear state.
#include <climits>

#include "lola_chain.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace chain;

constexpr int kSelWarps = kThreads / kWarp;
constexpr int kSPW = kWarp / kSG;          // slots per warp
constexpr int kSPC = kSelWarps * kSPW;     // slots per CTA
constexpr int kMaxCluster = 16;
constexpr int kPF = 4;                     // evictee prefetch distance (steps)
constexpr int kNEB = 8;                    // evictee ring buffers (indexed by step & 7)
constexpr uint64_t kXWaitNs = 1000000000ull;  // a cluster exchange not complete within 1 s is an error

struct SelArgs {
    int n, eta, lam, chunk, nck, CL, cl_shift, io_bf16;
    const float* phiK;   // [BH][n][D]
    const void* K;       // io [BH][n][D]
    const void* V;       // io [BH][n][DV]
    int32_t* wpos;       // [BH][n]
    int32_t* wstep;      // [BH][n]
    float* snapH;        // [BH][nck][D*DV] float32, or
    __nv_bfloat16* snapHb;  // the same in bf16 (exactly one of the two is set)
    float* snapS;        // [BH][nck][D]
    int32_t* snapC;      // [BH][nck][lam]
    int32_t* slotpos;    // [BH][lam]
    char* state;
    Layout L;
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
// ---- the cluster exchange: DSMEM pushes completing on the receiver's mbarrier ----
__device__ __forceinline__ void st_async_v2(uint32_t raddr, uint32_t x, uint32_t y, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
                 "r"(x), "r"(y), "r"(rbar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     raddr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Waits (acquire, cluster scope) for the phase of `parity` to complete, for at most
// kXWaitNs of wall time; false when it gave up.
__device__ __forceinline__ bool xbar_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = tc::globaltimer_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (tc::globaltimer_ns() - t0 > kXWaitNs) return false;
    }
}
// named barrier 1: the helper warps arrive, the evictee warp waits
__device__ __forceinline__ void named_arrive(int nthreads) {
    asm volatile("bar.arrive 1, %0;" ::"r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D, int DV, typename T>
struct SelSmem {
    // dynamic shared memory: the warp-best candidates' phi (float32) and v (input type),
    // double-buffered by step parity; (float32 inputs only) the slots' value rows; then
    // (clusters only) the rows the peer CTAs push, [2][CL] records of phi then v
    static constexpr size_t kRowBytes = sizeof(float) * D + sizeof(T) * DV;
    static constexpr size_t kXPhi = sizeof(float) * 2 * kSelWarps * D;
    static constexpr size_t kXV = sizeof(T) * 2 * kSelWarps * DV;
    static constexpr size_t kSV = sizeof(T) == 4 ? sizeof(float) * kSPC * DV : 0;
    static size_t bytes(int CL) { return kXPhi + kXV + kSV + (CL > 1 ? 2 * (size_t)CL * kRowBytes : 0); }
    static_assert(kRowBytes % 16 == 0, "pushed rows move in 16-byte pieces");
};

template <int D, int DV, bool CLUSTER, typename T>
__global__ void __launch_bounds__(kThreads, 1) select_kernel(const SelArgs a) {
    using S = Shape<D, DV>;
    using M = SelSmem<D, DV, T>;
    constexpr int PD = S::PD, PV = S::PV, NRG = S::NRG, HR = S::HR, HC = S::HC;
    constexpr int VCH = DV * (int)sizeof(T) / 16;  // 16-byte chunks of one value row
    constexpr int RCH = (int)(M::kRowBytes / 16);  // 16-byte chunks of one pushed row
    // Evictee roles: kHelp helper warps (warps 0, 1, 2, 6; helper i sums columns 32 i ..
    // 32 i + 31 of the H^T phi partials) and warp 0 also forms the previous write's gram with
    // the evictee; warp kSWarp holds s and forms the next evictee's z'; warp kVvWarp its
    // |v|^2; the last warp corrects N and z by the write and scores the evictee.  Named
    // barrier 1 hands the partial sums and the gram to the last warp.  Warp w issues from
    // scheduler w % 4: the roles leave the last warp's scheduler to it alone.
    constexpr int kEvWarp = kSelWarps - 1;
    constexpr int kHelp = DV / kWarp;
    constexpr int kSWarp = 5;
    constexpr int kVvWarp = 4;
    constexpr int kHandoff = (kHelp + 1) * kWarp;  // threads on named barrier 1
    static_assert(kHelp <= 4 && kSelWarps == 16, "roles");
    constexpr bool kPackV = sizeof(T) == 2;        // bfloat16 slot values stay in registers
    constexpr int VW = SlotWords<DV, T>::kWords;

    extern __shared__ __align__(16) unsigned char dyn_sm[];
    float (*xphi)[kSelWarps][D] = reinterpret_cast<float (*)[kSelWarps][D]>(dyn_sm);
    T (*xv)[kSelWarps][DV] = reinterpret_cast<T (*)[kSelWarps][DV]>(dyn_sm + M::kXPhi);
    float (*sv_sm)[DV] = reinterpret_cast<float (*)[DV]>(dyn_sm + M::kXPhi + M::kXV);
    unsigned char* rows = dyn_sm + M::kXPhi + M::kXV + M::kSV;   // pushed rows [2][CL]
    __shared__ __align__(16) float ebuf[kNEB][D];    // evictee phi(k), by step & 7
    __shared__ __align__(16) T evraw[kNEB][DV];      // evictee v as stored, by step & 7
    __shared__ __align__(16) float zero_phi[D];      // the "nothing written" winner
    __shared__ __align__(16) T zero_v[DV];
    __shared__ __align__(16) float red[2][NRG][DV];  // partials of the next evictee's H^T phi
    __shared__ __align__(16) float npart[2][DV];     // the evictee's summed partials
    __shared__ __align__(16) float nbuf[2][DV];      // the evictee's N (for its move into a slot)
    __shared__ float zbuf[2], gbuf[2], zpbuf[2], vvbuf[4];
    __shared__ uint2 wkey[2][kSelWarps + 1];         // per-warp minima; [16] = the evictee
    __shared__ uint2 exch[2][kMaxCluster];
    __shared__ __align__(8) uint64_t xbar[2];        // key exchange mbarriers (clusters)
    __shared__ __align__(8) uint64_t rbar[2];        // winner-row mbarriers (clusters)
    __shared__ int x_abort;
    __shared__ __align__(16) float s_sm[D];          // s, written only by the evictee warp's lanes 0-7

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int hidx = warp < 3 ? warp : (warp == 6 ? 3 : kHelp);   // helper index (kHelp: none)
    const int rank = CLUSTER ? (int)cluster_rank() : 0;
    const int CL = CLUSTER ? a.CL : 1;
    const int bh = CLUSTER ? (int)(blockIdx.x >> a.cl_shift) : (int)blockIdx.x;
    const int n = a.n, eta = a.eta, lam = a.lam;

    // slot role: phi and N in registers; v as raw words (bfloat16 pairs in registers,
    // float32 rows in shared memory)
    const int sl = lane / kSG, sub = lane % kSG;
    const int ls = warp * kSPW + sl;          // local slot
    const int gslot = ls * CL + rank;         // global slot (fill order)
    float sphi[PD], sN[PV], sz = 0.f, svv = 0.f;
    uint32_t svw[kPackV ? VW : 1];
    int spos = -1;
#pragma unroll
    for (int i = 0; i < PD; ++i) sphi[i] = 0.f;
#pragma unroll
    for (int i = 0; i < PV; ++i) sN[i] = 0.f;
#pragma unroll
    for (int i = 0; i < (kPackV ? VW : 1); ++i) svw[i] = 0u;
    if constexpr (!kPackV) {
        if (sub == 0)
            for (int i = 0; i < DV; ++i) sv_sm[ls][i] = 0.f;
    }
    auto slot_v = [&](float* out) {
        if constexpr (kPackV) slot_widen<DV, T>(svw, out);
        else slot_load<DV>(sv_sm[ls], sub, out);
    };

    // H role
    float h[HR * HC];
#pragma unroll
    for (int r = 0; r < HR * HC; ++r) h[r] = 0.f;
    if (tid < D) s_sm[tid] = 0.f;
    if (tid < 2) zpbuf[tid] = 0.f;    // z' against the empty memory
    const uint32_t xbar0 = smem_addr(&xbar[0]), rbar0 = smem_addr(&rbar[0]);
    if (tid == 0) {
        x_abort = 0;
        if (CLUSTER) {
            tc::mbar_init(xbar0, 1);
            tc::mbar_init(xbar0 + 8, 1);
            tc::mbar_init(rbar0, 1);
            tc::mbar_init(rbar0 + 8, 1);
        }
    }
    uint32_t rphase = 0u;   // completed phases of rbar[0] (bit 0) and rbar[1] (bit 1) in this CTA

    const float* phiK = a.phiK + (int64_t)bh * n * D;
    const int64_t vrow0 = (int64_t)bh * n;
    int32_t* wpos = a.wpos + (int64_t)bh * n;
    int32_t* wstep = a.wstep + (int64_t)bh * n;
    if (rank == 0)
        for (int i = tid; i < n; i += kThreads) wstep[i] = -1;

    // Evictee rows of step `step` (e = step - eta, for step <= n) arrive by cp.async:
    // threads [0, D/4) copy phi(k_e), threads [D/4, D/4 + VCH) copy v_e; one group per call.
    auto prefetch = [&](int step) {
        const int e = step - eta;
        if (step <= n && e >= 0) {
            if (tid < D / 4) {
                cp_async16(&ebuf[step & (kNEB - 1)][4 * tid], phiK + (int64_t)e * D + 4 * tid);
            } else if (tid < D / 4 + VCH) {
                const char* src = reinterpret_cast<const char*>(static_cast<const T*>(a.V) + (vrow0 + e) * DV);
                cp_async16(reinterpret_cast<char*>(evraw[step & (kNEB - 1)]) + 16 * (tid - D / 4),
                           src + 16 * (tid - D / 4));
            }
        }
        cp_async_commit();
    };
    // phi rows of steps before the first eviction stay zero (their partials are never used)
    for (int i = tid; i < kNEB * D; i += kThreads) (&ebuf[0][0])[i] = 0.f;
    for (int i = tid; i < D; i += kThreads) zero_phi[i] = 0.f;
    for (int i = tid; i < DV; i += kThreads) IO<T>::st(zero_v, i, 0.f);
    // the first evictee's partials are against the empty memory
    for (int i = tid; i < NRG * DV; i += kThreads) red[0][0][i] = 0.f;
    __syncthreads();
    for (int st = 0; st < kPF; ++st) prefetch(st);
    cp_async_wait<0>();
    int n_cached = 0, n_written = 0;
    // (clusters: every peer's exchange mbarriers are initialised before anything is pushed)
    if constexpr (CLUSTER) cluster_barrier(); else __syncthreads();
    // |v_e|^2 of the evictee of step t is computed at step t - 1; step 0's here
    auto prep_vv = [&](int step) {
        if (warp == kVvWarp && step <= n && step - eta >= 0) {
            float ve[PV];
            slot_load_io<DV, T>(evraw[step & (kNEB - 1)], sub, ve);
            const float vv = slot_vv<DV>(ve);
            if (lane == 0) vvbuf[step & 3] = vv;
        }
    };
    prep_vv(0);
    __syncthreads();

    // the decision of the previous step, held by every thread
    int d_write = 0, d_isev = 0, d_cta = 0, d_ws = 0;

    // The written candidate of step tp (phi, v) in this CTA's shared memory: the evictee
    // ring, this CTA's warp-best rows, or the row the owner CTA pushed; the zero row when
    // nothing was written.
    struct Win {
        const float* phi;
        const T* v;
    };
    auto winner = [&](bool wrote, int tp) -> Win {
        if (!wrote) return Win{zero_phi, zero_v};
        if (d_isev) return Win{ebuf[tp & (kNEB - 1)], evraw[tp & (kNEB - 1)]};
        const int wb = d_ws / kSPW;
        if (!CLUSTER || d_cta == rank) return Win{xphi[tp & 1][wb], xv[tp & 1][wb]};
        const unsigned char* r = rows + ((size_t)(tp & 1) * CL + d_cta) * M::kRowBytes;
        return Win{reinterpret_cast<const float*>(r), reinterpret_cast<const T*>(r + sizeof(float) * D)};
    };

    // Slots, then H, absorb the previous step's write (an exact zero update when nothing
    // was written, so the common path has no branch; an empty slot has phi = 0, g = 0).
    auto absorb_slot = [&](const Win& w) {
        const float g = slot_gram<D>(w.phi, sphi, sub);
        slot_axpy_io<DV, T>(sN, g, w.v, sub);
        sz += g;
    };
    auto absorb_h = [&](const Win& w) {
        float vh[HC];
        h_cols<DV, T>(w.v, lane, vh);
        h_update<D, DV>(h, w.phi, vh, warp);
    };
    // s absorbs it too (warp kSWarp, D/32 consecutive entries per lane)
    constexpr int ES = D / kWarp, EV = DV / kWarp;
    auto absorb_s = [&](const Win& w) {
        float wp[ES], sr[ES];
        h_vec_load<ES>(w.phi + lane * ES, wp);
        h_vec_load<ES>(s_sm + lane * ES, sr);
#pragma unroll
        for (int i = 0; i < ES; ++i) sr[i] += wp[i];
        h_vec_store<ES>(s_sm + lane * ES, sr);
        __syncwarp();
    };
    auto store_s = [&](float* dst) {
        float sr[ES];
        h_vec_load<ES>(s_sm + lane * ES, sr);
        h_vec_store<ES>(dst + lane * ES, sr);
    };

    int snap_next = 0, snap_c = 0;
    bool aborted = false;
    for (int t = 0; t < n; ++t) {
        const bool prev_write = d_write;
        const bool ev = t >= eta;
        const Win W = winner(prev_write, t - 1);

        // ---- helper warps: the evictee's partials summed in row-group order (column j per
        //      lane; the per-element order of slot_reduce_partials); warp 0: the gram of the
        //      previous write with the evictee ----
        if (hidx < kHelp && ev) {
            if (warp == 0) {
                const float g = prev_write ? warp_dot<D>(W.phi, ebuf[t & (kNEB - 1)], lane) : 0.f;
                if (lane == 0) gbuf[t & 1] = g;
            }
            // (clusters: summed in the previous step's key exchange, except for step 0)
            if (!CLUSTER || t == 0) {
                const int j = hidx * kWarp + lane;
                npart[t & 1][j] = reduce_partials_col<D, DV>(&red[t & 1][0][0], j);
            }
            named_arrive(kHandoff);
        }

        // ---- every warp: slots absorb the previous write; slot SREs; per-warp minimum ----
        absorb_slot(W);
        {
            float vr[PV];
            slot_v(vr);
            const float sre = slot_sre2<DV>(sN, sz, vr, svv);
            uint32_t khi = spos < 0 ? kNoKey : key_hi(sre);
            uint32_t klo = spos < 0 ? kNoKey : key_lo(spos, ls);
            const uint32_t mylo = klo;
            warp_min_key(khi, klo);
            if (lane == 0) wkey[t & 1][warp] = make_uint2(khi, klo);
            if (mylo == klo && klo != kNoKey) {
                slot_store<D>(xphi[t & 1][warp], sub, sphi);
                if constexpr (kPackV) slot_store_words<DV, T>(xv[t & 1][warp], sub, svw);
                else slot_store<DV>(reinterpret_cast<float*>(xv[t & 1][warp]), sub, vr);
            }
        }

        // ---- last warp: the evictee of step t, DV/32 consecutive entries per lane.
        //      N = partials + g v_w (one fma per entry), z = z' + g, then warp_sre2 ----
        if (warp == kEvWarp) {
            uint32_t ehi = kNoKey, elo = kNoKey;
            if (ev) {
                float Ne[EV], ve[EV];
                named_sync(kHandoff);
                h_vec_load<EV>(&npart[t & 1][lane * EV], Ne);
                float ze = zpbuf[t & 1];
                if (prev_write) {
                    const float g = gbuf[t & 1];
                    float vw[EV];
                    h_cols<DV, T>(W.v, lane, vw);
#pragma unroll
                    for (int i = 0; i < EV; ++i) Ne[i] = __fmaf_rn(g, vw[i], Ne[i]);
                    ze += g;
                }
                h_cols<DV, T>(evraw[t & (kNEB - 1)], lane, ve);
                const float es = warp_sre2<DV>(Ne, ze, ve, vvbuf[t & 3]);
                h_vec_store<EV>(&nbuf[t & 1][lane * EV], Ne);
                if (lane == 0) zbuf[t & 1] = ze;
                ehi = key_hi(es);
                elo = key_lo(t - eta, kEvCode);
            }
            if (lane == 0) wkey[t & 1][kSelWarps] = make_uint2(ehi, elo);
        }
        // ---- warp kSWarp: s absorbs the write; the next evictee's z' against s before
        //      step t's write ----
        if (warp == kSWarp) {
            absorb_s(W);
            if (t + 1 - eta >= 0) {
                const float zp = warp_dot<D>(ebuf[(t + 1) & (kNEB - 1)], s_sm, lane);
                if (lane == 0) zpbuf[(t + 1) & 1] = zp;
            }
        }

        // ---- every warp: H absorbs the write; the next evictee's H^T phi partials against
        //      the memory before step t's write ----
        absorb_h(W);
        h_partial_store<D, DV>(&red[(t + 1) & 1][0][0], ebuf[(t + 1) & (kNEB - 1)], h, warp, lane);

        // chunk-start snapshot of the memory before step t
        if (t == snap_next) {
            const int c = snap_c;
            snap_next += a.chunk;
            ++snap_c;
            if (rank == 0) {
                if (a.snapHb) h_store_bf16<D, DV>(a.snapHb + ((int64_t)bh * a.nck + c) * D * DV, h, warp, lane);
                else h_store<D, DV>(a.snapH + ((int64_t)bh * a.nck + c) * D * DV, h, warp, lane);
                if (warp == kSWarp) store_s(a.snapS + ((int64_t)bh * a.nck + c) * D);
            }
            if (sub == 0 && gslot < lam) a.snapC[((int64_t)bh * a.nck + c) * lam + gslot] = spos;
        }

        prep_vv(t + 1);
        prefetch(t + kPF);
        cp_async_wait<kPF - 2>();   // this thread's copies for step t + 2 have landed
        __syncthreads();

        // ---- decide (every warp): CTA minimum, then the cluster exchange ----
        const bool write = ev && (n_cached + 1 > lam);
        uint2 k = lane <= kSelWarps ? wkey[t & 1][lane] : make_uint2(kNoKey, kNoKey);
        warp_min_key(k.x, k.y);
        int bc = 0;
        if constexpr (CLUSTER) {
            // push this CTA's best key (warp 0) to every peer; the exchange mbarrier of step
            // parity b completes once all CL - 1 peers' keys have landed here
            const int b = t & 1;
            const uint32_t xb = xbar0 + 8 * b;
            if (warp == 0 && lane < CL && lane != rank)
                st_async_v2(map_rank(smem_addr(&exch[b][rank]), lane), k.x, k.y, map_rank(xb, lane));
            // while the peers' keys travel: the helpers sum the next evictee's H^T phi partials
            // (complete since the barrier above), which the next step would otherwise start with
            if (hidx < kHelp && t + 1 >= eta) {
                const int j = hidx * kWarp + lane;
                npart[(t + 1) & 1][j] = reduce_partials_col<D, DV>(&red[(t + 1) & 1][0][0], j);
            }
            if (tid == kThreads - 1) {
                mbar_arrive_expect_tx(xb, (uint32_t)((CL - 1) * 8));
                if (!xbar_wait(xb, (uint32_t)(t >> 1) & 1u)) x_abort = 1;
            }
            __syncthreads();
            if (x_abort) {
                aborted = true;
                break;
            }
            uint2 c = lane < CL ? (lane == rank ? k : exch[b][lane]) : make_uint2(kNoKey, kNoKey);
            uint32_t hi = c.x, lo = c.y;
            warp_min_key(hi, lo);
            // the owner CTA: lowest rank holding the minimum (the evictee is held by all)
            const unsigned hold = __ballot_sync(kFull, lane < CL && c.x == hi && c.y == lo);
            bc = __ffs(hold) - 1;
            k = make_uint2(hi, lo);
            // a cached key of another CTA is written: its owner pushes the key's phi / v row
            // (warps 1..4) into rows[b][owner] of every peer, completing on the peer's rbar[b]
            const int wcode = (int)(k.y & 127u);
            if (ev && (n_cached + 1 > lam) && wcode != kEvCode) {
                const uint32_t rb = rbar0 + 8 * b;
                if (bc == rank) {
                    if (warp >= 1 && warp <= 4) {
                        const unsigned char* sphi_ = reinterpret_cast<const unsigned char*>(xphi[b][wcode / kSPW]);
                        const unsigned char* sv_ = reinterpret_cast<const unsigned char*>(xv[b][wcode / kSPW]);
                        const uint32_t dst0 = smem_addr(rows + ((size_t)b * CL + rank) * M::kRowBytes);
                        for (int i = tid - kWarp; i < (CL - 1) * RCH; i += 4 * kWarp) {
                            const int pr = i / RCH, ch = i % RCH;
                            const int peer = pr < rank ? pr : pr + 1;
                            const uint4 v = ch < D / 4 ? reinterpret_cast<const uint4*>(sphi_)[ch]
                                                       : reinterpret_cast<const uint4*>(sv_)[ch - D / 4];
                            st_async_v4(map_rank(dst0 + 16 * ch, peer), v, map_rank(rb, peer));
                        }
                    }
                } else {
                    if (tid == kThreads - 1) {
                        mbar_arrive_expect_tx(rb, (uint32_t)M::kRowBytes);
                        if (!xbar_wait(rb, (rphase >> b) & 1u)) x_abort = 1;
                    }
                    rphase ^= 1u << b;
                    __syncthreads();
                    if (x_abort) {
                        aborted = true;
                        break;
                    }
                }
            }
        }
        const int code = (int)(k.y & 127u);
        const int pos = (int)(k.y >> 7);
        d_write = write;
        d_isev = write && code == kEvCode;
        d_cta = bc;
        d_ws = code;
        if (rank == 0 && tid == 0) {
            wpos[t] = write ? pos : -1;
            if (write) wstep[pos] = t;
        }
        // the surviving evictee moves into its slot now; it absorbs this step's write at
        // the next step like every other cached key
        if (ev && !d_isev) {
            const int tcta = write ? bc : (CLUSTER ? n_cached & (CL - 1) : 0);
            const int tls = write ? code : (CLUSTER ? n_cached >> a.cl_shift : n_cached);
            if (tcta == rank && tls == ls) {
                slot_load<D>(ebuf[t & (kNEB - 1)], sub, sphi);
                if constexpr (kPackV) {
                    slot_load_words<DV, T>(evraw[t & (kNEB - 1)], sub, svw);
                } else {
                    float vr[PV];
                    slot_load_io<DV, T>(evraw[t & (kNEB - 1)], sub, vr);
                    slot_store<DV>(sv_sm[ls], sub, vr);
                }
                slot_load<DV>(nbuf[t & 1], sub, sN);
                sz = zbuf[t & 1];
                svv = vvbuf[t & 3];
                spos = t - eta;
            }
        }
        if (ev && !write) ++n_cached;
        if (write) ++n_written;
    }
    if (aborted) {
        // an exchange did not complete in time: flag the head, leave its state as it is, and
        // give pushes still in flight time to land before the cluster's CTAs exit
        cp_async_wait<0>();
        if (tid == 0) atomicOr(reinterpret_cast<int32_t*>(a.state + (int64_t)bh * a.L.head_bytes) + HDR_STATUS,
                               (int)ST_TIMEOUT);
        if constexpr (CLUSTER) {
            const uint64_t t0 = tc::globaltimer_ns();
            while (tc::globaltimer_ns() - t0 < 20000ull) {
            }
            cluster_barrier();
        }
        return;
    }
    const bool last_write = d_write;
    const Win WL = winner(last_write, n - 1);
    absorb_slot(WL);
    absorb_h(WL);
    if (warp == kSWarp) absorb_s(WL);

    // ---- export the memory after token n-1 into the state record ----
    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    const T* Kin = static_cast<const T*>(a.K);
    const T* Vin = static_cast<const T*>(a.V);
    if (rank == 0) {
        int32_t* hdr = reinterpret_cast<int32_t*>(rec);
        if (tid == 0) {   // (the status word was cleared with the state before this launch)
            hdr[HDR_T] = n;
            hdr[HDR_NCACHE] = n_cached;
            hdr[HDR_NWRITTEN] = n_written;
        }
        h_store<D, DV>(reinterpret_cast<float*>(rec + a.L.H), h, warp, lane);
        if (warp == kSWarp) store_s(reinterpret_cast<float*>(rec + a.L.s));
        if (warp == kEvWarp) {
            // the next evictee (token n - eta): N against the memory after token n - 1
            if (eta > 0 && n - eta >= 0) {
                const float* eb = ebuf[n & (kNEB - 1)];
                float Ne[PV];
                slot_reduce_partials<D, DV>(&red[n & 1][0][0], sub, Ne);
                float ze = zpbuf[n & 1];
                if (last_write) {
                    const float g = warp_dot<D>(WL.phi, eb, lane);
                    slot_axpy_io<DV, T>(Ne, g, WL.v, sub);
                    ze += g;
                }
                float* evn = reinterpret_cast<float*>(rec + a.L.ev);
                if (lane < kSG) slot_store<DV>(evn, sub, Ne);
                if (lane == 0) evn[DV] = ze;
            }
        }
        // window ring: entry e holds the newest position p <= n-1 with p % eta == e
        int32_t* wp = reinterpret_cast<int32_t*>(rec + a.L.win_pos);
        T* wk = reinterpret_cast<T*>(rec + a.L.win_k);
        T* wv = reinterpret_cast<T*>(rec + a.L.win_v);
        float* wph = reinterpret_cast<float*>(rec + a.L.win_phi);
        for (int i = tid; i < eta * (1 + D + DV + D); i += kThreads) {
            const int e = i % eta, part = i / eta;
            const int p = (n - 1) - ((((n - 1) - e) % eta) + eta) % eta;
            if (part == 0) wp[e] = p >= 0 ? p : -1;
            else if (p < 0) continue;
            else if (part <= D) wk[(int64_t)e * D + (part - 1)] = Kin[(vrow0 + p) * D + (part - 1)];
            else if (part <= D + DV) wv[(int64_t)e * DV + (part - 1 - D)] = Vin[(vrow0 + p) * DV + (part - 1 - D)];
            else wph[(int64_t)e * D + (part - 1 - D - DV)] = phiK[(int64_t)p * D + (part - 1 - D - DV)];
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
    cnt += __shfl_xor_sync(kFull, cnt, 1);
    cnt += __shfl_xor_sync(kFull, cnt, 2);
    cnt += __shfl_xor_sync(kFull, cnt, 4);
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
        for (int r = n_cached + tid; r < lam; r += kThreads) reinterpret_cast<int32_t*>(rec + a.L.c_pos)[r] = -1;
}


template <int D, int DV, typename T>
cudaError_t launch_select_single(const Dims& d, const SelArgs& a, cudaStream_t st) {
    auto kern = select_kernel<D, DV, false, T>;
    const size_t smem = SelSmem<D, DV, T>::bytes(1);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<d.BH, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int D, int DV, typename T>
cudaError_t launch_select_cluster(const Dims& d, const SelArgs& a, cudaStream_t st) {
    auto kern = select_kernel<D, DV, true, T>;
    const size_t smem = SelSmem<D, DV, T>::bytes(a.CL);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (a.CL > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.BH * a.CL);
    cfg.blockDim = dim3(kThreads);
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
    e = cudaOccupancyMaxActiveClusters(&nclusters, (void*)kern, &cfg);
    if (e != cudaSuccess) return e;
    if (nclusters < 1) return cudaErrorInvalidConfiguration;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

// Number of CTAs per head: enough register slots for lambda cache entries (64 per CTA).
int select_cluster_size(int lam) {
    const int need = (lam + kSPC - 1) / kSPC;
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
    a.chunk = ws.snap_interval;
    a.nck = ws.nck;
    a.CL = select_cluster_size(d.lam);
    a.cl_shift = 0;
    while ((1 << a.cl_shift) < a.CL) ++a.cl_shift;
    a.io_bf16 = d.dtype == LOLA_BF16;
    a.phiK = ws.phiK;
    a.K = K;
    a.V = V;
    a.wpos = ws.wpos;
    a.wstep = ws.wstep;
    a.snapH = ws.snapH;
    a.snapHb = ws.snapHb;
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
