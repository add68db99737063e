// K3 (bf16, tensor cores): co-normalised LoLA output for every query, in parallel over
// (head, 128-query tile), as a warp-specialised tcgen05 pipeline.
//
// LoLA reading notes (arXiv 2505.23666v3), section 2.5, Eq. 14:
//   y_t = (H_t^T phi(q_t) + sum_{j in G_t ∪ W_t} a_tj v_j) / (phi(q_t)^T s_t + sum a_tj),
//   a_tj = exp(q_t . k_j / sqrt(d_k)).
// With w_j the step that wrote key j (none: never), key j is exact for query t iff
// j <= t < w_j and in the linear memory iff w_j <= t.  From the snapshot taken before the
// tile's chunk start c0 -- (H_c, s_c) and the cache positions -- the tile's pool is
// cache(c0) ∪ [c0 - eta, tile end), and for every query t of the tile
//   y_t = O_t / l_t,  O_t = 2^{-m} (phi(q_t)^T H_c + sum_pool p_tj v_j),
//                     l_t = 2^{-m} (phi(q_t)^T s_c + sum_pool p_tj),
//   p_tj = 2^{s_tj}             if j <= t < w_j   (s_tj = q_t . k_j log2(e) / sqrt(d_k)),
//        = phi(q_t) . phi(k_j)   if c0 <= w_j <= t  (written inside the chunk, before t),
//        = 0                     otherwise.
// The two cases exclude each other, so one weight matrix P carries both branches and one
// product P V accumulates the numerator.  m is a running maximum raised lazily: O is
// rescaled in TMEM only when a block's maximum exceeds m by more than 2^12 (m starts at 0,
// the scale of the snapshot term).
//
// Roles (416 threads):
//   * warps 9-12 (loaders): Q, phi(Q) and H_c tiles by TMA (cp.async.bulk.tensor, 128-byte
//     swizzle, rows past n zero-filled); per 64-key pool block the keys' positions and row
//     bounds (four blocks ahead, into a ring; the positions and write steps they need are
//     loaded an iteration earlier still), then its K, phi(K), V rows into one of three
//     stages -- a window block (consecutive positions) as TMA tiles, a cache block
//     (scattered positions) as 16-byte cp.async gathers from all 128 loader threads (many
//     requests in flight);
//   * warp 8 (MMA, one thread): O = phi(Q) H_c, then per block S = Q K^T and
//     L = phi(Q) phi(K)^T into one of two TMEM buffers, and O += P V of the block before
//     with P read from TMEM, each group committed to an mbarrier;
//   * warps 0-7 (weighting): two threads per query row (TMEM lane = row; warp w takes keys
//     32 (w / 4) .. + 31 of every block) read S and L, apply the masks, agree on the row
//     maximum, write bf16 P into one of two TMEM buffers and keep the row's partial
//     normaliser.
// Double buffers let block b + 1's S, L products and block b - 1's P V product run while
// block b is weighted.  Every wait is bounded by %globaltimer (1 s, then a status bit in
// the head's state and a per-launch abort flag).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace tc;

constexpr int kWeightWarps = 8;
constexpr int kMmaWarp = 8, kLoadWarp0 = 9, kLoadWarps = 4;
constexpr int kLoadThreads = kLoadWarps * kWarp;
constexpr int kThreadsTc = 13 * kWarp;   // 416
constexpr int kTM = 128;                 // query rows per tile (MMA M)
constexpr int kBN = 64;                  // pool keys per block (MMA N of S, L; K of P V)
constexpr int kD = 128;                  // d_k = d_v = D
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale2 = 12.0f;       // lazy rescale threshold (log2 units)
constexpr int kRing = 8;                 // blocks of key positions / row bounds kept
constexpr int kAhead = 4;                // blocks of row bounds computed ahead of the loads
constexpr uint64_t kWaitNs = 1000000000ull;  // a stage not reached within 1 s is an error

// shared-memory map (bytes from a 1024-aligned base): Q, phi(Q), then three stages of a pool
// block (K, phi(K) K-major [64 x 64] atoms; V MN-major [64 x d_v]).  Stage 1's K and phi(K)
// tiles reuse the H_c tile once phi(Q) H_c has completed.
constexpr int kStages = 3;
constexpr uint32_t SQ = 0;               // Q tile      K-major, 2 atoms x [128 x 64]
constexpr uint32_t SPQ = 32768;          // phi(Q) tile K-major
constexpr uint32_t SH = 98304;           // H_c         MN-major [K = D x N = d_v], 2 atoms
__device__ __forceinline__ uint32_t SK(int st) { return st == 0 ? 65536u : (st == 1 ? 98304u : 180224u); }
__device__ __forceinline__ uint32_t SPK(int st) { return st == 0 ? 81920u : (st == 1 ? 114688u : 196608u); }
__device__ __forceinline__ uint32_t SV(int st) { return 131072u + 16384u * (uint32_t)st; }
constexpr uint32_t SEND = 212992;
// TMEM columns: S and L double-buffered, O, then the bf16 weights P (two buffers of 128 x 64,
// two per 32-bit column): the P V product reads its A operand from TMEM
__device__ __forceinline__ uint32_t TS(int st) { return st ? 64u : 0u; }
__device__ __forceinline__ uint32_t TL(int st) { return st ? 192u : 128u; }
constexpr uint32_t TO = 256;
__device__ __forceinline__ uint32_t TP(int st) { return st ? 416u : 384u; }

// barrier slots
enum {
    B_Q = 0, B_H = 1, B_O = 2, B_KVFULL = 3, B_KVEMPTY = B_KVFULL + kStages, B_SFULL = B_KVEMPTY + kStages,
    B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_NBARS = B_PFULL + 2
};
// a pool block's stage is full after kLoadThreads + 1 arrivals: every loader thread's (its
// cp.async gathers landed, or a plain arrival for a TMA block), and loader 0's after the
// row bounds written ahead are in

struct TcMaps {
    CUtensorMap q, pq, k, pk, v, h;      // 3-D bf16 maps, 64-column boxes, 128-byte swizzle
};

struct TcArgs {
    int n, eta, lam, chunk, nck, read_mask;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    __nv_bfloat16* Y;
    const __nv_bfloat16* phiKb;  // [BH][n][D] bf16
    const int32_t* wstep;
    const float* snapS;
    const int32_t* snapC;
    char* state;                 // per-head status words (timeouts)
    int64_t head_bytes;
    int* abort_flag;             // set by any CTA whose wait timed out; later CTAs skip their work
    // cache-read mode (the write-magnitude cache on a delta-rule state): Q and K are the
    // RMS-scaled rows, the pool has no linear part, a null sink joins the softmax and
    // y = ystate + gate_h * (the softmax read)
    int hola, Hh;
    const float* sink;           // [Hh] the sink's logit
    const float* gate;           // [Hh] the cache read's weight
    const float* ystate;         // [BH][n][d_v] float32 state read-out
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void weight_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// barrier over the four loader warps that also ORs a predicate across them (every loader
// thread takes the same branch afterwards)
__device__ __forceinline__ bool loaders_or(bool x) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, 2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)x)
        : "memory");
    return r != 0;
}
// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreadsTc, 1) output_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    __shared__ __align__(8) uint64_t bars[B_NBARS];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_sm;
    __shared__ int kpos[kRing][kBN];
    __shared__ __align__(16) uint32_t kinfo[kRing][kBN];   // per key: soft rows [lo, hi), linear rows >= llo
    __shared__ uint32_t kfull[kRing][2];   // per half block: max lo | min hi << 8 | min llo << 16 over its 32 keys
    __shared__ float sS[kD];
    __shared__ float bmx[2][2][kTM];     // per block parity, the two half-block maxima of each row
    __shared__ float lpart[2][kTM];      // the two partial normalisers of each row

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.y;
    const int n = a.n;
    const int t0 = blockIdx.x * kTM, t1 = min(n, t0 + kTM);
    const int c = t0 / a.chunk, c0 = c * a.chunk;
    const int wlo = max(0, c0 - a.eta);
    const int P = a.lam + (t1 - wlo);
    const int nblk = (P + kBN - 1) / kBN;
    const int64_t row0 = (int64_t)bh * n;
    const bool hide_state = (a.read_mask & LOLA_READ_HIDE_STATE) != 0 || a.hola;
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        mbar_init(bar(B_H), 1);
        mbar_init(bar(B_O), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KVFULL + s), kLoadThreads + 1);
            mbar_init(bar(B_KVEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_SFULL + s), 1);
            mbar_init(bar(B_SFREE + s), kWeightWarps);
            mbar_init(bar(B_PFULL + s), kWeightWarps);
        }
        abort_sm = *reinterpret_cast<volatile int*>(a.abort_flag) != 0;
    }
    if (tid < kD) sS[tid] = a.hola ? 0.f : a.snapS[((int64_t)bh * a.nck + c) * kD + tid];
    if (warp == kMmaWarp) tmem_alloc<512>(smem_u32(&tmem_base));
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_base;

    // bounded wait on a barrier phase; gives up at once when another role has given up
    auto wait = [&](int i, uint32_t parity) -> bool {
        const uint32_t b = bar(i);
        uint64_t start = 0;
        for (int it = 0;; ++it) {
            uint32_t ok;
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}\n"
                : "=r"(ok)
                : "r"(b), "r"(parity)
                : "memory");
            if (ok) return true;
            if (*reinterpret_cast<volatile int*>(&abort_sm)) return false;
            const uint64_t now = globaltimer_ns();
            if (it == 0) start = now;
            else if (now - start > kWaitNs) {
                abort_sm = 1;
                return false;
            }
        }
    };

    if (warp >= kLoadWarp0) {
        // ================================ loaders ================================
        const int ltid = tid - kLoadWarp0 * kWarp;
        const int32_t* cpos = a.snapC + ((int64_t)bh * a.nck + c) * a.lam;
        const int32_t* wst = a.wstep ? a.wstep + row0 : nullptr;
        bool ok = !abort_sm;
        if (ok && ltid == 0) {
            mbar_expect(bar(B_Q), (a.hola ? 1 : 3) * 32768);
            for (int x = 0; x < 2; ++x) {
                tma_load3(sb + SQ + 16384 * x, &maps.q, 64 * x, t0, bh, bar(B_Q));
                if (!a.hola) {
                    tma_load3(sb + SPQ + 16384 * x, &maps.pq, 64 * x, t0, bh, bar(B_Q));
                    tma_load3(sb + SH + 16384 * x, &maps.h, 64 * x, 0, bh * a.nck + c, bar(B_Q));
                }
            }
        }
        // Positions and row bounds of block bb into ring slot bb % kRing (threads 0..63, one key
        // each).  A key's position (a cache list entry or a window index) and its write step are
        // two dependent global loads; they are issued ahead (the prologue batches blocks 0..5, the
        // loop issues block b + 6's position and block b + 5's write step while it finishes block
        // b + 4), so no block's bounds wait for memory on the loaders' path.
        auto load_p = [&](int bb) -> int {
            const int u = bb * kBN + ltid;
            if (ltid >= kBN || u >= P) return -1;
            return u < a.lam ? cpos[u] : wlo + (u - a.lam);
        };
        auto load_w = [&](int p) -> int { return (p >= 0 && !a.hola) ? wst[p] : -1; };   // (cache read: never written)
        auto finish = [&](int bb, int p, int w) {
            const int sl = bb & (kRing - 1);
            if (ltid < kBN) {
                // row r = t - t0 sees key p exactly iff lo <= r < hi, linearly iff r >= llo
                const int lo = p < 0 ? 255 : min(max(p - t0, 0), 255);
                int hi = p < 0 ? 0 : (w < 0 ? 255 : min(max(w - t0, 0), 255));
                // the read mask's HIDE_CACHE: only while the key is in the window (t < p + eta)
                if (p >= 0 && (a.read_mask & LOLA_READ_HIDE_CACHE)) hi = min(hi, min(max(p + a.eta - t0, 0), 255));
                const int llo = (p < 0 || w < c0 || hide_state) ? 255 : min(max(w - t0, 0), 255);
                kpos[sl][ltid] = p;
                kinfo[sl][ltid] = (uint32_t)lo | ((uint32_t)hi << 8) | ((uint32_t)llo << 16);
                // the rows for which every key of this half block is exact: [max lo, min hi)
                const uint32_t mlo = __reduce_max_sync(0xffffffffu, (uint32_t)lo);
                const uint32_t mhi = __reduce_min_sync(0xffffffffu, (uint32_t)hi);
                const uint32_t mll = __reduce_min_sync(0xffffffffu, (uint32_t)llo);
                if ((ltid & 31) == 0) kfull[sl][ltid >> 5] = mlo | (mhi << 8) | (mll << 16);
            }
        };
        int pq[kAhead + 2], wq[kAhead + 1];
#pragma unroll
        for (int bb = 0; bb < kAhead + 2; ++bb) pq[bb] = load_p(bb);
#pragma unroll
        for (int bb = 0; bb < kAhead + 1; ++bb) wq[bb] = load_w(pq[bb]);
#pragma unroll
        for (int bb = 0; bb < kAhead; ++bb)
            if (bb < nblk) finish(bb, pq[bb], wq[bb]);
        // the pipeline: block b + 4's (position, write step), block b + 5's position
        int p4 = pq[kAhead], w4 = wq[kAhead], p5 = pq[kAhead + 1];
        ok = !loaders_or(!ok);
        int issued = 0;
        for (int b = 0; b < nblk && ok; ++b) {
            const int st = b % kStages, u0 = b * kBN, sl = b & (kRing - 1);
            // block b + 5's write step and block b + 6's position, a whole iteration ahead of use
            const int w5 = load_w(p5), p6 = load_p(b + kAhead + 2);
            bool fail = false;
            if (ltid == 0) {
                if (b == 1) fail = !wait(B_H, 0);                      // stage 1 overlaps H_c
                if (!fail && b >= kStages) fail = !wait(B_KVEMPTY + st, ((b - kStages) / kStages) & 1);
            }
            if (loaders_or(fail)) {
                ok = false;
                break;
            }
            if (u0 >= a.lam) {
                // window block: consecutive positions wlo + u - lam (rows past the pool are masked)
                if (ltid == 0) {
                    const int r0 = wlo + (u0 - a.lam);
                    mbar_expect(bar(B_KVFULL + st), (a.hola ? 2 : 3) * 16384);
                    for (int x = 0; x < 2; ++x) {
                        tma_load3(sb + SK(st) + 8192 * x, &maps.k, 64 * x, r0, bh, bar(B_KVFULL + st));
                        if (!a.hola) tma_load3(sb + SPK(st) + 8192 * x, &maps.pk, 64 * x, r0, bh, bar(B_KVFULL + st));
                        tma_load3(sb + SV(st) + 8192 * x, &maps.v, 64 * x, r0, bh, bar(B_KVFULL + st));
                    }
                } else {
                    mbar_arrive1(bar(B_KVFULL + st));
                }
            } else {
                // cache (or mixed) block: gathered rows, zero rows for empty slots; each thread's
                // arrival waits for its own copies, so the loaders move on at once
                for (int i = ltid; i < kBN * 16; i += kLoadThreads) {
                    const int r = i >> 4, c16 = i & 15;
                    const int p = kpos[sl][r];
                    const uint32_t off = (c16 >> 3) * 8192 + kmaj_chunk(r, c16 & 7);
                    const uint32_t voff = mnmaj_chunk(r, c16 * 8, kBN);
                    const int64_t g = (row0 + (p >= 0 ? p : 0)) * kD + c16 * 8;
                    const uint32_t nb = p >= 0 ? 16u : 0u;
                    cp_async16_z(sb + SK(st) + off, a.K + g, nb);
                    if (!a.hola) cp_async16_z(sb + SPK(st) + off, a.phiKb + g, nb);
                    cp_async16_z(sb + SV(st) + voff, a.V + g, nb);
                }
                cp_async_arrive_noinc(bar(B_KVFULL + st));
            }
            if (b + kAhead < nblk) finish(b + kAhead, p4, w4);   // its slot's block (b - 4) is long weighted
            p4 = p5;
            w4 = w5;
            p5 = p6;
            loaders_or(false);                           // the ring slot is written before it is read
            if (ltid == 0) mbar_arrive1(bar(B_KVFULL + st));   // (releases the ring slots written so far)
            issued = b + 1;
        }
        // leave no copy in flight: this thread's gathers, then the stages the loaders filled
        // (bounded)
        cp_async_wait_all();
        if (ltid == 0 && issued > 0) {
            const uint64_t t_start = globaltimer_ns();
            for (int b = max(0, issued - kStages); b < issued; ++b)
                while (!mbar_wait(bar(B_KVFULL + b % kStages), (b / kStages) & 1, 1000000ull))
                    if (globaltimer_ns() - t_start > kWaitNs) break;
        }
    } else if (warp == kMmaWarp) {
        // ================================ MMA issue ================================
        bool ok = !abort_sm && wait(B_Q, 0);
        fence_after();
        if (lane == 0) {
            if (ok && !hide_state) {
                constexpr uint32_t id = idesc_bf16(kTM, kD, 1);
                for (int k = 0; k < kD / 16; ++k) {
                    const uint64_t ad = sdesc(sb + SPQ + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc(sb + SH + k * 2048, 16384, 1024);
                    mma_bf16(tb + TO, ad, bd, id, k > 0);
                }
            }
            mma_commit(bar(B_H));
            auto pv = [&](int j) -> bool {
                const int sj = j & 1, kv = j % kStages;
                if (!wait(B_PFULL + sj, (j >> 1) & 1)) return false;
                fence_after();
                constexpr uint32_t id = idesc_bf16(kTM, kD, 1);
                for (int k = 0; k < kBN / 16; ++k) {
                    const uint64_t vd = sdesc(sb + SV(kv) + k * 2048, 8192, 1024);
                    mma_bf16_ts(tb + TO, tb + TP(sj) + 8 * k, vd, id, !(hide_state && j == 0 && k == 0));
                }
                mma_commit(bar(B_KVEMPTY + kv));
                return true;
            };
            for (int b = 0; b < nblk && ok; ++b) {
                const int st = b & 1, kv = b % kStages;
                ok = wait(B_KVFULL + kv, (b / kStages) & 1);
                if (ok && b >= 2) ok = wait(B_SFREE + st, ((b - 2) >> 1) & 1);
                if (!ok) break;
                fence_after();
                fence_async_smem();   // rows gathered by cp.async (generic proxy) before the MMA reads them
                // L only when some key of the block is linear for some row of the tile
                const uint32_t f0 = kfull[b & (kRing - 1)][0], f1 = kfull[b & (kRing - 1)][1];
                const bool need_l = min((f0 >> 16) & 255u, (f1 >> 16) & 255u) < (uint32_t)kTM;
                constexpr uint32_t id = idesc_bf16(kTM, kBN, 0);
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t ao = (k >> 2) * 16384 + (k & 3) * 32, bo = (k >> 2) * 8192 + (k & 3) * 32;
                    mma_bf16(tb + TS(st), sdesc(sb + SQ + ao, 16, 1024), sdesc(sb + SK(kv) + bo, 16, 1024), id, k > 0);
                    if (need_l)
                        mma_bf16(tb + TL(st), sdesc(sb + SPQ + ao, 16, 1024), sdesc(sb + SPK(kv) + bo, 16, 1024), id, k > 0);
                }
                mma_commit(bar(B_SFULL + st));
                if (b >= 1) ok = pv(b - 1);
            }
            if (ok) ok = pv(nblk - 1);
            mma_commit(bar(B_O));
            // leave no MMA in flight
            if (!mbar_wait(bar(B_O), 0, kWaitNs)) abort_sm = 1;
        }
        __syncwarp();
    } else {
        // ================================ weighting ================================
        // Every weighting warp runs all nblk iterations and both named-barrier syncs of each,
        // whatever happens, so the barrier counts always match; after a failed wait (warp-
        // uniform through __all_sync) an iteration only keeps the counts.
        const int hf = warp >> 2, row = ((warp & 3) << 5) + lane, t = t0 + row;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const float c2 = kLog2e / sqrtf((float)kD);
        auto wwait = [&](int i, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(i, parity)); };
        float m_run = 0.f, lp = 0.f;
        bool ok = __all_sync(0xffffffffu, !abort_sm) && wwait(B_Q, 0);
        if (ok && !hide_state) {
            // phi(q_t)^T s_c over features 64 hf .. 64 hf + 63, from the bf16 phi(Q) tile
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const int c16 = 8 * hf + c8;
                const uint4 x = *reinterpret_cast<const uint4*>(sm + SPQ + (c16 >> 3) * 16384 + kmaj_chunk(row, c16 & 7));
                const uint32_t wds[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    lp = fmaf(__uint_as_float(wds[q] << 16), sS[c16 * 8 + 2 * q], lp);
                    lp = fmaf(__uint_as_float(wds[q] & 0xffff0000u), sS[c16 * 8 + 2 * q + 1], lp);
                }
            }
        }
        for (int b = 0; b < nblk; ++b) {
            const int st = b & 1;
            if (ok) ok = wwait(B_SFULL + st, (b >> 1) & 1) && wwait(B_KVFULL + b % kStages, (b / kStages) & 1);
            float sv[32];
            uint32_t vis = 0u;
            float bm = -INFINITY;
            const uint32_t* ki = kinfo[b & (kRing - 1)] + 32 * hf;
            // every key of this half block exact for all 32 rows of the warp: no masks, no L
            const uint32_t kf = kfull[b & (kRing - 1)][hf];
            const int rbase = (warp & 3) * 32;
            const bool full = (int)(kf & 255u) <= rbase && (int)((kf >> 8) & 255u) >= rbase + 32;
            if (ok) {
                fence_after();
                tmem_ld32(tb + lane_off + TS(st) + 32 * hf, sv);
                tmem_wait_ld();
                // ---- masks and this half's maximum ----
                if (full) {
                    vis = 0xffffffffu;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) bm = fmaxf(bm, sv[jj]);
                } else {
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const uint4 in4 = reinterpret_cast<const uint4*>(ki)[j4];
                        const uint32_t iv[4] = {in4.x, in4.y, in4.z, in4.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int jj = 4 * j4 + q;
                            const bool vs = row >= (int)(iv[q] & 255u) && row < (int)((iv[q] >> 8) & 255u);
                            vis |= (uint32_t)vs << jj;
                            bm = vs ? fmaxf(bm, sv[jj]) : bm;
                        }
                    }
                }
            }
            bmx[st][hf][row] = bm;
            weight_sync();
            if (!ok) continue;
            bm = fmaxf(bmx[st][0][row], bmx[st][1][row]) * c2;
            // lazy rescale: both threads of a row take the same decision; TMEM accesses stay
            // warp-uniform (factor 1 for the rows that keep m)
            const bool need = bm > m_run + kRescale2;
            if (__any_sync(0xffffffffu, need)) {
                if (b == 0 && hide_state) {
                    if (need) m_run = bm;                  // O holds nothing yet
                } else {
                    // O is quiescent once the product before this block has completed
                    ok = b >= 1 ? wwait(B_KVEMPTY + (b - 1) % kStages, ((b - 1) / kStages) & 1) : wwait(B_H, 0);
                    if (!ok) continue;
                    fence_after();
                    const float f = need ? ex2(m_run - bm) : 1.f;
                    lp *= f;
#pragma unroll
                    for (int cc = 0; cc < kD / 2; cc += 32) {
                        float o[32];
                        tmem_ld32(tb + lane_off + TO + 64 * hf + cc, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] *= f;
                        tmem_st32(tb + lane_off + TO + 64 * hf + cc, o);
                    }
                    tmem_wait_st();
                    fence_before();
                    if (need) m_run = bm;
                }
            }
            const float mr = m_run, em = ex2(-m_run);
            float lnext[8];
            // P[st] is free once the product of block b - 2 has completed
            if (b >= 2) {
                ok = wwait(B_KVEMPTY + (b - 2) % kStages, ((b - 2) / kStages) & 1);
                if (!ok) continue;
            }
            uint32_t pw[16];   // this thread's 32 weights, bf16 pairs
            if (full) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float e0 = ex2(fmaf(sv[2 * i], c2, -mr)), e1 = ex2(fmaf(sv[2 * i + 1], c2, -mr));
                    const __nv_bfloat162 bp = __floats2bfloat162_rn(e0, e1);
                    const float2 fp = __bfloat1622float2(bp);
                    lp += fp.x + fp.y;
                    pw[i] = *reinterpret_cast<const uint32_t*>(&bp);
                }
            } else
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float lv[8];
                if (hide_state) {
                    // no key is linear for any row (llo = 255) and L was never computed
#pragma unroll
                    for (int j = 0; j < 8; ++j) lv[j] = 0.f;
                } else if ((c4 & 1) == 0) {
                    float l16[16];
                    tmem_ld16(tb + lane_off + TL(st) + 32 * hf + 8 * c4, l16);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j) lv[j] = l16[j];
                    lnext[0] = l16[8]; lnext[1] = l16[9]; lnext[2] = l16[10]; lnext[3] = l16[11];
                    lnext[4] = l16[12]; lnext[5] = l16[13]; lnext[6] = l16[14]; lnext[7] = l16[15];
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) lv[j] = lnext[j];
                }
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    float e[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int jj = c4 * 8 + 2 * hh + u;
                        const bool vs = (vis >> jj) & 1u;
                        const bool vl = row >= (int)((ki[jj] >> 16) & 255u);
                        e[u] = vs ? ex2(fmaf(sv[jj], c2, -mr)) : (vl ? lv[jj - 8 * c4] * em : 0.f);
                    }
                    const __nv_bfloat162 bp = __floats2bfloat162_rn(e[0], e[1]);
                    const float2 fp = __bfloat1622float2(bp);
                    lp += fp.x + fp.y;
                    pw[4 * c4 + hh] = *reinterpret_cast<const uint32_t*>(&bp);
                }
            }
            tmem_st16(tb + lane_off + TP(st) + 16 * hf, pw);
            tmem_wait_st();
            // S[st], L[st] are read and P[st] is written: the MMA may overwrite S, L with block
            // b + 2's products and read P
            fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive1(bar(B_SFREE + st));
                mbar_arrive1(bar(B_PFULL + st));
            }
        }
        // ---- epilogue: y = O / l; thread (row, hf) writes output columns 64 hf .. 64 hf + 63 ----
        // (cache read: the head's sink and gate and this thread's 64 state read-out values are
        // fetched before the last product is waited for)
        float sink_l2 = 0.f, gh = 1.f;
        float4 yst[16];
        if (a.hola) {
            const int h = bh % a.Hh;
            sink_l2 = a.sink[h] * kLog2e;
            gh = a.gate[h];
            if (t < n) {
                const float4* ys = reinterpret_cast<const float4*>(a.ystate + (row0 + t) * kD + 64 * hf);
#pragma unroll
                for (int j4 = 0; j4 < 16; ++j4) yst[j4] = ys[j4];
            }
        }
        if (ok) ok = wwait(B_O, 0);
        fence_after();
        lpart[hf][row] = lp;
        weight_sync();
        if (ok) {
            float l = lpart[0][row] + lpart[1][row];
            // the null sink (value 0) joins the normaliser at the row's scale 2^-m
            if (a.hola) l += ex2(sink_l2 - m_run);
            const float inv = t < n ? gh / l : 0.f;
#pragma unroll
            for (int cc = 0; cc < kD / 2; cc += 32) {
                float o[32];
                tmem_ld32(tb + lane_off + TO + 64 * hf + cc, o);
                tmem_wait_ld();
                if (a.hola && t < n) {
                    // y = the state read-out + gate * the cache read
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 y4 = yst[cc / 4 + j4];
                        o[4 * j4] = fmaf(o[4 * j4], inv, y4.x);
                        o[4 * j4 + 1] = fmaf(o[4 * j4 + 1], inv, y4.y);
                        o[4 * j4 + 2] = fmaf(o[4 * j4 + 2], inv, y4.z);
                        o[4 * j4 + 3] = fmaf(o[4 * j4 + 3], inv, y4.w);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= inv;
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const __nv_bfloat162 bv = __floats2bfloat162_rn(o[j], o[j + 1]);
                    pk[j / 2] = *reinterpret_cast<const uint32_t*>(&bv);
                }
                if (t < n) {
                    __nv_bfloat16* y = a.Y + (row0 + t) * kD + 64 * hf + cc;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(y + 8 * q) =
                            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (abort_sm && tid == 0) {
        atomicOr(reinterpret_cast<int32_t*>(a.state + (int64_t)bh * a.head_bytes) + HDR_STATUS, (int)ST_TIMEOUT);
        atomicExch(a.abort_flag, 1);
    }
    if (warp == kMmaWarp) tmem_dealloc<512>(tb);
}

// bf16 tensor [depth][rows][128], boxes of 64 columns x box_rows rows x 1, 128-byte swizzle,
// rows past `rows` zero-filled
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t depth, int box_rows) {
    return make_tmap3(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, kD, rows, depth, 64, box_rows);
}

}  // namespace

namespace tc {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool make_tmap3(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* base, int64_t inner,
                int64_t rows, int64_t depth, int box_inner, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)depth};
    const cuuint64_t strides[2] = {(cuuint64_t)(inner * elem_bytes), (cuuint64_t)(inner * elem_bytes * rows)};
    const cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace tc

bool output_tc_supported(const Dims& d) { return d.dtype == LOLA_BF16 && d.D == kD && d.dk == kD && d.dv == kD; }

cudaError_t launch_output_tc(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K, const void* V,
                             void* Y, char* state, int64_t head_bytes, cudaStream_t st) {
    TcMaps maps;
    if (!make_map(&maps.q, Q, n, d.BH, kTM) || !make_map(&maps.pq, ws.phiQb, n, d.BH, kTM) ||
        !make_map(&maps.k, K, n, d.BH, kBN) || !make_map(&maps.pk, ws.phiKb, n, d.BH, kBN) ||
        !make_map(&maps.v, V, n, d.BH, kBN) || !make_map(&maps.h, ws.snapHb, kD, (int64_t)d.BH * ws.nck, kD))
        return cudaErrorInvalidValue;
    TcArgs a;
    a.n = n;
    a.eta = d.eta;
    a.lam = d.lam;
    a.chunk = ws.snap_interval;
    a.nck = ws.nck;
    a.read_mask = d.read_mask;
    a.K = static_cast<const __nv_bfloat16*>(K);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.phiKb = ws.phiKb;
    a.wstep = ws.wstep;
    a.snapS = ws.snapS;
    a.snapC = ws.snapC;
    a.state = state;
    a.head_bytes = head_bytes;
    a.abort_flag = ws.abort_flag;
    a.hola = 0;
    a.Hh = d.Hh;
    a.sink = a.gate = a.ystate = nullptr;
    const size_t smem = SEND + 1024;
    cudaError_t e = cudaFuncSetAttribute(output_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    output_tc_kernel<<<dim3((n + kTM - 1) / kTM, d.BH), kThreadsTc, smem, st>>>(maps, a);
    return cudaGetLastError();
}

// The cache read of the write-magnitude cache layer: Qt, Kt the RMS-scaled rows (bf16), pool =
// the persistent cache listed per chunk in snapC ([BH][nck][w], -1 empty) and the chunk's own
// tokens up to the query (eta = 0, never written); y = ystate + gate_h * softmax read with a
// null sink of logit sink_h.  status: [BH][4] int32 (ST_TIMEOUT in word 3 of a head).
cudaError_t launch_output_tc_hola(int BH, int Hh, int n, int w, int chunk, const void* Qt, const void* Kt,
                                  const void* V, void* Y, const int32_t* snapC, int nck, const float* ystate,
                                  const float* sink, const float* gate, int32_t* status, int* abort_flag,
                                  cudaStream_t st) {
    TcMaps maps;
    // the phi(Q), phi(K) and H_c maps are never used in this mode: any valid tensor serves
    if (!make_map(&maps.q, Qt, n, BH, kTM) || !make_map(&maps.pq, Qt, n, BH, kTM) || !make_map(&maps.k, Kt, n, BH, kBN) ||
        !make_map(&maps.pk, Kt, n, BH, kBN) || !make_map(&maps.v, V, n, BH, kBN) || !make_map(&maps.h, Qt, n, BH, kD))
        return cudaErrorInvalidValue;
    TcArgs a;
    a.n = n;
    a.eta = 0;
    a.lam = w;
    a.chunk = chunk;
    a.nck = nck;
    a.read_mask = 0;
    a.K = static_cast<const __nv_bfloat16*>(Kt);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.phiKb = nullptr;
    a.wstep = nullptr;
    a.snapS = nullptr;
    a.snapC = snapC;
    a.state = reinterpret_cast<char*>(status);
    a.head_bytes = 4 * sizeof(int32_t);
    a.abort_flag = abort_flag;
    a.hola = 1;
    a.Hh = Hh;
    a.sink = sink;
    a.gate = gate;
    a.ystate = ystate;
    const size_t smem = SEND + 1024;
    cudaError_t e = cudaFuncSetAttribute(output_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    output_tc_kernel<<<dim3((n + kTM - 1) / kTM, BH), kThreadsTc, smem, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace lola
