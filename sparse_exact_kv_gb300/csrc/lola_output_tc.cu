// K3 (bf16, tensor cores): co-normalised LoLA output for every query, in parallel over
// (head, 128-query tile), with tcgen05 MMAs accumulating in TMEM.
//
// LoLA reading notes (arXiv 2505.23666v3), section 2.5, Eq. 14:
//   y_t = (H_t^T phi(q_t) + sum_{j in G_t ∪ W_t} a_tj v_j) / (phi(q_t)^T s_t + sum a_tj),
//   a_tj = exp(q_t . k_j / sqrt(d_k)).
// With w_j the step that wrote key j (none: never), key j is exact for query t iff
// j <= t < w_j and in the linear memory iff w_j <= t.  From the snapshot taken before
// the tile's chunk start c0 -- (H_c, s_c) and the cache positions -- the tile's pool is
// cache(c0) ∪ [c0 - eta, tile end), and for every query t of the tile
//   O_soft = sum_pool [j <= t < w_j] 2^(s_tj - m) v_j,      l_soft = sum of the weights,
//   O_lin  = phi(q_t)^T H_c + sum_pool [c0 <= w_j <= t] (phi(q_t) . phi(k_j)) v_j,
//   l_lin  = phi(q_t)^T s_c + sum of those linear weights,
//   y_t    = (O_soft + 2^{-m} O_lin) / (l_soft + 2^{-m} l_lin),
// with scores s_tj = q_t . k_j log2(e) / sqrt(d_k) in log2 units.
// The tensor cores compute S = Q K^T, L = phi(Q) phi(K)^T (per 64-key pool block),
// O_soft += P_soft V, O_lin += P_lin V and O_lin = phi(Q) H_c, all bf16 x bf16 -> fp32 in
// TMEM (M = 128: TMEM lane = query row).  Two threads per query row (warps w and w + 4
// share TMEM lanes) each take half of a block's keys: they read S and L from TMEM, apply
// the masks (each key's visible rows are precomputed once per block as three row bounds)
// and an online maximum m that is raised lazily (O_soft is rescaled in TMEM only when the
// block maximum exceeds m by more than 2^12), and write the bf16 weights to shared memory
// for the P V products.  Before their half, warps 4-7 start the cp.async gathers of the
// next block's keys into the other half of a two-stage buffer (the pool keys are
// scattered: the cache positions come from the snapshot).  One commit per block covers
// that block's P V products and the next block's S, L.
#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace tc;

constexpr int kThreadsTc = 256;          // two threads per query row (warps w and w + 4)
constexpr int kTM = 128;                 // query rows per tile (MMA M)
constexpr int kBN = 64;                  // pool keys per block (MMA N of S, L; K of P V)
constexpr int kD = 128;                  // d_k = d_v = D
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale2 = 12.0f;       // lazy rescale threshold (log2 units)
constexpr uint64_t kWaitNs = 1000000000ull;  // an MMA group that has not completed in 1 s is an error

// shared-memory map (bytes from a 1024-aligned base).  Key blocks are double-buffered;
// stage 1's K and phi(K) tiles reuse the H_c tile once phi(Q) H_c has been issued (the
// first wait covers it).
constexpr int SQ = 0;                    // Q tile      K-major, 2 atoms x [128 x 64]
constexpr int SPQ = 32768;               // phi(Q) tile K-major
constexpr int SH = 98304;                // H_c         MN-major [K = D x N = d_v]
// stage st: K block K-major, 2 atoms x [64 x 64]; phi(K) block; V block MN-major [64 x d_v]
__device__ __forceinline__ uint32_t SK(int st) { return st ? 98304u : 65536u; }
__device__ __forceinline__ uint32_t SPK(int st) { return st ? 114688u : 81920u; }
__device__ __forceinline__ uint32_t SV(int st) { return st ? 147456u : 131072u; }
constexpr int SPS = 163840;              // soft weights K-major [128 x 64]
constexpr int SPL = 180224;              // linear weights
constexpr int SEND = 196608;
// TMEM columns
constexpr uint32_t TS = 0, TL = 64, TOS = 128, TOL = 256;

struct TcArgs {
    int n, eta, lam, chunk, nck, read_mask;
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    __nv_bfloat16* Y;
    const __nv_bfloat16* phiQb;  // [BH][n][D] bf16
    const __nv_bfloat16* phiKb;
    const int32_t* wstep;
    const __nv_bfloat16* snapHb; // [BH][nck][D][DV] bf16
    const float* snapS;
    const int32_t* snapC;
    char* state;                 // per-head status words (timeouts)
    int64_t head_bytes;
    int* abort_flag;             // set by any CTA whose wait timed out; later CTAs skip their work
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void producers_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kThreadsTc, 1) output_tc_kernel(const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_base;
    __shared__ int kpos[2][kBN];
    __shared__ __align__(16) uint32_t kinfo[2][kBN];   // per key: soft rows [lo, hi), linear rows >= llo
    __shared__ float sS[kD];
    __shared__ float bmx[2][kTM];        // the two half-block maxima of each row
    __shared__ float lsum[2][2][kTM];    // [soft, linear][half][row] partial denominators

    const int tid = threadIdx.x, warp = tid / 32;
    const int bh = blockIdx.y;
    const int n = a.n;
    const int t0 = blockIdx.x * kTM, t1 = min(n, t0 + kTM);
    const int c = t0 / a.chunk, c0 = c * a.chunk;
    const int wlo = max(0, c0 - a.eta);
    const int P = a.lam + (t1 - wlo);
    const int nblk = (P + kBN - 1) / kBN;
    const int64_t row0 = (int64_t)bh * n;
    const int32_t* cpos = a.snapC + ((int64_t)bh * a.nck + c) * a.lam;
    const int32_t* wst = a.wstep + row0;

    if (tid == 0) mbar_init(smem_u32(&mbar), 1);
    if (warp == 0) tmem_alloc<512>(smem_u32(&tmem_base));

    // ---- producers (warps 4-7): the keys of block bb and their rows into stage st ----
    const int ptid = tid - 128;
    auto gather = [&](int bb, int st) {
        if (ptid < kBN) {
            const int u = bb * kBN + ptid;
            int p = -1;
            if (u < P) p = u < a.lam ? cpos[u] : wlo + (u - a.lam);
            const int w = p >= 0 ? wst[p] : -1;
            // row r = t - t0 sees key p exactly iff lo <= r < hi, linearly iff r >= llo
            const int lo = p < 0 ? 255 : min(max(p - t0, 0), 255);
            int hi = p < 0 ? 0 : (w < 0 ? 255 : min(max(w - t0, 0), 255));
            // the read mask's HIDE_CACHE: only while the key is in the window (t < p + eta)
            if (p >= 0 && (a.read_mask & LOLA_READ_HIDE_CACHE)) hi = min(hi, min(max(p + a.eta - t0, 0), 255));
            const int llo = (p < 0 || w < c0) ? 255 : min(max(w - t0, 0), 255);
            kpos[st][ptid] = p;
            kinfo[st][ptid] = (uint32_t)lo | ((uint32_t)hi << 8) | ((uint32_t)llo << 16);
        }
        producers_sync();
        for (int i = ptid; i < kBN * 16; i += 128) {
            const int r = i >> 4, c16 = i & 15;
            const int p = kpos[st][r];
            const uint32_t off = (c16 >> 3) * 8192 + kmaj_chunk(r, c16 & 7);
            const uint32_t voff = mnmaj_chunk(r, c16 * 8, kBN);
            if (p >= 0) {
                cp_async16(sb + SK(st) + off, a.K + (row0 + p) * kD + c16 * 8);
                cp_async16(sb + SPK(st) + off, a.phiKb + (row0 + p) * kD + c16 * 8);
                cp_async16(sb + SV(st) + voff, a.V + (row0 + p) * kD + c16 * 8);
            } else {
                *reinterpret_cast<uint4*>(sm + SK(st) + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + SPK(st) + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + SV(st) + voff) = make_uint4(0, 0, 0, 0);
            }
        }
    };

    // ---- stage Q, phi(Q) (rows t0 .. t0 + 127; beyond n: zero), H_c, s_c; block 0 ----
    for (int i = tid; i < kTM * 16; i += kThreadsTc) {
        const int r = i >> 4, c16 = i & 15;
        const uint32_t off = (c16 >> 3) * 16384 + kmaj_chunk(r, c16 & 7);
        const int t = t0 + r;
        if (t < n) {
            cp_async16(sb + SQ + off, a.Q + (row0 + t) * kD + c16 * 8);
            cp_async16(sb + SPQ + off, a.phiQb + (row0 + t) * kD + c16 * 8);
        } else {
            *reinterpret_cast<uint4*>(sm + SQ + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sm + SPQ + off) = make_uint4(0, 0, 0, 0);
        }
    }
    {
        const __nv_bfloat16* sh = a.snapHb + ((int64_t)bh * a.nck + c) * kD * kD;
        for (int i = tid; i < kD * (kD / 8); i += kThreadsTc) {
            const int k = i / (kD / 8), n8 = (i % (kD / 8)) * 8;
            cp_async16(sb + SH + mnmaj_chunk(k, n8, kD), sh + k * kD + n8);
        }
    }
    if (tid < kD) sS[tid] = a.snapS[((int64_t)bh * a.nck + c) * kD + tid];
    if (warp >= 4) gather(0, 0);
    cp_async_wait_all();
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();

    // per-row state: thread tid owns query row t0 + (tid & 127) and key half hf = tid >> 7
    // (pool keys 32 hf .. 32 hf + 31 of every block, output columns 64 hf .. 64 hf + 63);
    // scores in log2 units
    const int row = tid & (kTM - 1), hf = tid >> 7;
    const int t = t0 + row;
    const float c2 = kLog2e / sqrtf((float)kD);
    float m_run = -INFINITY, l_soft = 0.f, l_lin = 0.f;
    if (hf == 0) {
        // phi(q_t)^T s_c from the bf16 phi(Q) tile, in feature order
        float acc = 0.f;
#pragma unroll
        for (int c16 = 0; c16 < 16; ++c16) {
            const uint4 x = *reinterpret_cast<const uint4*>(sm + SPQ + (c16 >> 3) * 16384 + kmaj_chunk(row, c16 & 7));
            const uint32_t wds[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fmaf(__uint_as_float(wds[q] << 16), sS[c16 * 8 + 2 * q], acc);
                acc = fmaf(__uint_as_float(wds[q] & 0xffff0000u), sS[c16 * 8 + 2 * q + 1], acc);
            }
        }
        l_lin = acc;
    }
    const uint32_t tb = tmem_base;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t mb = smem_u32(&mbar);
    uint32_t phase = 0;
    bool bad = __syncthreads_or(*reinterpret_cast<volatile int*>(a.abort_flag) != 0) != 0;

    // O_lin = phi(Q) H_c, then S, L of block 0
    auto issue_sl = [&](int st) {
        constexpr uint32_t id = idesc_bf16(kTM, kBN, 0);
        for (int k = 0; k < kD / 16; ++k) {
            const uint32_t ao = (k >> 2) * 16384 + (k & 3) * 32, bo = (k >> 2) * 8192 + (k & 3) * 32;
            mma_bf16(tb + TS, sdesc(sb + SQ + ao, 16, 1024), sdesc(sb + SK(st) + bo, 16, 1024), id, k > 0);
            mma_bf16(tb + TL, sdesc(sb + SPQ + ao, 16, 1024), sdesc(sb + SPK(st) + bo, 16, 1024), id, k > 0);
        }
    };
    if (tid == 0 && !bad) {
        constexpr uint32_t id = idesc_bf16(kTM, kD, 1);
        for (int k = 0; k < kD / 16; ++k) {
            const uint64_t ad = sdesc(sb + SPQ + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc(sb + SH + k * 2048, 16384, 1024);
            mma_bf16(tb + TOL, ad, bd, id, k > 0);
        }
        issue_sl(0);
        mma_commit(mb);
    }

    for (int b = 0; b < nblk && !bad; ++b) {
        const int st = b & 1;
        // S, L of block b (and the previous P V, and phi(Q) H_c) have completed
        const bool ok = mbar_wait(mb, phase, kWaitNs);
        phase ^= 1;
        fence_after();
        const bool prod = warp >= 4 && b + 1 < nblk;
        if (prod) gather(b + 1, st ^ 1);   // copies land while this block is weighted
        {
            // ---- masks, block maximum, weights for keys 32 hf .. 32 hf + 31 ----
            const uint32_t* ki = kinfo[st] + 32 * hf;
            float sv[32];
            uint32_t vis = 0u;
            float bm = -INFINITY;
            tmem_ld32(tb + lane_off + TS + 32 * hf, sv);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const uint32_t info = ki[jj];
                const bool vs = row >= (int)(info & 255u) && row < (int)((info >> 8) & 255u);
                vis |= (uint32_t)vs << jj;
                bm = vs ? fmaxf(bm, sv[jj]) : bm;
            }
            bmx[hf][row] = bm;
            __syncthreads();
            bm = fmaxf(bmx[0][row], bmx[1][row]) * c2;
            // lazy rescale of O_soft (columns 64 hf ..); both threads of a row take the same
            // decision; TMEM accesses stay warp-uniform (factor 1 for the rows that keep m)
            const bool first = bm > m_run && m_run == -INFINITY;
            const bool need = bm > m_run && m_run != -INFINITY && bm - m_run > kRescale2;
            if (first) m_run = bm;
            if (__any_sync(0xffffffffu, need)) {
                const float f = need ? ex2(m_run - bm) : 1.f;
                l_soft *= f;
                float o[32];
#pragma unroll
                for (int cc = 0; cc < kD / 2; cc += 32) {
                    tmem_ld32(tb + lane_off + TOS + 64 * hf + cc, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= f;
                    tmem_st32(tb + lane_off + TOS + 64 * hf + cc, o);
                }
                tmem_wait_st();
                if (need) m_run = bm;
            }
            const float mr = m_run;
            float lv[32];
            tmem_ld32(tb + lane_off + TL + 32 * hf, lv);
            tmem_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t ps[4], pl[4];
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    float e[2], g[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int jj = c4 * 8 + 2 * hh + u;
                        const bool vs = (vis >> jj) & 1u;
                        const bool vl = row >= (int)((ki[jj] >> 16) & 255u);
                        e[u] = vs ? ex2(fmaf(sv[jj], c2, -mr)) : 0.f;
                        g[u] = vl ? lv[jj] : 0.f;
                    }
                    const __nv_bfloat162 bs = __floats2bfloat162_rn(e[0], e[1]);
                    const __nv_bfloat162 bl = __floats2bfloat162_rn(g[0], g[1]);
                    const float2 fs = __bfloat1622float2(bs), fl = __bfloat1622float2(bl);
                    l_soft += fs.x + fs.y;
                    l_lin += fl.x + fl.y;
                    ps[hh] = *reinterpret_cast<const uint32_t*>(&bs);
                    pl[hh] = *reinterpret_cast<const uint32_t*>(&bl);
                }
                const int c16 = 4 * hf + c4;
                *reinterpret_cast<uint4*>(sm + SPS + kmaj_chunk(row, c16)) = make_uint4(ps[0], ps[1], ps[2], ps[3]);
                *reinterpret_cast<uint4*>(sm + SPL + kmaj_chunk(row, c16)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            fence_async_smem();
        }
        if (prod) {
            cp_async_wait_all();
            fence_async_smem();
        }
        fence_before();
        bad = __syncthreads_or(!ok) != 0;
        fence_after();
        if (bad) break;
        // ---- O_soft += P_soft V, O_lin += P_lin V; then S, L of the next block ----
        if (tid == 0) {
            constexpr uint32_t id = idesc_bf16(kTM, kD, 1);
            for (int k = 0; k < kBN / 16; ++k) {
                const uint64_t vd = sdesc(sb + SV(st) + k * 2048, 8192, 1024);
                mma_bf16(tb + TOS, sdesc(sb + SPS + k * 32, 16, 1024), vd, id, (b > 0 || k > 0));
                mma_bf16(tb + TOL, sdesc(sb + SPL + k * 32, 16, 1024), vd, id, 1);
            }
            if (b + 1 < nblk) issue_sl(st ^ 1);
            mma_commit(mb);
        }
    }
    if (!bad) {
        const bool ok = mbar_wait(mb, phase, kWaitNs);
        fence_after();
        bad = __syncthreads_or(!ok) != 0;
    }
    // ---- epilogue: y = (O_soft + 2^{-m} O_lin) / (l_soft + 2^{-m} l_lin); thread (row, hf)
    //      writes output columns 64 hf .. 64 hf + 63 ----
    lsum[0][hf][row] = l_soft;
    lsum[1][hf][row] = l_lin;
    __syncthreads();
    if (!bad) {
        const float ls = lsum[0][0][row] + lsum[0][1][row], ll = lsum[1][0][row] + lsum[1][1][row];
        const bool any = m_run != -INFINITY;
        // HIDE_STATE: the linear terms stay out of the read (then the window's current token
        // makes any true)
        const float em = any ? ((a.read_mask & LOLA_READ_HIDE_STATE) ? 0.f : ex2(-m_run)) : 1.f;
        const float den = any ? fmaf(em, ll, ls) : ll;
        const float inv = t < n ? 1.0f / den : 0.f;
        __nv_bfloat16* y = a.Y + (row0 + (t < n ? t : 0)) * kD + 64 * hf;
        for (int cc = 0; cc < kD / 2; cc += 32) {
            float os[32], ol[32];
            tmem_ld32(tb + lane_off + TOS + 64 * hf + cc, os);
            tmem_ld32(tb + lane_off + TOL + 64 * hf + cc, ol);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float y0 = (any ? fmaf(em, ol[j], os[j]) : ol[j]) * inv;
                const float y1 = (any ? fmaf(em, ol[j + 1], os[j + 1]) : ol[j + 1]) * inv;
                const __nv_bfloat162 bv = __floats2bfloat162_rn(y0, y1);
                pk[j / 2] = *reinterpret_cast<const uint32_t*>(&bv);
            }
            if (t < n) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(y + cc + 8 * q) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
    }
    if (bad && tid == 0) {
        atomicOr(reinterpret_cast<int32_t*>(a.state + (int64_t)bh * a.head_bytes) + HDR_STATUS, (int)ST_TIMEOUT);
        atomicExch(a.abort_flag, 1);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc<512>(tb);
}

}  // namespace

bool output_tc_supported(const Dims& d) { return d.dtype == LOLA_BF16 && d.D == kD && d.dk == kD && d.dv == kD; }

cudaError_t launch_output_tc(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K, const void* V,
                             void* Y, char* state, int64_t head_bytes, cudaStream_t st) {
    TcArgs a;
    a.n = n;
    a.eta = d.eta;
    a.lam = d.lam;
    a.chunk = ws.snap_interval;
    a.nck = ws.nck;
    a.read_mask = d.read_mask;
    a.Q = static_cast<const __nv_bfloat16*>(Q);
    a.K = static_cast<const __nv_bfloat16*>(K);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.phiQb = ws.phiQb;
    a.phiKb = ws.phiKb;
    a.wstep = ws.wstep;
    a.snapHb = ws.snapHb;
    a.snapS = ws.snapS;
    a.snapC = ws.snapC;
    a.state = state;
    a.head_bytes = head_bytes;
    a.abort_flag = ws.abort_flag;
    const size_t smem = SEND + 1024;
    cudaError_t e = cudaFuncSetAttribute(output_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    output_tc_kernel<<<dim3((n + kTM - 1) / kTM, d.BH), kThreadsTc, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace lola
