// K7b: the gated delta-rule state path of the write-magnitude cache layer in its chunked
// form, on tcgen05.
//
// "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes, sections 3.1 and
// 3.5: e_t = v_t - alpha_t S_{t-1}^T k^_t, S_t = alpha_t S_{t-1} + beta_t k^_t e_t^T, read-out
// S_t^T q^_t, score m_t = beta_t ||e_t||.
//
// A pass covers tokens [s0, s1) of a 64-token chunk and starts from S = R_0 (the decay before
// it folded into R).  With c_t = alpha_{s0} ... alpha_t and u'_t = beta_t e_t / c_t, the
// recurrence unrolls exactly into
//   (I + A') U' = W',   A'_tj = beta_t (k^_t . k^_j)  (j < t),
//                       W'_t  = beta_t (v_t / c_t - R_0^T k^_t),
//   y_t  = c_t (R_0^T q^_t + sum_{j <= t} (q^_t . k^_j) u'_j),
//   R_end = R_0 + sum_j k^_j u'_j^T,   m_t = c_t ||u'_t||,   S_end = c_{s1-1} R_end
// (S_t = c_t R_t with R_t = R_0 + sum_{j <= t} k^_j u'_j^T).  A pass ends before the token whose
// c_t would fall below 2^-100, so 1 / c_t stays far inside float32; with the notes' decays
// (close to 1) every chunk is one pass.
//
// The state is kept transposed in TMEM (lane = value column c, columns = key index), so every
// product comes out with the value column on the lane and the solve needs no transposition:
//   P1  D1 = R_0^T [K^; Q^]^T   (128 x 128: columns 0-63 the keys' predictions, 64-127 the
//                                queries' read-outs)       and   GM = [K^; Q^] K^^T (128 x 64);
//   the solve: thread c holds column c of W' in registers; the substitution runs in four blocks
//   of 16 rows -- a diagonal block right-looking from registers with its A' entries read from
//   shared memory (broadcast, float32), the rows below it updated by the split product
//   TZ[:, 16 b ..] += U'_b^T A'_b^T (tcgen05, TMEM on the same lanes) -- so a thread loads the
//   480 entries of the diagonal blocks instead of all 2,016 of A';
//   P3  D1[:, 64..] += U'^T A_read^T (the chunk's read-out; A_read = masked Q^ K^^T)  and
//       R^T += U'^T K^ (the state update; K^ read from the same tile as X, MN-major).
// Float32 operands are split into bf16 hi + lo; each product is hi.hi + hi.lo + lo.hi with
// float32 accumulation.  The unit rows arrive pre-split in the tile layout the descriptors read
// (written by the row kernel, 64 KB per chunk, one bulk copy, two chunks in flight); the chunk's
// value rows by a bulk copy one chunk ahead; X K^^T of the next chunk is issued by a second
// thread as soon as the current chunk's last products are.  One CTA of 256 threads per head.
#include <utility>

#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace tc;

constexpr int kD = 128;          // d_k = d_v
constexpr int kC = 64;           // tokens per chunk
constexpr int kThr = 256;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr float kMinC = 0x1p-100f;   // a pass ends before its decay falls below this

// TMEM columns (128 lanes, lane = value column c): R^T, D1 = R_0^T X^T, GM = X K^^T (lane = X row)
constexpr uint32_t TRT = 0, TD1 = 128, TGM = 256;
constexpr uint32_t TZ = 320;   // the substitution's off-diagonal sums: lane c, column t - 16 (t = 16 .. 63)

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t SX = 0;                     // two chunk tiles X = [K^; Q^] (hi, lo), kHolaXTile each
constexpr uint32_t SRT = 2 * kHolaXTile;       // R_0^T hi, lo: K-major 128 x 128 (32 KB each)
constexpr uint32_t kRTB = 32768;
constexpr uint32_t SU = SRT;                   // (after P1, over R_0^T) U'^T hi, lo: K-major 128 x 64
constexpr uint32_t kUB = 16384;
constexpr uint32_t SAR = SRT + 32768;          // (after P1) A_read hi, lo: K-major 64 x 64
constexpr uint32_t kARB = 8192;
constexpr uint32_t SAB = SRT + 49152;          // (after P1) A' hi, lo: K-major 64 x 64 (row t, K = j)
constexpr uint32_t kABB = 8192;
constexpr uint32_t SAm = SRT + 2 * kRTB;       // A''s four diagonal 16 x 16 blocks, float32, [block][j][t]
constexpr uint32_t SVEC = SAm + 4 * 16 * 16 * 4;   // per-pass vectors (float32 [64] each): see the kernel
constexpr uint32_t SV = SAm + 4 * kC * kC;     // the chunk's value rows, bf16 [64][128]
constexpr uint32_t SEND = SV + 2 * kC * kD;
static_assert(SEND + 1024 + 2048 <= 232448, "shared memory plan exceeds 227 KB");
static_assert(SVEC + 4 * kC * 8 <= SV, "per-pass vectors overlap the value rows");

struct TcStateArgs {
    int n, nck;                 // tokens, 64-token chunks
    const uint8_t* xtile;       // [BH][nck][kHolaXTile]
    const __nv_bfloat16* V;     // [BH][n][d]
    const float* alpha;         // [BH][n]
    const float* beta;
    float* ystate;              // [BH][n][d]
    float* scores;              // [BH][n]
    float* S_out;               // [BH][d][d] or null
    int32_t* status;            // [BH][4] (word 3)
};

__device__ __forceinline__ void split2(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}
// 8 float32 values as two 16-byte chunks of bf16 (hi, lo)
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat16 h0, l0, h1, l1;
        split2(v[2 * i], h0, l0);
        split2(v[2 * i + 1], h1, l1);
        h[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        l[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}
// instruction descriptor with an MN-major A as well
__host__ __device__ constexpr uint32_t idesc_ab(int M, int N, int a_mn, int b_mn) {
    return idesc_bf16(M, N, b_mn) | ((uint32_t)a_mn << 15);
}
// D (+)= A B over `ksteps` K-steps of 16, with split operands: hi.hi + hi.lo + lo.hi.  ad/bd give
// the descriptor of term (0: hi, 1: lo) at K-step k.
template <typename FA, typename FB>
__device__ __forceinline__ void mma_split(uint32_t d, uint32_t idesc, int ksteps, bool accumulate, FA ad, FB bd) {
    const int ta[3] = {0, 0, 1}, tb[3] = {0, 1, 0};
#pragma unroll
    for (int p = 0; p < 3; ++p)
        for (int k = 0; k < ksteps; ++k)
            mma_bf16(d, ad(ta[p], k), bd(tb[p], k), idesc, (accumulate || p > 0 || k > 0) ? 1 : 0);
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// The substitution (I + A') u = w in four blocks of 16 rows.  A diagonal block is solved from
// registers (right-looking, the block of A' transposed in shared memory:
// Am[256 B' + 16 (j - 16 B') + (t - 16 B')] = A'_tj, four rows per load); the rows below take the
// block's u through a split product on tcgen05 (see the kernel).
template <int B>
__device__ __forceinline__ void solve_diag(float (&acc)[kC], const float* Am) {
#pragma unroll
    for (int j = 16 * B; j < 16 * B + 15; ++j) {
        const float uj = acc[j];
#pragma unroll
        for (int t4 = (j + 1) & ~3; t4 < 16 * B + 16; t4 += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(Am + 256 * B + 16 * (j - 16 * B) + (t4 - 16 * B));
            if (t4 + 0 > j) acc[t4 + 0] = fmaf(-a4.x, uj, acc[t4 + 0]);
            if (t4 + 1 > j) acc[t4 + 1] = fmaf(-a4.y, uj, acc[t4 + 1]);
            if (t4 + 2 > j) acc[t4 + 2] = fmaf(-a4.z, uj, acc[t4 + 2]);
            if (t4 + 3 > j) acc[t4 + 3] = fmaf(-a4.w, uj, acc[t4 + 3]);
        }
    }
}
// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective)
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// the solve warps (0-3) only
__device__ __forceinline__ void solve_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// a load the compiler keeps where it is written (issued a chunk before its use)
__device__ __forceinline__ float ld_early(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// The sums over the warp's lanes of 64 per-lane values: after five halving exchanges lane l
// holds the sums for tokens T(l) and T(l) + 1, T(l) = 32 b4 + 16 b3 + 8 b2 + 4 b1 + 2 b0 (b the
// bits of l).  v is consumed.
__device__ __forceinline__ void token_sums(float (&v)[kC], int lane) {
#pragma unroll
    for (int o = 16, cnt = kC; o > 0; o >>= 1, cnt >>= 1) {
        const bool up = lane & o;
        const int h = cnt / 2;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[h + i];
            const float keep = up ? v[h + i] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
}
__device__ __forceinline__ int token_of_lane(int lane) {
    return 32 * ((lane >> 4) & 1) + 16 * ((lane >> 3) & 1) + 8 * ((lane >> 2) & 1) + 4 * ((lane >> 1) & 1) +
           2 * (lane & 1);
}

__global__ void __launch_bounds__(kThr, 1) hola_state_tc_kernel(const TcStateArgs a) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float* Am = reinterpret_cast<float*>(sm + SAm);
    const __nv_bfloat16* Vs = reinterpret_cast<const __nv_bfloat16*>(sm + SV);
    // mbarriers: 0 MMA commits (thread 0), 1-2 the X tiles, 3 value rows, 4 solve products,
    // 5 X K^T (thread 128)
    __shared__ __align__(8) uint64_t bars[6];
    __shared__ uint32_t tmem_base;
    __shared__ int pass_end, gm_bad;
    // per-pass vectors: c_t by pass parity (the read-outs of a pass are stored during the next
    // pass's first phase), 1 / c_t, beta_t (1, 1, 0 outside the pass), and the per-warp partial
    // sums of ||u_t||^2
    float (*cs2)[kC] = reinterpret_cast<float (*)[kC]>(sm + SVEC);
    float* ics = reinterpret_cast<float*>(sm + SVEC + 2 * 4 * kC);
    float* bs = reinterpret_cast<float*>(sm + SVEC + 3 * 4 * kC);
    float (*sp)[kC] = reinterpret_cast<float (*)[kC]>(sm + SVEC + 4 * 4 * kC);
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x, n = a.n, nck = a.nck;
    const uint8_t* xg = a.xtile + (int64_t)bh * nck * kHolaXTile;
    const __nv_bfloat16* V = a.V + (int64_t)bh * n * kD;
    const float* al = a.alpha + (int64_t)bh * n;
    const float* be = a.beta + (int64_t)bh * n;
    float* ys = a.ystate + (int64_t)bh * n * kD;
    float* scores = a.scores + (int64_t)bh * n;
    const uint32_t bar_mma = smem_u32(&bars[0]), bar_v = smem_u32(&bars[3]);
    const uint32_t bar_x0 = smem_u32(&bars[1]), bar_z = smem_u32(&bars[4]), bar_gm = smem_u32(&bars[5]);
    constexpr int kGmThread = 128;   // issues X K^T (a lane of warp 4, which reads it first)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;   // this warp's TMEM lane quarter
    const int row = (warp & 3) * 32 + lane;                         // its TMEM lane
    const int half = warp >> 2;

    // bulk loads and products in flight (for the abort path): thread 0 issues the loads, D1, the
    // solve products and P3; thread kGmThread X K^T; each waits once on every phase it needs
    int x_issued[2] = {0, 0}, x_done[2] = {0, 0}, v_issued = 0, v_done = 0;
    bool mma_pending = false, z_pending = false, gm_pending = false;
    if (tid == 0) {
        mbar_init(bar_mma, 1);
        mbar_init(bar_x0, 1);
        mbar_init(bar_x0 + 8, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_z, 1);
        mbar_init(bar_gm, 1);
        gm_bad = 0;
        for (int c = 0; c < 2 && c < nck; ++c) {
            mbar_expect(bar_x0 + 8 * c, kHolaXTile);
            bulk_load(sb + SX + c * kHolaXTile, xg + (int64_t)c * kHolaXTile, kHolaXTile, bar_x0 + 8 * c);
            ++x_issued[c];
        }
        const uint32_t vb = (uint32_t)min(kC, n) * kD * 2;
        mbar_expect(bar_v, vb);
        bulk_load(sb + SV, V, vb, bar_v);
        ++v_issued;
    }
    if (warp == 0) tmem_alloc<512>(smem_u32(&tmem_base));
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_base;
    {   // R = 0
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 32) tmem_st32(tb + lane_base + TRT + 64 * half + c, z);
        tmem_wait_st();
    }
    // warp 0: this chunk's and the next chunk's alpha, beta at tokens 2 lane, 2 lane + 1
    float na0 = 1.f, na1 = 1.f, nb0 = 0.f, nb1 = 0.f;
    auto fetch_ab = [&](int c0) {
        const int t0 = c0 + 2 * lane;
        na0 = t0 < n ? ld_early(al + t0) : 1.f;
        na1 = t0 + 1 < n ? ld_early(al + t0 + 1) : 1.f;
        nb0 = t0 < n ? ld_early(be + t0) : 0.f;
        nb1 = t0 + 1 < n ? ld_early(be + t0 + 1) : 0.f;
    };
    if (warp == 0) fetch_ab(0);
    // GM = X K^^T of a chunk needs only its tile: thread kGmThread issues it as soon as the tile is
    // in (for chunk i + 1 right after chunk i's last products) and commits it to bar_gm; the
    // warps that read GM wait there (chunk i: parity i & 1).  A tile that never lands sets gm_bad
    // and completes the phase without products.
    int gx_done[2] = {0, 0};
    auto issue_gm = [&](int c) {
        const int bb = c & 1;
        const uint32_t sxc = sb + SX + bb * kHolaXTile;
        if (mbar_wait(bar_x0 + 8 * bb, (uint32_t)(gx_done[bb] & 1), kWaitNs)) {
            ++gx_done[bb];
            mma_split(tb + TGM, idesc_ab(128, 64, 0, 0), kD / 16, false,
                      [&](int h, int k) { return sdesc(sxc + h * 32768 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); },
                      [&](int h, int k) { return sdesc(sxc + h * 32768 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); });
            mma_commit(bar_gm);
            gm_pending = true;
        } else {
            gm_bad = 1;
            mbar_arrive1(bar_gm);
        }
    };
    if (tid == kGmThread) issue_gm(0);
    uint32_t ph_mma = 0, ph_z = 0;
    float G = 1.f;          // the decay not yet folded into R
    bool bad = false;       // uniform: set after a barrier reports a failed wait
    // the read-outs of a pass are stored while the next pass splits R_0: y_t = c_t D1[c][64 + t]
    // (warp w: tokens 32 (w >> 2) + 0..31 of the pass [y_s0, y_s1) of the chunk at y_c0)
    int pb = 0, y_c0 = -1, y_s0 = 0, y_s1 = 0;
    auto store_readouts = [&]() {
        float x[32];
        tmem_ld32(tb + lane_base + TD1 + 64 + 32 * half, x);
        tmem_wait_ld();
        float* y = ys + (int64_t)y_c0 * kD + row;
        const float* cp = cs2[pb ^ 1];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int t = 32 * half + j;
            if (t >= y_s0 && t < y_s1) y[(int64_t)t * kD] = cp[t] * x[j];
        }
    };
    for (int i = 0; i < nck && !bad; ++i) {
        const int c0 = i * kC, m = min(kC, n - c0), b = i & 1;
        const uint32_t sx = sb + SX + b * kHolaXTile;
        float ca0 = 1.f, ca1 = 1.f, cb0 = 0.f, cb1 = 0.f;
        if (warp == 0) {
            ca0 = na0; ca1 = na1; cb0 = nb0; cb1 = nb1;
            if (i + 1 < nck) fetch_ab(c0 + kC);
        }
        // thread 0 reads the tile in D1 and P3: it waits for it too (normally long landed)
        bool xfail = false;
        if (tid == 0) {
            if (mbar_wait(bar_x0 + 8 * b, (uint32_t)(x_done[b] & 1), kWaitNs)) ++x_done[b];
            else xfail = true;
        }
        for (int s0 = 0; s0 < m && !bad;) {
            // ---- the pass's decays (warp 0): c_t from s0, the pass ends before c_t < 2^-100 ----
            if (warp == 0) {
                const int t0 = 2 * lane, t1 = t0 + 1;
                const bool in0 = t0 >= s0 && t0 < m, in1 = t1 >= s0 && t1 < m;
                const float a0 = in0 ? fmaxf(ca0, kMinC) : 1.f, a1 = in1 ? fmaxf(ca1, kMinC) : 1.f;
                const float p = a0 * a1;
                float incl = p;
#pragma unroll
                for (int o = 1; o < kWarp; o <<= 1) {
                    const float x = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl *= x;
                }
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 1.f;
                const float c0v = excl * a0, c1v = excl * p;
                const unsigned f0 = __ballot_sync(0xffffffffu, in0 && c0v < kMinC);
                const unsigned f1 = __ballot_sync(0xffffffffu, in1 && c1v < kMinC);
                int s1 = m;
                if (f0) s1 = min(s1, 2 * (__ffs(f0) - 1));
                if (f1) s1 = min(s1, 2 * (__ffs(f1) - 1) + 1);
                const bool on0 = in0 && t0 < s1, on1 = in1 && t1 < s1;
                cs2[pb][t0] = on0 ? c0v : 1.f;
                cs2[pb][t1] = on1 ? c1v : 1.f;
                ics[t0] = on0 ? 1.0f / c0v : 1.f;
                ics[t1] = on1 ? 1.0f / c1v : 1.f;
                bs[t0] = on0 ? cb0 : 0.f;
                bs[t1] = on1 ? cb1 : 0.f;
                if (lane == 0) pass_end = s1;
            }
            // ---- R_0 = G R (written back when G != 1), split into R_0^T hi, lo (K-major) ----
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                float x[32];
                tmem_ld32(tb + lane_base + TRT + 64 * half + cc, x);
                tmem_wait_ld();
                if (G != 1.f) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= G;
                    tmem_st32(tb + lane_base + TRT + 64 * half + cc, x);
                }
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 hi, lo;
                    split8(x + j, hi, lo);
                    const uint32_t off = (uint32_t)half * 16384u + kmaj_chunk(row, (cc + j) >> 3);
                    *reinterpret_cast<uint4*>(sm + SRT + off) = hi;
                    *reinterpret_cast<uint4*>(sm + SRT + kRTB + off) = lo;
                }
            }
            if (G != 1.f) tmem_wait_st();
            G = 1.f;
            if (y_c0 >= 0) store_readouts();   // the previous pass's (D1 is rewritten after the barrier)
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            const int s1 = pass_end;
            const bool last = s1 >= m;
            const float* cs = cs2[pb];
            if (tid == 0) xfail = xfail || gm_bad;
            // ---- P1: D1 = R_0^T X^T (GM was issued with the tile) ----
            if (tid == 0) {
                if (!xfail) {
                    mma_split(tb + TD1, idesc_ab(128, 128, 0, 0), kD / 16, false,
                              [&](int h, int k) { return sdesc(sb + SRT + h * kRTB + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); },
                              [&](int h, int k) { return sdesc(sx + h * 32768 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); });
                    mma_commit(bar_mma);
                    mma_pending = true;
                } else {
                    mbar_arrive1(bar_mma);   // nothing issued: complete the phase so no thread waits
                }
            }
            {
                const bool ok = mbar_wait(bar_mma, ph_mma, kWaitNs) && !xfail;
                if (tid == 0 && ok) mma_pending = false;
                ph_mma ^= 1u;
                fence_after();
                if (!__syncthreads_and(ok)) {
                    bad = true;
                    break;
                }
            }
            // ---- A' (warps 4, 5: key rows), A_read (warps 6, 7: query rows), W' (warps 0-3) ----
            float acc[kC];
            bool vok = true;
            bool gok = true;
            if (warp >= 4) {   // GM of this chunk (issued a chunk ahead)
                gok = mbar_wait(bar_gm, (uint32_t)(i & 1), kWaitNs);
                if (tid == kGmThread && gok) gm_pending = false;
                fence_after();
            }
            if (warp >= 4 && warp < 6) {
                // A'_tj = beta_t (k^_t . k^_j) for j < t: the diagonal blocks transposed
                const int t = row;
                const float bt = bs[t];
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    float x[32];
                    tmem_ld32(tb + lane_base + TGM + cc, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        x[j] = cc + j < t ? bt * x[j] : 0.f;
                        if (((cc + j) >> 4) == (t >> 4)) Am[256 * (t >> 4) + 16 * ((cc + j) & 15) + (t & 15)] = x[j];
                    }
                    // and row-major, split (K-major, row t): the B operand of the block products
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 hi, lo;
                        split8(x + j, hi, lo);
                        const uint32_t off = kmaj_chunk(t, (cc + j) >> 3);
                        *reinterpret_cast<uint4*>(sm + SAB + off) = hi;
                        *reinterpret_cast<uint4*>(sm + SAB + kABB + off) = lo;
                    }
                }
            } else if (warp >= 6) {
                // A_read_tj = q^_t . k^_j for j <= t, split (K-major, row t)
                const int t = row - 64;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    float x[32];
                    tmem_ld32(tb + lane_base + TGM + cc, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        float v8[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) v8[q] = cc + j + q <= t ? x[j + q] : 0.f;
                        uint4 hi, lo;
                        split8(v8, hi, lo);
                        const uint32_t off = kmaj_chunk(t, (cc + j) >> 3);
                        *reinterpret_cast<uint4*>(sm + SAR + off) = hi;
                        *reinterpret_cast<uint4*>(sm + SAR + kARB + off) = lo;
                    }
                }
            } else {
                // W'_t = beta_t (v_t / c_t - R_0^T k^_t) for column c = row, tokens of the pass only
                vok = mbar_wait(bar_v, (uint32_t)(i & 1), kWaitNs);
                const int c = row;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    float x[32];
                    tmem_ld32(tb + lane_base + TD1 + cc, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int t = cc + j;
                        const float v = __bfloat162float(Vs[t * kD + c]);
                        acc[t] = (t >= s0 && t < s1) ? bs[t] * fmaf(v, ics[t], -x[j]) : 0.f;
                    }
                }
            }
            fence_async_smem();   // A' and A_read tiles are read by the tensor core
            if (!__syncthreads_and(vok && gok)) {
                bad = true;
                break;
            }
            if (tid == 0 && s0 == 0) ++v_done;   // (thread 0 waited for the rows and got them)
            // ---- U' by blocks of 16 rows (warps 0-3): block b solved from registers and split into
            //      U'^T (K-major, row c); the rows below it take TZ[:, 16 b ..] (+)= U'_b^T A'_b^T
            //      (M = 128, N = 48 - 16 b, K = 16) on tcgen05, read back before their own block ----
            bool zok = true;
            if (warp < 4) {
                auto block_done = [&](auto bc) {
                    constexpr int B = decltype(bc)::value;
                    solve_diag<B>(acc, Am);
#pragma unroll
                    for (int t = 16 * B; t < 16 * B + 16; t += 8) {
                        uint4 hi, lo;
                        split8(acc + t, hi, lo);
                        const uint32_t off = kmaj_chunk(row, t >> 3);
                        *reinterpret_cast<uint4*>(sm + SU + off) = hi;
                        *reinterpret_cast<uint4*>(sm + SU + kUB + off) = lo;
                    }
                    if constexpr (B < 3) {
                        fence_async_smem();
                        fence_before();
                        solve_sync();
                        fence_after();
                        if (tid == 0) {
                            mma_split(tb + TZ + 16 * B, idesc_ab(128, 48 - 16 * B, 0, 0), 1, B > 0,
                                      [&](int h, int k) { return sdesc(sb + SU + h * kUB + 32 * B, 16, 1024); },
                                      [&](int h, int k) {
                                          return sdesc(sb + SAB + h * kABB + 2048 * (B + 1) + 32 * B, 16, 1024);
                                      });
                            mma_commit(bar_z);
                        }
                        zok = mbar_wait(bar_z, ph_z, kWaitNs) && zok;
                        ph_z ^= 1u;
                        fence_after();
                        float z[16];
                        tmem_ld16f(tb + lane_base + TZ + 16 * B, z);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 16; ++q) acc[16 * (B + 1) + q] -= z[q];
                    }
                };
                block_done(std::integral_constant<int, 0>{});
                block_done(std::integral_constant<int, 1>{});
                block_done(std::integral_constant<int, 2>{});
                block_done(std::integral_constant<int, 3>{});
                // ||u_t||^2 = ||c_t u'_t||^2 (scaled before squaring: u' alone may be near 2^100)
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    const float ut = cs[t] * acc[t];
                    acc[t] = ut * ut;
                }
                token_sums(acc, lane);
                const int t = token_of_lane(lane);
                sp[warp][t] = acc[0];
                sp[warp][t + 1] = acc[1];
            }
            if (tid == 0 && !zok) z_pending = true;
            fence_async_smem();
            fence_before();
            if (!__syncthreads_and(zok)) {
                bad = true;
                break;
            }
            fence_after();
            // ---- P3: D1[:, 64..] += U'^T A_read^T, R^T += U'^T K^ ----
            if (tid == 0) {
                mma_split(tb + TD1 + 64, idesc_ab(128, 64, 0, 0), kC / 16, true,
                          [&](int h, int k) { return sdesc(sb + SU + h * kUB + k * 32, 16, 1024); },
                          [&](int h, int k) { return sdesc(sb + SAR + h * kARB + k * 32, 16, 1024); });
                mma_split(tb + TRT, idesc_ab(128, 128, 0, 1), kC / 16, true,
                          [&](int h, int k) { return sdesc(sb + SU + h * kUB + k * 32, 16, 1024); },
                          [&](int h, int k) { return sdesc(sx + h * 32768 + k * 2048, 16384, 1024); });
                mma_commit(bar_mma);
                mma_pending = true;
                if (last && i + 1 < nck) {
                    // the value rows were read before the last barrier: bring in the next chunk's
                    const int mn = min(kC, n - c0 - kC);
                    fence_async_smem();
                    mbar_expect(bar_v, (uint32_t)mn * kD * 2);
                    bulk_load(sb + SV, V + (int64_t)(c0 + kC) * kD, (uint32_t)mn * kD * 2, bar_v);
                    ++v_issued;
                }
            }
            if (tid == kGmThread && last && i + 1 < nck) issue_gm(i + 1);
            // scores m_t = ||c_t u'_t|| of the pass's tokens
            if (tid < kC && tid >= s0 && tid < s1)
                scores[c0 + tid] = sqrtf((sp[0][tid] + sp[1][tid]) + (sp[2][tid] + sp[3][tid]));
            {
                const bool ok = mbar_wait(bar_mma, ph_mma, kWaitNs);
                if (tid == 0 && ok) mma_pending = false;
                ph_mma ^= 1u;
                fence_after();
                if (!__syncthreads_and(ok)) {
                    bad = true;
                    break;
                }
            }
            if (tid == 0 && last && i + 2 < nck) {
                // P3 has read this tile: bring in chunk i + 2
                mbar_expect(bar_x0 + 8 * b, kHolaXTile);
                bulk_load(sx, xg + (int64_t)(i + 2) * kHolaXTile, kHolaXTile, bar_x0 + 8 * b);
                ++x_issued[b];
            }
            G = cs[s1 - 1];
            y_c0 = c0;
            y_s0 = s0;
            y_s1 = s1;
            pb ^= 1;
            s0 = s1;
        }
    }
    if (!bad) store_readouts();
    if (bad) {
        if (tid == 0) {
            atomicOr(a.status + 4 * bh + HDR_STATUS, (int)ST_TIMEOUT);
            // nothing asynchronous may still be writing TMEM or shared memory when the CTA ends
            if (mma_pending) mbar_wait(bar_mma, ph_mma ^ 1u, 20ull * kWaitNs);
            if (z_pending) mbar_wait(bar_z, ph_z ^ 1u, 20ull * kWaitNs);
            for (int c = 0; c < 2; ++c)
                if (x_issued[c] > x_done[c]) mbar_wait(bar_x0 + 8 * c, (uint32_t)(x_done[c] & 1), 20ull * kWaitNs);
            if (v_issued > v_done) mbar_wait(bar_v, (uint32_t)(v_done & 1), 20ull * kWaitNs);
        }
        if (tid == kGmThread && gm_pending) mbar_wait(bar_gm, (uint32_t)((gx_done[0] + gx_done[1] - 1) & 1), 20ull * kWaitNs);
    } else if (a.S_out) {
        // S = G R: thread (c, half) writes S[k][c] for its 64 keys k
        float* So = a.S_out + (int64_t)bh * kD * kD + (int64_t)(64 * half) * kD + row;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 32) {
            float x[32];
            tmem_ld32(tb + lane_base + TRT + 64 * half + cc, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) So[(int64_t)(cc + j) * kD] = G * x[j];
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc<512>(tb);
}

}  // namespace

cudaError_t launch_hola_state_tc(int BH, int n, const uint8_t* xtile, const void* V, const float* alpha,
                                 const float* beta, float* ystate, float* scores, float* S_out, int32_t* status,
                                 cudaStream_t st) {
    TcStateArgs a;
    a.n = n;
    a.nck = (n + kC - 1) / kC;
    a.xtile = xtile;
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.alpha = alpha;
    a.beta = beta;
    a.ystate = ystate;
    a.scores = scores;
    a.S_out = S_out;
    a.status = status;
    const size_t smem = SEND + 1024;
    cudaError_t e = cudaFuncSetAttribute(hola_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    hola_state_tc_kernel<<<BH, kThr, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace lola
