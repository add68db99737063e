// K7b (tensor cores): the gated delta-rule state path of the write-magnitude cache layer in
// its chunked form.
//
// "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes, sections 3.1 and
// 3.5: e_t = v_t - alpha_t S_{t-1}^T k^_t, S_t = alpha_t S_{t-1} + beta_t k^_t e_t^T, read-out
// S_t^T q^_t, score m_t = beta_t ||e_t||.  With u_t = beta_t e_t, the decay kept as a scalar
// (S_t = G_t R_t, G_t = alpha_0 ... alpha_t) and, inside a chunk of 64 tokens starting from R_0
// and G (the decay before it), c_t = the product of the chunk's alphas up to t and
// g_t = G c_t, the recurrence unrolls exactly into
//   (I + A) U = W,  A_tj = beta_t (c_t / c_j) (k^_t . k^_j)  (j < t),
//                   W_t  = beta_t (v_t - g_t R_0^T k^_t),
//   o_t  = g_t R_0^T q^_t + sum_{j <= t} (c_t / c_j) (q^_t . k^_j) u_j,
//   R_end = R_0 + sum_j (k^_j / g_j) u_j^T,   m_t = ||u_t||.
// The dense products -- [K^; Q^] R_0, [K^; Q^] K^^T, the read-out's (c-masked QK^T) U and the
// state update K'^T U -- run on tcgen05 with every float32 operand split into two bf16 terms
// (hi + lo; three partial products hi.hi + hi.lo + lo.hi, float32 accumulation); the triangular
// solve for U runs on CUDA cores (one column per thread, forward substitution in float32).
// R lives in TMEM for the whole sequence.  One CTA of 256 threads per head.
#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace tc;

constexpr int kD = 128;          // d_k = d_v
constexpr int kC = 64;           // tokens per chunk
constexpr int kThr = 256;
constexpr uint64_t kWaitNs = 1000000000ull;

// TMEM columns (128 lanes): R [d_k x d_v], P = [K^; Q^] R_0, G = [K^; Q^] K^^T, O = read-out
constexpr uint32_t TR = 0, TP = 128, TG = 256, TO = 320;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t SX = 0;                 // [K^; Q^] hi, lo: K-major 128 x 128, 2 atoms each (32 KB)
constexpr uint32_t kXB = 32768;
constexpr uint32_t SR = 65536;             // R_0 hi, lo: MN-major [K = 128 x N = 128] (32 KB each)
constexpr uint32_t kRB = 32768;
constexpr uint32_t SA = 65536;             // (after P1, over SR) read-out A hi, lo: K-major 128 x 64 (16 KB each)
constexpr uint32_t kAB = 16384;
constexpr uint32_t SU = 98304;             // (after P1, over SR) U hi, lo: MN-major [K = 64 x N = 128] (16 KB each)
constexpr uint32_t kUB = 16384;
constexpr uint32_t SK = 131072;            // K' = k^ / g hi, lo: MN-major A [K = 64 x M = 128] (16 KB each)
constexpr uint32_t kKB = 16384;
constexpr uint32_t SW = 163840;            // W, then U, then g_t Q R_0 rows: float32 [64][128]
constexpr uint32_t SAm = SW + 4 * kC * kD; // A: float32 [64][64]
constexpr uint32_t SEND = SAm + 4 * kC * kC;

struct TcStateArgs {
    int n;
    const float* qh;            // [BH][n][d] unit rows
    const float* kh;
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

__global__ void __launch_bounds__(kThr, 1) hola_state_tc_kernel(const TcStateArgs a) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float* Wm = reinterpret_cast<float*>(sm + SW);
    float* Am = reinterpret_cast<float*>(sm + SAm);
    __shared__ __align__(8) uint64_t mbar;
    __shared__ uint32_t tmem_base;
    __shared__ float cs[kC], gs[kC], bs[kC];
    __shared__ int fail;
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x, n = a.n;
    const float* qh = a.qh + (int64_t)bh * n * kD;
    const float* kh = a.kh + (int64_t)bh * n * kD;
    const __nv_bfloat16* V = a.V + (int64_t)bh * n * kD;
    const float* al = a.alpha + (int64_t)bh * n;
    const float* be = a.beta + (int64_t)bh * n;
    float* ys = a.ystate + (int64_t)bh * n * kD;
    float* scores = a.scores + (int64_t)bh * n;
    const uint32_t bar = smem_u32(&mbar);
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;   // this warp's TMEM lane quarter
    const int row = (warp & 3) * 32 + lane;                         // its TMEM lane
    const int chalf = warp >> 2;                                     // warps 4-7: the second half of the columns

    if (tid == 0) {
        mbar_init(bar, 1);
        fail = 0;
    }
    if (warp == 0) tmem_alloc<512>(smem_u32(&tmem_base));
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_base;
    // R = 0
    {
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 32) tmem_st32(tb + lane_base + TR + 64 * chalf + c, z);
        tmem_wait_st();
    }
    uint32_t phase = 0;
    float G = 1.f;
    auto wait_mma = [&]() -> bool {
        const bool ok = __syncthreads_and(mbar_wait(bar, phase, kWaitNs));
        phase ^= 1u;
        fence_after();
        return ok;
    };

    for (int c0 = 0; c0 < n && !fail; c0 += kC) {
        const int m = min(kC, n - c0);
        // ---- P0: the chunk's decays (prefix products of alpha; padding tokens: alpha 1, beta 0) ----
        if (warp == 0) {
            const int t0 = 2 * lane, t1 = 2 * lane + 1;
            const float a0 = t0 < m ? al[c0 + t0] : 1.f, a1 = t1 < m ? al[c0 + t1] : 1.f;
            float p = a0 * a1, incl = p;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const float x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl *= x;
            }
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 1.f;
            cs[t0] = excl * a0;
            cs[t1] = excl * p;
            gs[t0] = G * (excl * a0);
            gs[t1] = G * (excl * p);
            bs[t0] = t0 < m ? be[c0 + t0] : 0.f;
            bs[t1] = t1 < m ? be[c0 + t1] : 0.f;
        }
        __syncthreads();
        // ---- P0: X = [K^; Q^] (rows 0-63 keys, 64-127 queries) and K' = K^ / g, split ----
        for (int i = tid; i < 128 * 16; i += kThr) {
            const int r = i >> 4, c8 = i & 15, t = r & 63;
            float v[8];
            if (t < m) {
                const float* src = (r < 64 ? kh : qh) + (int64_t)(c0 + t) * kD + 8 * c8;
                const float4 x0 = *reinterpret_cast<const float4*>(src), x1 = *reinterpret_cast<const float4*>(src + 4);
                v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = 0.f;
            }
            uint4 hi, lo;
            split8(v, hi, lo);
            const uint32_t off = (uint32_t)(c8 >> 3) * 16384u + kmaj_chunk(r, c8 & 7);
            *reinterpret_cast<uint4*>(sm + SX + off) = hi;
            *reinterpret_cast<uint4*>(sm + SX + kXB + off) = lo;
            if (r < 64) {
                const float ig = 1.0f / gs[t];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] *= ig;
                split8(v, hi, lo);
                const uint32_t ko = mnmaj_chunk(t, 8 * c8, kC);
                *reinterpret_cast<uint4*>(sm + SK + ko) = hi;
                *reinterpret_cast<uint4*>(sm + SK + kKB + ko) = lo;
            }
        }
        // R_0 from TMEM (lane = row of R, warps 4-7 the second half of the columns), split, MN-major
        {
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                float x[32];
                tmem_ld32(tb + lane_base + TR + 64 * chalf + cc, x);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 hi, lo;
                    split8(x + j, hi, lo);
                    const uint32_t ro = mnmaj_chunk(row, 64 * chalf + cc + j, kD);
                    *reinterpret_cast<uint4*>(sm + SR + ro) = hi;
                    *reinterpret_cast<uint4*>(sm + SR + kRB + ro) = lo;
                }
            }
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
        fence_after();
        // ---- P1: P = X R_0 (128 x 128), Gm = X K^^T (128 x 64) ----
        if (tid == 0) {
            mma_split(tb + TP, idesc_ab(128, 128, 0, 1), kD / 16, false,
                      [&](int h, int k) { return sdesc(sb + SX + h * kXB + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); },
                      [&](int h, int k) { return sdesc(sb + SR + h * kRB + k * 2048, 16384, 1024); });
            mma_split(tb + TG, idesc_ab(128, 64, 0, 0), kD / 16, false,
                      [&](int h, int k) { return sdesc(sb + SX + h * kXB + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); },
                      [&](int h, int k) { return sdesc(sb + SX + h * kXB + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024); });
            mma_commit(bar);
        }
        if (!wait_mma()) {
            if (tid == 0) fail = 1;
            break;
        }
        // ---- P2: W, A (key rows: warps 0, 1 and 4, 5), the read-out's A (query rows: warps 2, 3) ----
        if ((warp & 3) < 2) {
            const int t = row;   // 0 .. 63
            const float bt = bs[t], gt = gs[t], ct = cs[t];
            // W_t = beta_t (v_t - g_t R_0^T k^_t): this warp's half of the columns
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                float x[32];
                tmem_ld32(tb + lane_base + TP + 64 * chalf + cc, x);
                tmem_wait_ld();
                const int col0 = 64 * chalf + cc;
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    float v8[8];
                    if (t < m) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(V + (int64_t)(c0 + t) * kD + col0 + j);
                        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            v8[2 * q] = __uint_as_float(w4[q] << 16);
                            v8[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) v8[q] = 0.f;
                    }
                    float4* dst = reinterpret_cast<float4*>(Wm + t * kD + col0 + j);
                    dst[0] = make_float4(bt * fmaf(-gt, x[j], v8[0]), bt * fmaf(-gt, x[j + 1], v8[1]),
                                         bt * fmaf(-gt, x[j + 2], v8[2]), bt * fmaf(-gt, x[j + 3], v8[3]));
                    dst[1] = make_float4(bt * fmaf(-gt, x[j + 4], v8[4]), bt * fmaf(-gt, x[j + 5], v8[5]),
                                         bt * fmaf(-gt, x[j + 6], v8[6]), bt * fmaf(-gt, x[j + 7], v8[7]));
                }
            }
            // A_tj = beta_t (c_t / c_j) (k^_t . k^_j), j < t: this warp's half of the 64 keys
            {
                float x[32];
                tmem_ld32(tb + lane_base + TG + 32 * chalf, x);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int jj = 32 * chalf + j;
                    Am[t * kC + jj] = jj < t ? bt * (ct / cs[jj]) * x[j] : 0.f;
                }
            }
        } else {
            // query rows: the read-out's A_tj = (c_t / c_j) (q^_t . k^_j), j <= t, split (rows 64+ stay 0)
            const int t = row - 64;
            const float ct = cs[t];
            float x[32];
            tmem_ld32(tb + lane_base + TG + 32 * chalf, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                float v8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int jj = 32 * chalf + j + q;
                    v8[q] = jj <= t ? (ct / cs[jj]) * x[j + q] : 0.f;
                }
                uint4 hi, lo;
                split8(v8, hi, lo);
                const uint32_t off = kmaj_chunk(t, (32 * chalf + j) >> 3);
                *reinterpret_cast<uint4*>(sm + SA + off) = hi;
                *reinterpret_cast<uint4*>(sm + SA + kAB + off) = lo;
            }
            // rows 64 .. 127 of the read-out's A are zero (the MMA is M = 128)
            const int r2 = row;   // 64 .. 127
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t off = kmaj_chunk(r2, 4 * chalf + j);
                *reinterpret_cast<uint4*>(sm + SA + off) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + SA + kAB + off) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncthreads();
        // ---- P2b: U = (I + A)^{-1} W by forward substitution, one column per thread ----
        if (tid < kD) {
            const int c = tid;
            float u[kC];
#pragma unroll
            for (int t = 0; t < kC; ++t) {
                float acc = Wm[t * kD + c];
#pragma unroll
                for (int j = 0; j < t; ++j) acc = fmaf(-Am[t * kC + j], u[j], acc);
                u[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < kC; ++t) {
                Wm[t * kD + c] = u[t];
                __nv_bfloat16 h, l;
                split2(u[t], h, l);
                const uint32_t off = mnmaj_chunk(t, c, kC) + 2 * (c & 7);
                *reinterpret_cast<__nv_bfloat16*>(sm + SU + off) = h;
                *reinterpret_cast<__nv_bfloat16*>(sm + SU + kUB + off) = l;
            }
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
        fence_after();
        // ---- P3: O = A_read U (128 x 128; rows 0-63 used), R += K'^T U ----
        if (tid == 0) {
            mma_split(tb + TO, idesc_ab(128, 128, 0, 1), kC / 16, false,
                      [&](int h, int k) { return sdesc(sb + SA + h * kAB + k * 32, 16, 1024); },
                      [&](int h, int k) { return sdesc(sb + SU + h * kUB + k * 2048, 8192, 1024); });
            mma_split(tb + TR, idesc_ab(128, 128, 1, 1), kC / 16, true,
                      [&](int h, int k) { return sdesc(sb + SK + h * kKB + k * 2048, 8192, 1024); },
                      [&](int h, int k) { return sdesc(sb + SU + h * kUB + k * 2048, 8192, 1024); });
            mma_commit(bar);
        }
        // scores m_t = ||u_t|| (warps 4-7: two lanes per token... 16 tokens per warp, 2 lanes each)
        if (warp >= 4) {
            const int t = (warp - 4) * 16 + (lane >> 1), h = lane & 1;
            float s = 0.f;
            for (int c = 64 * h; c < 64 * h + 64; ++c) s = fmaf(Wm[t * kD + c], Wm[t * kD + c], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            if (h == 0 && t < m) scores[c0 + t] = sqrtf(s);
        }
        if (!wait_mma()) {
            if (tid == 0) fail = 1;
            break;
        }
        // ---- P4: the read-outs y_t = O_t + g_t R_0^T q^_t ----
        if ((warp & 3) >= 2) {
            const int t = row - 64;
            const float gt = gs[t];
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                float x[32];
                tmem_ld32(tb + lane_base + TP + 64 * chalf + cc, x);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(Wm + t * kD + 64 * chalf + cc + j) =
                        make_float4(gt * x[j], gt * x[j + 1], gt * x[j + 2], gt * x[j + 3]);
            }
        }
        __syncthreads();
        if ((warp & 3) < 2) {
            const int t = row;
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                float x[32];
                tmem_ld32(tb + lane_base + TO + 64 * chalf + cc, x);
                tmem_wait_ld();
                if (t < m) {
                    float* y = ys + (int64_t)(c0 + t) * kD + 64 * chalf + cc;
                    const float* qr = Wm + t * kD + 64 * chalf + cc;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(y + j) =
                            make_float4(x[j] + qr[j], x[j + 1] + qr[j + 1], x[j + 2] + qr[j + 2], x[j + 3] + qr[j + 3]);
                }
            }
        }
        // ---- the decay after the chunk; fold it into R when it gets small ----
        G = gs[kC - 1];
        if (G < 0x1p-40f) {
            float x[32];
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                tmem_ld32(tb + lane_base + TR + 64 * chalf + cc, x);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] *= G;
                tmem_st32(tb + lane_base + TR + 64 * chalf + cc, x);
            }
            tmem_wait_st();
            G = 1.f;
        }
        fence_before();
        __syncthreads();
        fence_after();
    }
    if (fail) {
        if (tid == 0) atomicOr(a.status + 4 * bh + HDR_STATUS, (int)ST_TIMEOUT);
        // no MMA may still be writing TMEM when it is released
        if (tid == 0) mbar_wait(bar, phase, 20ull * kWaitNs);
    } else if (a.S_out) {
        float* So = a.S_out + (int64_t)bh * kD * kD + (int64_t)row * kD + 64 * chalf;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 32) {
            float x[32];
            tmem_ld32(tb + lane_base + TR + 64 * chalf + cc, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(So + cc + j) = make_float4(G * x[j], G * x[j + 1], G * x[j + 2], G * x[j + 3]);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc<512>(tb);
}

}  // namespace

cudaError_t launch_hola_state_tc(int BH, int n, const float* qh, const float* kh, const void* V, const float* alpha,
                                 const float* beta, float* ystate, float* scores, float* S_out, int32_t* status,
                                 cudaStream_t st) {
    TcStateArgs a;
    a.n = n;
    a.qh = qh;
    a.kh = kh;
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
