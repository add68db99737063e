// K7: the write-magnitude exact cache on a gated delta-rule state.
//
// "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes, method sections
// 3.1-3.5.  Per head, with S of shape d_k x d_v (S_{-1} = 0):
//   state path (section 3.1, Eq. 1; the gated form of section 3.5): k^ = k / ||k||,
//     e_t = v_t - alpha_t S_{t-1}^T k^_t,  S_t = alpha_t S_{t-1} + beta_t k^_t e_t^T,
//     read-out S_t^T q^_t (q^ = q / ||q||);
//   write-magnitude score (section 3.3, Eqs. 5-6): m_t = beta_t ||e_t||, fixed at the write;
//   persistent cache (section 3.3): the w best scores so far, changing at chunk starts;
//   cache read (section 3.4, Eq. 7): RMS-scaled q~, k~ (own scales), softmax over the cache,
//     the chunk's tokens up to t and a null sink; y = S_t^T q^_t + gate_h * read.
//
// Four launches:
//   K7a hola_prep_kernel   every row's q^, k^ (float32) and q~, k~ (bf16), one warp per row;
//   K7b hola_state_kernel  the sequential state path, one CTA of 512 threads per head, S in
//                          registers by columns (warp w: columns 8w..8w+7, lane l: rows
//                          4l..4l+3), so a token needs no CTA barrier: the prediction's and the
//                          read-out's column sums are lane reductions, the residual is shuffled
//                          across the warp's columns, the write is local; one barrier per block
//                          of 8 tokens publishes the next block's rows;
//   K7c hola_cache_kernel  the persistent cache at every chunk start from the fixed scores, one
//                          CTA per head: per chunk, the w best of the cache and the chunk's
//                          tokens by (higher score, older position), ranked by counting;
//   K7d the output pass (lola_output_tc.cu) in its cache-read mode: the pool is the chunk's
//       persistent cache plus the chunk's tokens, on tcgen05, with the sink and the gated sum
//       in its epilogue.
#include "lola_chain.cuh"
#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using namespace chain;

constexpr int kHD = 128;             // d_k = d_v
constexpr float kRmsEps = 1e-6f;

// ---------------------------------------------------------------------------------------
// K7a: lane l holds entries 4l .. 4l + 3 of the row
// ---------------------------------------------------------------------------------------
constexpr int kPrepRows = 8;   // rows per CTA (one per warp)
__global__ void __launch_bounds__(kPrepRows * kWarp) hola_prep_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                      const __nv_bfloat16* __restrict__ K,
                                                                      const float* __restrict__ gq,
                                                                      const float* __restrict__ gk, int64_t rows,
                                                                      float* __restrict__ qh, float* __restrict__ kh,
                                                                      __nv_bfloat16* __restrict__ qt,
                                                                      __nv_bfloat16* __restrict__ kt) {
    const int lane = threadIdx.x % kWarp;
    const int64_t r = (int64_t)blockIdx.x * kPrepRows + threadIdx.x / kWarp;
    if (r >= rows) return;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        const __nv_bfloat16* X = which ? K : Q;
        const float* g = which ? gk : gq;
        const uint2 raw = *reinterpret_cast<const uint2*>(X + r * kHD + 4 * lane);
        const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
        float ss = x[0] * x[0];
#pragma unroll
        for (int i = 1; i < 4; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
        const float il2 = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;          // a zero row stays zero
        const float irms = 1.0f / sqrtf(ss / (float)kHD + kRmsEps);
        const float4 gg = *reinterpret_cast<const float4*>(g + 4 * lane);
        *reinterpret_cast<float4*>((which ? kh : qh) + r * kHD + 4 * lane) =
            make_float4(x[0] * il2, x[1] * il2, x[2] * il2, x[3] * il2);
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(gg.x * (x[0] * irms), gg.y * (x[1] * irms));
        const __nv_bfloat162 b1 = __floats2bfloat162_rn(gg.z * (x[2] * irms), gg.w * (x[3] * irms));
        *reinterpret_cast<uint2*>((which ? kt : qt) + r * kHD + 4 * lane) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
    }
}

// ---------------------------------------------------------------------------------------
// K7b
// ---------------------------------------------------------------------------------------
struct StateArgs {
    int n;
    const float* qh;               // [BH][n][d_k] unit rows
    const float* kh;
    const __nv_bfloat16* V;        // [BH][n][d_v]
    const float* alpha;            // [BH][n]
    const float* beta;
    float* ystate;                 // [BH][n][d_v]
    float* scores;                 // [BH][n]
    float* S_out;                  // [BH][d_k][d_v] or null
};

// Warp w owns columns 8w .. 8w+7 of S and lane l its rows 4l .. 4l+3 (32 registers), so a token
// needs no CTA barrier: the column sums of S^T k^ and S^T q^ are lane reductions inside the warp.
// The decay is kept as a scalar: S_t = G_t R_t with G_t = alpha_0 ... alpha_t (renormalised into
// R when it falls below 2^-40), so the write is R += (beta_t / G_t) k^ e^T and the prediction and
// read-out take G times R's products -- equal to the recurrence in exact arithmetic.
// Token rows arrive in blocks of kBlk tokens by cp.async, one block ahead; a CTA barrier per
// block publishes the next block and the score partials of the last one.
constexpr int kBlk = 8;
constexpr int kTRing = 2 * kBlk;   // token row slots: the block in use and the one arriving

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async16g(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The sums over the warp's 32 lanes of 8 per-lane values x[0..7] (one per column): after
// three halving exchanges and two butterflies, lane l holds the sum of column l >> 2.
__device__ __forceinline__ float col_reduce8(const float (&x)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float q[4], r[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? x[i] : x[i + 4];
        q[i] = (b4 ? x[i + 4] : x[i]) + __shfl_xor_sync(kFull, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? q[i] : q[i + 2];
        r[i] = (b3 ? q[i + 2] : q[i]) + __shfl_xor_sync(kFull, send, 8);
    }
    float s = (b2 ? r[1] : r[0]) + __shfl_xor_sync(kFull, b2 ? r[0] : r[1], 4);
    s += __shfl_xor_sync(kFull, s, 2);
    s += __shfl_xor_sync(kFull, s, 1);
    return s;
}

__global__ void __launch_bounds__(kThreads, 1) hola_state_kernel(const StateArgs a) {
    constexpr int kCols = kHD / (kThreads / kWarp);   // 8 columns per warp
    constexpr int kRows = kHD / kWarp;                // 4 rows per lane
    static_assert(kCols == 8 && kRows == 4, "layout");
    __shared__ __align__(16) float kr[kTRing][kHD];
    __shared__ __align__(16) float qr[kTRing][kHD];
    __shared__ __align__(16) __nv_bfloat16 vr[kTRing][kHD];
    __shared__ float ar[kTRing], br[kTRing];
    __shared__ float esq[kTRing][kThreads / kWarp];   // per token and warp: sum of e^2 over the warp's columns
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x, n = a.n;
    const int col = warp * kCols + (lane >> 2);       // the column this lane's reductions end in
    const float* qh = a.qh + (int64_t)bh * n * kHD;
    const float* kh = a.kh + (int64_t)bh * n * kHD;
    const __nv_bfloat16* V = a.V + (int64_t)bh * n * kHD;
    const float* al = a.alpha + (int64_t)bh * n;
    const float* be = a.beta + (int64_t)bh * n;
    float* ys = a.ystate + (int64_t)bh * n * kHD;
    float* scores = a.scores + (int64_t)bh * n;

    // the rows of tokens [t0, t0 + kBlk) into their slots (one commit group per call, every thread)
    auto prefetch_block = [&](int t0) {
        for (int i = tid; i < kBlk * 82; i += kThreads) {
            const int j = i / 82, part = i % 82, t = t0 + j;
            if (t >= n) continue;
            const int sl = t % kTRing;
            if (part < 32) cp_async16g(&kr[sl][4 * part], kh + (int64_t)t * kHD + 4 * part);
            else if (part < 64) cp_async16g(&qr[sl][4 * (part - 32)], qh + (int64_t)t * kHD + 4 * (part - 32));
            else if (part < 80) cp_async16g(&vr[sl][8 * (part - 64)], V + (int64_t)t * kHD + 8 * (part - 64));
            else if (part == 80) cp_async4(&ar[sl], al + t);
            else cp_async4(&br[sl], be + t);
        }
        cp_commit();
    };
    // the scores of tokens [t0, t1) from the warps' partials (beta from global memory: its ring
    // slot may already be receiving the next block)
    auto emit_scores = [&](int t0, int t1) {
        if (tid < t1 - t0) {
            const int t = t0 + tid, sl = t % kTRing;
            float s2 = 0.f;
#pragma unroll
            for (int w = 0; w < kThreads / kWarp; ++w) s2 += esq[sl][w];
            scores[t] = be[t] * sqrtf(s2);
        }
    };

    float S[kRows][kCols];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int c = 0; c < kCols; ++c) S[r][c] = 0.f;
    float qprev[kRows] = {0.f, 0.f, 0.f, 0.f};
    float G = 1.f;   // the decay so far, S = G R (R is held in S[][])

    prefetch_block(0);
    for (int t0 = 0; t0 < n; t0 += kBlk) {
        cp_wait<0>();            // this thread's copies of block t0 have landed
        __syncthreads();         // ... and everyone's; every warp is done with block t0 - kBlk
        if (t0 > 0) emit_scores(t0 - kBlk, t0);
        prefetch_block(t0 + kBlk);   // into block t0 - kBlk's slots
        const int t1 = min(n, t0 + kBlk);
        for (int t = t0; t < t1; ++t) {
            const int sl = t % kTRing;
            const float4 k4 = *reinterpret_cast<const float4*>(&kr[sl][4 * lane]);
            const float kv[kRows] = {k4.x, k4.y, k4.z, k4.w};
            // ---- R^T k^_t (the prediction / G_{t-1}) and R^T q^_{t-1} (the last read-out / G_{t-1}),
            //      column pairs with paired FMAs ----
            float pk[kCols], pq[kCols];
#pragma unroll
            for (int c = 0; c < kCols; c += 2) {
                float2 ak = __fmul2_rn(make_float2(kv[0], kv[0]), make_float2(S[0][c], S[0][c + 1]));
                float2 aq = __fmul2_rn(make_float2(qprev[0], qprev[0]), make_float2(S[0][c], S[0][c + 1]));
#pragma unroll
                for (int r = 1; r < kRows; ++r) {
                    ak = __ffma2_rn(make_float2(kv[r], kv[r]), make_float2(S[r][c], S[r][c + 1]), ak);
                    aq = __ffma2_rn(make_float2(qprev[r], qprev[r]), make_float2(S[r][c], S[r][c + 1]), aq);
                }
                pk[c] = ak.x;
                pk[c + 1] = ak.y;
                pq[c] = aq.x;
                pq[c + 1] = aq.y;
            }
            const float pred = col_reduce8(pk, lane);
            const float outp = col_reduce8(pq, lane);
            if (t >= 1 && (lane & 3) == 0) ys[(int64_t)(t - 1) * kHD + col] = G * outp;
            // ---- the residual of this lane's column, then every column of the warp ----
            const float a_t = ar[sl], b_t = br[sl];
            G *= a_t;                                         // G_t
            const float e_mine = fmaf(-G, pred, __bfloat162float(vr[sl][col]));
            float e[kCols], e2 = 0.f;
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                e[c] = __shfl_sync(kFull, e_mine, 4 * c);
                e2 = fmaf(e[c], e[c], e2);
            }
            if (lane == 0) esq[sl][warp] = e2;
            // ---- the write R += (beta / G) k^ e^T (S = alpha S + beta k^ e^T) ----
            const float bg = b_t / G;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float kb = bg * kv[r];
#pragma unroll
                for (int c = 0; c < kCols; c += 2) {
                    const float2 y = __ffma2_rn(make_float2(kb, kb), make_float2(e[c], e[c + 1]),
                                                make_float2(S[r][c], S[r][c + 1]));
                    S[r][c] = y.x;
                    S[r][c + 1] = y.y;
                }
            }
            if (G < 0x1p-40f) {   // fold the decay back into R (the same G in every thread)
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int c = 0; c < kCols; ++c) S[r][c] *= G;
                G = 1.f;
            }
            const float4 q4 = *reinterpret_cast<const float4*>(&qr[sl][4 * lane]);
            qprev[0] = q4.x;
            qprev[1] = q4.y;
            qprev[2] = q4.z;
            qprev[3] = q4.w;
        }
    }
    // ---- the last token's read-out, the last block's scores, the final state ----
    {
        float pq[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
            pq[c] = qprev[0] * S[0][c];
#pragma unroll
            for (int r = 1; r < kRows; ++r) pq[c] = fmaf(qprev[r], S[r][c], pq[c]);
        }
        const float outp = col_reduce8(pq, lane);
        if ((lane & 3) == 0) ys[(int64_t)(n - 1) * kHD + col] = G * outp;
    }
    cp_wait<0>();
    __syncthreads();
    const int last0 = ((n - 1) / kBlk) * kBlk;
    emit_scores(last0, n);
    if (a.S_out) {
        float* So = a.S_out + (int64_t)bh * kHD * kHD;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            float4* dst = reinterpret_cast<float4*>(So + (int64_t)(4 * lane + r) * kHD + warp * kCols);
            dst[0] = make_float4(G * S[r][0], G * S[r][1], G * S[r][2], G * S[r][3]);
            dst[1] = make_float4(G * S[r][4], G * S[r][5], G * S[r][6], G * S[r][7]);
        }
    }
}

// ---------------------------------------------------------------------------------------
// K7c: one CTA per head walks the chunks; the cache after chunk c is the w best, by (higher
// score, older position), of the cache before it and the chunk's tokens -- each candidate's rank
// is the number of candidates that beat it.  New tokens are always younger than the cached ones,
// so this is the token-by-token rule (a strictly larger score replaces the worst entry) applied a
// chunk at a time.
// ---------------------------------------------------------------------------------------
constexpr int kMaxCache = 128;
constexpr int kMaxChunk = 1024;
constexpr int kCacheThreads = 256;
// rank key: a larger key is better (higher score, then the older position)
__device__ __forceinline__ uint64_t cache_key(float score, int pos) {
    return ((uint64_t)__float_as_uint(score) << 32) | (uint64_t)(0xffffffffu - (uint32_t)pos);
}
__global__ void __launch_bounds__(kCacheThreads) hola_cache_kernel(const float* __restrict__ scores, int n, int w,
                                                                   int chunk, int nck, int32_t* __restrict__ cache) {
    __shared__ uint64_t ck[kMaxCache + kMaxChunk];   // the candidates of one merge
    __shared__ uint64_t hk[kMaxCache];               // the cache, best first
    const int tid = threadIdx.x, bh = blockIdx.x;
    const float* sc = scores + (int64_t)bh * n;
    int32_t* out = cache + (int64_t)bh * nck * w;
    int count = 0;
    for (int c = 0; c < nck; ++c) {
        for (int i = tid; i < w; i += kCacheThreads)
            out[(int64_t)c * w + i] = i < count ? (int32_t)(0xffffffffu - (uint32_t)(hk[i] & 0xffffffffu)) : -1;
        if (c == nck - 1) break;
        const int c0 = c * chunk, m = min(chunk, n - c0), N = count + m;
        for (int i = tid; i < N; i += kCacheThreads) ck[i] = i < count ? hk[i] : cache_key(sc[c0 + i - count], c0 + i - count);
        __syncthreads();
        for (int i = tid; i < N; i += kCacheThreads) {
            const uint64_t ki = ck[i];
            int rank = 0;
#pragma unroll 8
            for (int j = 0; j < N; ++j) rank += ck[j] > ki ? 1 : 0;
            if (rank < w) hk[rank] = ki;
        }
        __syncthreads();
        count = min(w, N);
    }
}

}  // namespace

cudaError_t launch_hola_prep(int64_t rows, const void* Q, const void* K, const float* gq, const float* gk, float* qh,
                             float* kh, __nv_bfloat16* qt, __nv_bfloat16* kt, cudaStream_t st) {
    const int64_t grid = (rows + kPrepRows - 1) / kPrepRows;
    hola_prep_kernel<<<(unsigned)grid, kPrepRows * kWarp, 0, st>>>(static_cast<const __nv_bfloat16*>(Q),
                                                                   static_cast<const __nv_bfloat16*>(K), gq, gk, rows,
                                                                   qh, kh, qt, kt);
    return cudaGetLastError();
}

cudaError_t launch_hola_state(int BH, int n, const float* qh, const float* kh, const void* V, const float* alpha,
                              const float* beta, float* ystate, float* scores, float* S_out, cudaStream_t st) {
    StateArgs a;
    a.n = n;
    a.qh = qh;
    a.kh = kh;
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.alpha = alpha;
    a.beta = beta;
    a.ystate = ystate;
    a.scores = scores;
    a.S_out = S_out;
    hola_state_kernel<<<BH, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_hola_cache(int BH, int n, int w, int chunk, int nck, const float* scores, int32_t* cache,
                              cudaStream_t st) {
    if (w > kMaxCache || chunk > kMaxChunk) return cudaErrorInvalidValue;
    hola_cache_kernel<<<BH, kCacheThreads, 0, st>>>(scores, n, w, chunk, nck, cache);
    return cudaGetLastError();
}

int hola_max_cache() { return kMaxCache; }

}  // namespace lola
