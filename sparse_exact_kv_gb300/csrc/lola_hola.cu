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
//                          registers with the prefill chain's H layout (warp w: rows 8w..8w+7,
//                          lane l: columns 4l..4l+3); per token two CTA barriers: the
//                          prediction's and the previous read-out's row-group partials, then
//                          the residual e (one column per thread), then the rank-one write;
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

constexpr int kSPF = 4;            // token rows prefetched ahead
constexpr int kSRing = 8;          // ring of token rows (> kSPF + 1)

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

__global__ void __launch_bounds__(kThreads, 1) hola_state_kernel(const StateArgs a) {
    using Sh = Shape<kHD, kHD>;
    constexpr int HR = Sh::HR, HC = Sh::HC;
    __shared__ __align__(16) float kr[kSRing][kHD];
    __shared__ __align__(16) float qr[kSRing][kHD];
    __shared__ __align__(16) __nv_bfloat16 vr[kSRing][kHD];
    __shared__ float ar[kSRing], br[kSRing];
    __shared__ __align__(16) float redk[Sh::NRG][kHD];
    __shared__ __align__(16) float redq[Sh::NRG][kHD];
    __shared__ __align__(16) float es[kHD];
    __shared__ float esq[kHD / kWarp];
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x, n = a.n;
    const float* qh = a.qh + (int64_t)bh * n * kHD;
    const float* kh = a.kh + (int64_t)bh * n * kHD;
    const __nv_bfloat16* V = a.V + (int64_t)bh * n * kHD;
    const float* al = a.alpha + (int64_t)bh * n;
    const float* be = a.beta + (int64_t)bh * n;
    float* ys = a.ystate + (int64_t)bh * n * kHD;

    // token `step`'s rows into ring slot step % kSRing (one commit group per call, every thread)
    auto prefetch = [&](int step) {
        if (step < n) {
            const int sl = step % kSRing;
            if (tid < 32) cp_async16g(&kr[sl][4 * tid], kh + (int64_t)step * kHD + 4 * tid);
            else if (tid < 64) cp_async16g(&qr[sl][4 * (tid - 32)], qh + (int64_t)step * kHD + 4 * (tid - 32));
            else if (tid < 80) cp_async16g(&vr[sl][8 * (tid - 64)], V + (int64_t)step * kHD + 8 * (tid - 64));
            else if (tid == 80) cp_async4(&ar[sl], al + step);
            else if (tid == 81) cp_async4(&br[sl], be + step);
        }
        cp_commit();
    };
    float h[HR * HC];
#pragma unroll
    for (int i = 0; i < HR * HC; ++i) h[i] = 0.f;
    for (int st = 0; st < kSPF; ++st) prefetch(st);
    cp_wait<0>();
    __syncthreads();

    for (int t = 0; t < n; ++t) {
        const int sl = t % kSRing, ps = (t + kSRing - 1) % kSRing;
        // ---- the prediction's partials S_{t-1}^T k^_t, and the read-out of token t - 1 ----
        h_partial_store<kHD, kHD>(&redk[0][0], kr[sl], h, warp, lane);
        if (t >= 1) h_partial_store<kHD, kHD>(&redq[0][0], qr[ps], h, warp, lane);
        __syncthreads();
        // ---- the residual (one column per thread of warps 0-3), the read-out's columns ----
        if (tid < kHD) {
            const float pred = reduce_partials_col<kHD, kHD>(&redk[0][0], tid);
            const float v = __bfloat162float(vr[sl][tid]);
            const float e = fmaf(-ar[sl], pred, v);
            es[tid] = e;
            float e2 = e * e;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) e2 += __shfl_xor_sync(kFull, e2, o);
            if (lane == 0) esq[warp] = e2;
        } else if (tid < 2 * kHD && t >= 1) {
            const int c = tid - kHD;
            ys[(int64_t)(t - 1) * kHD + c] = reduce_partials_col<kHD, kHD>(&redq[0][0], c);
        }
        prefetch(t + kSPF);
        cp_wait<kSPF - 1>();   // this thread's copies of token t + 1 have landed
        __syncthreads();
        // ---- the write S = alpha S + beta k^ e^T; the score beta ||e|| ----
        const float a_t = ar[sl], b_t = br[sl];
        float ec[HC];
        h_vec_load<HC>(es + lane * HC, ec);
#pragma unroll
        for (int r4 = 0; r4 < HR / 4; ++r4) {
            const float4 k4 = *reinterpret_cast<const float4*>(&kr[sl][warp * HR + 4 * r4]);
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float kb = b_t * kk[rr];
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    float& x = h[(4 * r4 + rr) * HC + c];
                    x = fmaf(kb, ec[c], a_t * x);
                }
            }
        }
        if (tid == 0) {
            float s2 = 0.f;
#pragma unroll
            for (int w = 0; w < kHD / kWarp; ++w) s2 += esq[w];
            a.scores[(int64_t)bh * n + t] = b_t * sqrtf(s2);
        }
    }
    // ---- the last token's read-out; the final state ----
    h_partial_store<kHD, kHD>(&redq[0][0], qr[(n - 1) % kSRing], h, warp, lane);
    __syncthreads();
    if (tid < kHD) ys[(int64_t)(n - 1) * kHD + tid] = reduce_partials_col<kHD, kHD>(&redq[0][0], tid);
    if (a.S_out) h_store<kHD, kHD>(a.S_out + (int64_t)bh * kHD * kHD, h, warp, lane);
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
__global__ void __launch_bounds__(kCacheThreads) hola_cache_kernel(const float* __restrict__ scores, int n, int w,
                                                                   int chunk, int nck, int32_t* __restrict__ cache) {
    __shared__ float cs[kMaxCache + kMaxChunk];
    __shared__ int cp[kMaxCache + kMaxChunk];
    __shared__ float hs[kMaxCache];
    __shared__ int hp[kMaxCache];
    const int tid = threadIdx.x, bh = blockIdx.x;
    const float* sc = scores + (int64_t)bh * n;
    int32_t* out = cache + (int64_t)bh * nck * w;
    int count = 0;
    for (int c = 0; c < nck; ++c) {
        for (int i = tid; i < w; i += kCacheThreads) out[(int64_t)c * w + i] = i < count ? hp[i] : -1;
        if (c == nck - 1) break;
        const int c0 = c * chunk, m = min(chunk, n - c0), N = count + m;
        for (int i = tid; i < N; i += kCacheThreads) {
            cs[i] = i < count ? hs[i] : sc[c0 + i - count];
            cp[i] = i < count ? hp[i] : c0 + i - count;
        }
        __syncthreads();
        for (int i = tid; i < N; i += kCacheThreads) {
            const float si = cs[i];
            const int pi = cp[i];
            int rank = 0;
            for (int j = 0; j < N; ++j) rank += (cs[j] > si || (cs[j] == si && cp[j] < pi)) ? 1 : 0;
            if (rank < w) {
                hs[rank] = si;
                hp[rank] = pi;
            }
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
