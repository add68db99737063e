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
//   K7a hola_prep_kernel     every row's q^, k^ (split into bf16 hi + lo, in the state path's
//                            chunk tiles) and q~, k~ (bf16), one warp per row;
//   K7b hola_state_tc_kernel the state path in chunked form on tcgen05 (lola_hola_tc.cu);
//   K7c hola_cache_kernel    the persistent cache at every chunk start from the fixed scores, one
//                            CTA per head: per chunk, the w best of the cache and the chunk's
//                            tokens by (higher score, older position), ranked by counting among
//                            the cache and the tokens that beat a full cache's w-th key;
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
// K7a: one warp per row; lane l holds entries 4l .. 4l + 3.  Rows are walked over whole 64-token
// chunks, so the rows past n write the zero rows of the last chunk tile.
// ---------------------------------------------------------------------------------------
constexpr int kPrepRows = 8;   // rows per CTA (one per warp)
constexpr int kTileRows = 64;  // tokens per chunk tile
__global__ void __launch_bounds__(kPrepRows * kWarp) hola_prep_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                      const __nv_bfloat16* __restrict__ K,
                                                                      const float* __restrict__ gq,
                                                                      const float* __restrict__ gk, int n, int nck,
                                                                      int64_t rows, uint8_t* __restrict__ xtile,
                                                                      __nv_bfloat16* __restrict__ qt,
                                                                      __nv_bfloat16* __restrict__ kt) {
    const int lane = threadIdx.x % kWarp;
    const int64_t r = (int64_t)blockIdx.x * kPrepRows + threadIdx.x / kWarp;
    if (r >= rows) return;
    const int64_t per = (int64_t)nck * kTileRows;
    const int64_t bh = r / per;
    const int t = (int)(r - bh * per);
    uint8_t* tile = xtile + (bh * nck + t / kTileRows) * (int64_t)kHolaXTile;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        float u[4] = {0.f, 0.f, 0.f, 0.f};
        if (t < n) {
            const __nv_bfloat16* X = which ? K : Q;
            const float* g = which ? gk : gq;
            const int64_t src = (bh * n + t) * kHD + 4 * lane;
            const uint2 raw = *reinterpret_cast<const uint2*>(X + src);
            const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
            float ss = x[0] * x[0];
#pragma unroll
            for (int i = 1; i < 4; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
            const float il2 = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;          // a zero row stays zero
            const float irms = 1.0f / sqrtf(ss / (float)kHD + kRmsEps);
            const float4 gg = *reinterpret_cast<const float4*>(g + 4 * lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = x[i] * il2;
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(gg.x * (x[0] * irms), gg.y * (x[1] * irms));
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(gg.z * (x[2] * irms), gg.w * (x[3] * irms));
            *reinterpret_cast<uint2*>((which ? kt : qt) + src) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
        }
        // the unit row, split: hi = bf16(u), lo = bf16(u - hi); keys at tile rows 0-63, queries 64-127
        uint32_t hw[2], lw[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(u[2 * i]), h1 = __float2bfloat16_rn(u[2 * i + 1]);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(u[2 * i] - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(u[2 * i + 1] - __bfloat162float(h1));
            hw[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lw[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        const int tr = (t % kTileRows) + (which ? 0 : kTileRows);
        *reinterpret_cast<uint2*>(tile + hola_xtile_off(tr, 4 * lane, 0)) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(tile + hola_xtile_off(tr, 4 * lane, 1)) = make_uint2(lw[0], lw[1]);
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
    __shared__ int wsum[kCacheThreads / kWarp + 1];
    const int tid = threadIdx.x, bh = blockIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const float* sc = scores + (int64_t)bh * n;
    int32_t* out = cache + (int64_t)bh * nck * w;
    int count = 0;
    for (int c = 0; c < nck; ++c) {
        for (int i = tid; i < w; i += kCacheThreads)
            out[(int64_t)c * w + i] = i < count ? (int32_t)(0xffffffffu - (uint32_t)(hk[i] & 0xffffffffu)) : -1;
        if (c == nck - 1) break;
        const int c0 = c * chunk, m = min(chunk, n - c0);
        // A full cache keeps its w-th best key unless a new key beats it (keys are unique: score
        // bits, then the inverted position), so only the chunk's tokens above that key compete.
        const uint64_t floor_key = count == w && w > 0 ? hk[w - 1] : 0ull;
        for (int i = tid; i < count; i += kCacheThreads) ck[i] = hk[i];
        int N = count;
        for (int base = 0; base < m; base += kCacheThreads) {
            const int i = base + tid;
            const uint64_t key = i < m ? cache_key(sc[c0 + i], c0 + i) : 0ull;
            const bool in = i < m && key > floor_key;
            const unsigned bal = __ballot_sync(0xffffffffu, in);
            if (lane == 0) wsum[warp] = __popc(bal);
            __syncthreads();
            int off = N;
            for (int q = 0; q < warp; ++q) off += wsum[q];
            int tot = 0;
            for (int q = 0; q < kCacheThreads / kWarp; ++q) tot += wsum[q];
            if (in) ck[off + __popc(bal & ((1u << lane) - 1u))] = key;
            N += tot;
            __syncthreads();
        }
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

cudaError_t launch_hola_prep(int BH, int n, const void* Q, const void* K, const float* gq, const float* gk,
                             uint8_t* xtile, __nv_bfloat16* qt, __nv_bfloat16* kt, cudaStream_t st) {
    const int nck = (n + kTileRows - 1) / kTileRows;
    const int64_t rows = (int64_t)BH * nck * kTileRows;
    const int64_t grid = (rows + kPrepRows - 1) / kPrepRows;
    hola_prep_kernel<<<(unsigned)grid, kPrepRows * kWarp, 0, st>>>(static_cast<const __nv_bfloat16*>(Q),
                                                                   static_cast<const __nv_bfloat16*>(K), gq, gk, n, nck,
                                                                   rows, xtile, qt, kt);
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
