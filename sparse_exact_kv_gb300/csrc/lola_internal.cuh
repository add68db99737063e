// Internal declarations shared by the liblola translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lola.h"

namespace lola {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------------
// Sizes and the public per-head state layout (see lola.h)
// ---------------------------------------------------------------------------------
struct Dims {
    int B, Hh, BH, dk, dv, D, eta, lam, chunk, dtype, read_mask, alloc, score;
    int io_bytes() const { return dtype == LOLA_BF16 ? 2 : 4; }
};

__host__ __device__ inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

struct Layout {
    int64_t head_bytes;
    int64_t H, s, win_pos, win_k, win_v, win_phi, c_pos, c_k, c_v, c_phi, c_N, c_z, ev, tok_phi;
};

inline Layout make_layout(const Dims& d) {
    Layout L;
    int64_t o = 256;  // header
    const int64_t io = d.io_bytes();
    L.H = o;        o = align256(o + 4ll * d.D * d.dv);
    L.s = o;        o = align256(o + 4ll * d.D);
    L.win_pos = o;  o = align256(o + 4ll * d.eta);
    L.win_k = o;    o = align256(o + io * d.eta * d.dk);
    L.win_v = o;    o = align256(o + io * d.eta * d.dv);
    L.win_phi = o;  o = align256(o + 4ll * d.eta * d.D);
    L.c_pos = o;    o = align256(o + 4ll * d.lam);
    L.c_k = o;      o = align256(o + io * d.lam * d.dk);
    L.c_v = o;      o = align256(o + io * d.lam * d.dv);
    L.c_phi = o;    o = align256(o + 4ll * d.lam * d.D);
    L.c_N = o;      o = align256(o + 4ll * d.lam * d.dv);
    L.c_z = o;      o = align256(o + 4ll * d.lam);
    L.ev = o;       o = align256(o + 4ll * (d.dv + 4));
    L.tok_phi = o;  o = align256(o + 4ll * 2 * d.D);
    L.head_bytes = o;
    return L;
}

// header words of a head record
enum { HDR_T = 0, HDR_NCACHE = 1, HDR_NWRITTEN = 2, HDR_STATUS = 3, HDR_WORDS = 16 };

// device-side status bits
enum : int32_t { ST_SLOT_OVERFLOW = 1, ST_BAD_STATE = 2, ST_TIMEOUT = 4 };

// ---------------------------------------------------------------------------------
// Prefill workspace: per-head arrays used between the kernels
// ---------------------------------------------------------------------------------
struct Workspace {
    float* phiK;       // [BH][n][D]    phi(k_t), float32 (selection precision)
    float* phiQ;       // [BH][n][D]    phi(q_t) (float32 output path only)
    __nv_bfloat16* phiKb;  // [BH][n][D] bf16 copies for the tensor-core output kernel (bf16 mode)
    __nv_bfloat16* phiQb;
    int32_t* wstep;    // [BH][n]       step at which token j was written, -1 never
    int32_t* wpos;     // [BH][n]       position written at step t, -1 none
    float* snapH;      // [BH][nck][D*dv]  H before the first step of each chunk (float32 path)
    __nv_bfloat16* snapHb;  // the same in bf16 (tensor-core path: its MMA operand)
    float* snapS;      // [BH][nck][D]
    int32_t* snapC;    // [BH][nck][lam]   cache slot positions before each chunk (-1 empty)
    int32_t* slotpos;  // [BH][lam]        final slot positions (export scratch)
    float* score;      // [BH][n]       query-dependent cache scores (score != LOLA_SCORE_SRE only)
    float* dH;         // [BH][nck][D*dv]  per-interval write sums (score != LOLA_SCORE_SRE only)
    float* dS;         // [BH][nck][D]
    int* abort_flag;   // one int, cleared by every lola_prefill call
    int snap_interval;  // steps between snapshots: max(C, 128), one tensor-core query tile
    int nck;
    size_t bytes;
};

Workspace carve_workspace(const Dims& d, int n, void* base);

// ---------------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------------
template <typename T> struct IO;
template <> struct IO<float> {
    static __device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
    static __device__ __forceinline__ void st(float* p, int64_t i, float x) { p[i] = x; }
};
template <> struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) {
        return __bfloat162float(p[i]);
    }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float x) {
        p[i] = __float2bfloat16_rn(x);
    }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// ---------------------------------------------------------------------------------
// phi(x) = [softmax(W x), softmax(-W x)] for R rows at a time, computed by one warp.
//   xs: the R rows x (d_k floats each, row stride DK) in shared memory;  Ws: W in shared
//   memory with row stride DK + 4 (16-byte aligned rows).  Lane l returns phi[l + 32 m]
//   of row r in out[r][m], m < D / 32.  Each z = W x is summed on four chains (entries
//   c = 0, 1, 2, 3 mod 4, each in increasing c) added as (c0 + c1) + (c2 + c3); the order
//   does not depend on R, so every kernel that needs phi produces identical bits.
// ---------------------------------------------------------------------------------
template <int DK>
__host__ __device__ constexpr int w_stride() { return DK + 4; }

template <int DK, int D, int R>
__device__ __forceinline__ void phi_rows(const float* xs, const float* Ws, int lane, float (&out)[R][D / 32]) {
    constexpr int HM = D / 64;  // z values per lane and row
    float acc[R][HM][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < HM; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[r][m][j] = 0.f;
#pragma unroll 4
    for (int c = 0; c < DK; c += 4) {
        float4 w[HM];
#pragma unroll
        for (int m = 0; m < HM; ++m)
            w[m] = *reinterpret_cast<const float4*>(Ws + (lane + 32 * m) * w_stride<DK>() + c);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4 x = *reinterpret_cast<const float4*>(xs + r * DK + c);
#pragma unroll
            for (int m = 0; m < HM; ++m) {
                acc[r][m][0] = fmaf(w[m].x, x.x, acc[r][m][0]);
                acc[r][m][1] = fmaf(w[m].y, x.y, acc[r][m][1]);
                acc[r][m][2] = fmaf(w[m].z, x.z, acc[r][m][2]);
                acc[r][m][3] = fmaf(w[m].w, x.w, acc[r][m][3]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float z[HM];
#pragma unroll
        for (int m = 0; m < HM; ++m) z[m] = (acc[r][m][0] + acc[r][m][1]) + (acc[r][m][2] + acc[r][m][3]);
        float mx = z[0], mn = z[0];
#pragma unroll
        for (int m = 1; m < HM; ++m) { mx = fmaxf(mx, z[m]); mn = fminf(mn, z[m]); }
        mx = warp_max(mx);
        mn = -warp_max(-mn);
        float ep[HM], en[HM], sp = 0.f, sn = 0.f;
#pragma unroll
        for (int m = 0; m < HM; ++m) {
            ep[m] = expf(z[m] - mx);
            en[m] = expf(mn - z[m]);
            sp += ep[m];
            sn += en[m];
        }
        sp = warp_sum(sp);
        sn = warp_sum(sn);
#pragma unroll
        for (int m = 0; m < HM; ++m) {
            out[r][m] = ep[m] / sp;
            out[r][HM + m] = en[m] / sn;
        }
    }
}

// One row: the same arithmetic as phi_rows.
template <int DK, int D>
__device__ __forceinline__ void phi_warp(const float* xs, const float* Ws, int lane, float (&out)[D / 32]) {
    float o[1][D / 32];
    phi_rows<DK, D, 1>(xs, Ws, lane, o);
#pragma unroll
    for (int m = 0; m < D / 32; ++m) out[m] = o[0][m];
}

// Stage W (D/2 x DK, float32, row-major) into shared memory with row stride DK + 4, all
// loads issued before any store (16-byte loads and stores, fully unrolled).
template <int DK, int D, int NT>
__device__ __forceinline__ void stage_w(float* Ws, const float* W, int tid) {
    constexpr int N4 = (D / 2) * DK / 4;                 // float4 chunks
    constexpr int PER = (N4 + NT - 1) / NT;
    float4 v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int c = tid + i * NT;
        if (c < N4) v[i] = reinterpret_cast<const float4*>(W)[c];
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int c = tid + i * NT;
        if (c < N4) {
            const int r = (4 * c) / DK, k = (4 * c) % DK;
            *reinterpret_cast<float4*>(Ws + r * w_stride<DK>() + k) = v[i];
        }
    }
}

// Records the CUDA error text for lola_last_cuda_error() (the calling thread's) and
// returns LOLA_ERR_CUDA.
int32_t cuda_fail(cudaError_t e, const char* where);

// ---------------------------------------------------------------------------------
// Launchers (each returns the launch's cudaError_t)
// ---------------------------------------------------------------------------------
// phi of every row of X ([BH][n][d_k]) into out (float32) and/or out_bf16 ([BH][n][D]); a wait
// that times out sets ST_TIMEOUT in a head's status word (state, head_bytes) and *abort_flag
cudaError_t launch_phi(const Dims& d, int n, const void* X, const float* W, int64_t w_head_stride,
                       float* out, __nv_bfloat16* out_bf16, char* state, int64_t head_bytes, int* abort_flag,
                       cudaStream_t st);
// bf16 rows, d_k = D = 128 and one W for every head: phi runs on the tensor cores (the
// arithmetic of lola_phi_tc.cuh), in the prefill and in the decode step alike
bool phi_uses_tc(const Dims& d, int64_t w_head_stride);
cudaError_t launch_select(const Dims& d, int n, const Workspace& ws, const void* K, const void* V,
                          char* state, const Layout& L, cudaStream_t st);
// the chunk-granular allocation (alloc = LOLA_ALLOC_CHUNK); chunk_mode_fits: its shared
// memory plan fits one CTA
bool chunk_mode_fits(const Dims& d);
cudaError_t launch_chunk_select(const Dims& d, int n, const Workspace& ws, const void* K, const void* V,
                                char* state, const Layout& L, cudaStream_t st);
// the SRE map of the keys held by each snapshot of a prefill's workspace
cudaError_t launch_sre_map(const Dims& d, int n, const Workspace& ws, const void* V, float* out, cudaStream_t st);
// the relative SRE map: the map above, minus each key's SRE at its first write (kept in base)
cudaError_t launch_sre_map_relative(const Dims& d, int n, const Workspace& ws, const void* V, float* out,
                                    float* base, cudaStream_t st);
// the allocation with a query-dependent score (d.score != LOLA_SCORE_SRE): chain-free
cudaError_t launch_fixed_select(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K,
                                const void* V, char* state, const Layout& L, cudaStream_t st);
cudaError_t launch_output(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K,
                          const void* V, void* Y, cudaStream_t st);
bool output_tc_supported(const Dims& d);
// the cache read of the write-magnitude cache layer (d_k = d_v = 128, bf16): see lola_output_tc.cu
cudaError_t launch_output_tc_hola(int BH, int Hh, int n, int w, int chunk, const void* Qt, const void* Kt,
                                  const void* V, void* Y, const int32_t* snapC, int nck, const float* ystate,
                                  const float* sink, const float* gate, int32_t* status, int* abort_flag,
                                  cudaStream_t st);
cudaError_t launch_output_tc(const Dims& d, int n, const Workspace& ws, const void* Q, const void* K,
                             const void* V, void* Y, char* state, int64_t head_bytes, cudaStream_t st);
// The decode step reads phi(q), phi(k) of the token from the state's tok_phi scratch (the
// fast kernel always; the general kernel when phi_uses_tc): when decode_uses_tok_phi(d,
// w_head_stride), launch_tok_phi must run on the stream first.
bool decode_uses_tok_phi(const Dims& d, int64_t w_head_stride);
cudaError_t launch_tok_phi(const Dims& d, char* state, const Layout& L, const float* W, int64_t w_head_stride,
                           const void* q, const void* k, cudaStream_t st);
cudaError_t launch_decode(const Dims& d, char* state, const Layout& L, const float* W,
                          int64_t w_head_stride, const void* q, const void* k, const void* v, void* y,
                          int32_t* written_pos, cudaStream_t st);
cudaError_t launch_state_init(const Dims& d, char* state, const Layout& L, cudaStream_t st);
// the write-magnitude cache layer (lola_hola.cu, lola_hola_tc.cu; d_k = d_v = 128, bf16 rows)
// The state path's chunk tile: 64 tokens' unit keys (rows 0-63) and unit queries (rows
// 64-127), every float32 entry split into bf16 hi + lo, in the 128-byte-swizzled K-major layout
// the tensor-core descriptors read: term h (0 hi, 1 lo) at h * 32 KB; entries 64 e .. 64 e + 63
// of every row in atom column e (16 KB: 128 rows of 128 B, the 16-byte chunk index XORed with
// the row mod 8).  Byte offset of entry d of row r, term h.
constexpr uint32_t kHolaXTile = 65536;
__host__ __device__ __forceinline__ uint32_t hola_xtile_off(int r, int d, int h) {
    return (uint32_t)h * 32768u + (uint32_t)(d >> 6) * 16384u + (uint32_t)r * 128u +
           ((((uint32_t)(d & 63) >> 3) ^ (uint32_t)r) & 7u) * 16u + (uint32_t)(d & 7) * 2u;
}
// rows: BH x (64-token chunks x 64); tile: [BH][nck64][kHolaXTile] (rows past n are zero)
cudaError_t launch_hola_prep(int BH, int n, const void* Q, const void* K, const float* gq, const float* gk,
                             uint8_t* xtile, __nv_bfloat16* qt, __nv_bfloat16* kt, cudaStream_t st);
cudaError_t launch_hola_cache(int BH, int n, int w, int chunk, int nck, const float* scores, int32_t* cache,
                              cudaStream_t st);
int hola_max_cache();
// the state path in chunked form on tcgen05 (lola_hola_tc.cu); status: [BH][4]
cudaError_t launch_hola_state_tc(int BH, int n, const uint8_t* xtile, const void* V, const float* alpha,
                                 const float* beta, float* ystate, float* scores, float* S_out, int32_t* status,
                                 cudaStream_t st);

}  // namespace lola
