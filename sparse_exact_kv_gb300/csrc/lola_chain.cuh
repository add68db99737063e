// Arithmetic of the allocation rule shared by the prefill chain (lola_select.cu) and the
// decode step (lola_decode.cu).  Both kernels run 512 threads per head with the same three
// data layouts and call these functions, so a decode step continues a prefill bit for bit.
//
// LoLA reading notes (arXiv 2505.23666v3): SRE (section 2.3, Eq. 10), the candidate set
// and "score before write" (section 2.4, Eqs. 11-13), the rank-1 memory update (section
// 2.2, Eqs. 3-5).
//
// Layouts
//   H role    thread tid holds column hj = tid % DV of H for the HR consecutive rows
//             hrg*HR .. hrg*HR + HR - 1 (hrg = tid / DV), in registers.
//   slot role 8 lanes per cached candidate ("slot"); lane `sub` holds entries
//             slot_dim(sub, i) of phi(k), v and N = H^T phi(k) (float4 chunks interleaved
//             across the 8 lanes), and every lane holds the slot's z = s^T phi(k).
//   chunk     warp 0 holds D/32 (or DV/32) consecutive entries per lane of s and of the
//             evictee's N, for the evictee's SRE.
// The evictee's N is computed one step ahead: N' = H^T phi(k_e) against the memory before
// the previous write, then corrected by that write, N = N' + (phi_w . phi_e) v_w, exactly
// like every cached slot absorbs a write.
#pragma once

#include "lola_internal.cuh"

namespace lola {
namespace chain {

constexpr int kThreads = 512;
constexpr int kSG = 8;                 // lanes per slot
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kNoKey = 0xffffffffu;
constexpr int kEvCode = 127;           // owner code of the evictee in a packed key

template <int D, int DV>
struct Shape {
    static constexpr int NRG = kThreads / DV;  // H row groups
    static constexpr int HR = D / NRG;         // H rows per thread
    static constexpr int PD = D / kSG;         // phi entries per slot lane
    static constexpr int PV = DV / kSG;        // v / N entries per slot lane
    static constexpr int CD = D / 32;          // chunk entries per lane (D vectors)
    static constexpr int CV = DV / 32;         // chunk entries per lane (DV vectors)
    static_assert(kThreads % DV == 0 && D % NRG == 0 && HR % 4 == 0 && PD % 4 == 0 && PV % 4 == 0, "shape");
};

__device__ __forceinline__ int slot_dim(int sub, int i) { return 4 * sub + 32 * (i >> 2) + (i & 3); }

// ---- packed keys: smaller SRE^2 first (the bits of a non-negative float order like an
// unsigned int), then the older position, then the owner code (slot index or kEvCode) ----
__device__ __forceinline__ uint32_t key_hi(float sre2) { return __float_as_uint(sre2); }
__device__ __forceinline__ uint32_t key_lo(int pos, int code) { return ((uint32_t)pos << 7) | (uint32_t)code; }
__device__ __forceinline__ void warp_min_key(uint32_t& hi, uint32_t& lo) {
    const uint32_t mh = __reduce_min_sync(kFull, hi);
    lo = __reduce_min_sync(kFull, hi == mh ? lo : kNoKey);
    hi = mh;
}

// ---- H role ----
template <int D, int DV>
__device__ __forceinline__ float h_partial(const float* phi, const float* h, int hrg) {
    constexpr int HR = Shape<D, DV>::HR;
    const float4* p4 = reinterpret_cast<const float4*>(phi + hrg * HR);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < HR / 4; ++c) {
        const float4 f = p4[c];
        acc = fmaf(f.x, h[4 * c + 0], acc);
        acc = fmaf(f.y, h[4 * c + 1], acc);
        acc = fmaf(f.z, h[4 * c + 2], acc);
        acc = fmaf(f.w, h[4 * c + 3], acc);
    }
    return acc;
}

template <int D, int DV>
__device__ __forceinline__ void h_update(float* h, const float* phi_w, float vj, int hrg) {
    constexpr int HR = Shape<D, DV>::HR;
    const float4* p4 = reinterpret_cast<const float4*>(phi_w + hrg * HR);
#pragma unroll
    for (int c = 0; c < HR / 4; ++c) {
        const float4 f = p4[c];
        h[4 * c + 0] = fmaf(f.x, vj, h[4 * c + 0]);
        h[4 * c + 1] = fmaf(f.y, vj, h[4 * c + 1]);
        h[4 * c + 2] = fmaf(f.z, vj, h[4 * c + 2]);
        h[4 * c + 3] = fmaf(f.w, vj, h[4 * c + 3]);
    }
}

// N'[j] = sum over row groups (in order) of the partials red[rg][j], j in lane's chunk
template <int D, int DV>
__device__ __forceinline__ void reduce_partials(const float* red, int lane, float* out) {
    constexpr int NRG = Shape<D, DV>::NRG, CV = Shape<D, DV>::CV;
#pragma unroll
    for (int i = 0; i < CV; ++i) {
        const int j = lane * CV + i;
        float acc = red[j];
#pragma unroll
        for (int rg = 1; rg < NRG; ++rg) acc += red[rg * DV + j];
        out[i] = acc;
    }
}

// ---- chunk layout (one warp) ----
// sum_k a[k] b[k] with a in registers (lane's chunk) and b in shared memory
template <int N>
__device__ __forceinline__ float chunk_dot_reg(const float* a_reg, const float* b, int lane) {
    constexpr int C = N / 32;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < C; ++i) acc = fmaf(a_reg[i], b[lane * C + i], acc);
    return warp_sum(acc);
}
template <int N>
__device__ __forceinline__ float chunk_dot(const float* a, const float* b, int lane) {
    constexpr int C = N / 32;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < C; ++i) acc = fmaf(a[lane * C + i], b[lane * C + i], acc);
    return warp_sum(acc);
}
// N += g v over the lane's chunk (v in shared memory)
template <int DV>
__device__ __forceinline__ void chunk_axpy(float* N, float g, const float* v, int lane) {
    constexpr int C = DV / 32;
#pragma unroll
    for (int i = 0; i < C; ++i) N[i] = fmaf(g, v[lane * C + i], N[i]);
}
// SRE^2 of (N, z, v); *vv receives ||v||^2 (the empty-memory SRE^2)
template <int DV>
__device__ __forceinline__ float chunk_sre2(const float* N, float z, const float* v, int lane, float* vv) {
    constexpr int C = DV / 32;
    float sse = 0.f, v2 = 0.f;
#pragma unroll
    for (int i = 0; i < C; ++i) {
        const float vi = v[lane * C + i];
        const float dlt = fmaf(-z, vi, N[i]);
        sse = fmaf(dlt, dlt, sse);
        v2 = fmaf(vi, vi, v2);
    }
    sse = warp_sum(sse);
    v2 = warp_sum(v2);
    *vv = v2;
    return z == 0.f ? v2 : sse / (z * z);
}

// ---- slot role (8 lanes per slot) ----
template <int D>
__device__ __forceinline__ float slot_gram(const float* wphi, const float* sphi, int sub) {
    constexpr int PD = D / kSG;
    float g = 0.f;
#pragma unroll
    for (int c = 0; c < PD / 4; ++c) {
        const float4 f = *reinterpret_cast<const float4*>(wphi + 32 * c + 4 * sub);
        g = fmaf(f.x, sphi[4 * c + 0], g);
        g = fmaf(f.y, sphi[4 * c + 1], g);
        g = fmaf(f.z, sphi[4 * c + 2], g);
        g = fmaf(f.w, sphi[4 * c + 3], g);
    }
    g += __shfl_xor_sync(kFull, g, 1);
    g += __shfl_xor_sync(kFull, g, 2);
    g += __shfl_xor_sync(kFull, g, 4);
    return g;
}
template <int DV>
__device__ __forceinline__ void slot_axpy(float* sN, float g, const float* wv, int sub) {
    constexpr int PV = DV / kSG;
#pragma unroll
    for (int c = 0; c < PV / 4; ++c) {
        const float4 f = *reinterpret_cast<const float4*>(wv + 32 * c + 4 * sub);
        sN[4 * c + 0] = fmaf(g, f.x, sN[4 * c + 0]);
        sN[4 * c + 1] = fmaf(g, f.y, sN[4 * c + 1]);
        sN[4 * c + 2] = fmaf(g, f.z, sN[4 * c + 2]);
        sN[4 * c + 3] = fmaf(g, f.w, sN[4 * c + 3]);
    }
}
template <int DV>
__device__ __forceinline__ float slot_sre2(const float* sN, float sz, const float* sv, float svv) {
    constexpr int PV = DV / kSG;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PV; ++i) {
        const float dlt = fmaf(-sz, sv[i], sN[i]);
        ss = fmaf(dlt, dlt, ss);
    }
    ss += __shfl_xor_sync(kFull, ss, 1);
    ss += __shfl_xor_sync(kFull, ss, 2);
    ss += __shfl_xor_sync(kFull, ss, 4);
    return sz == 0.f ? svv : ss / (sz * sz);
}
template <int DV>
__device__ __forceinline__ float slot_vv(const float* sv) {
    constexpr int PV = DV / kSG;
    float vv = 0.f;
#pragma unroll
    for (int i = 0; i < PV; ++i) vv = fmaf(sv[i], sv[i], vv);
    vv += __shfl_xor_sync(kFull, vv, 1);
    vv += __shfl_xor_sync(kFull, vv, 2);
    vv += __shfl_xor_sync(kFull, vv, 4);
    return vv;
}

}  // namespace chain
}  // namespace lola
