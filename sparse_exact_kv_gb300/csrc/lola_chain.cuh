// Arithmetic of the allocation rule shared by the prefill chain (lola_select.cu) and the
// decode step (lola_decode.cu).  Both kernels run 512 threads per head with the same three
// data layouts and call these functions, so a decode step continues a prefill bit for bit.
//
// LoLA reading notes (arXiv 2505.23666v3): SRE (section 2.3, Eq. 10), the candidate set
// and "score before write" (section 2.4, Eqs. 11-13), the rank-1 memory update (section
// 2.2, Eqs. 3-5).
//
// Layouts
//   H role    warp w holds the HR = D/16 rows w*HR .. w*HR + HR - 1 of H; lane l holds the
//             HC = DV/32 columns l*HC .. l*HC + HC - 1 of them, in registers (h[r*HC + c]).
//             A write then reads HR phi values (one broadcast per warp) and HC values of v;
//             H^T phi of a key is HR-row partials per warp, summed over the 16 row groups
//             in order.
//   slot role 8 lanes per cached candidate ("slot"); lane `sub` holds entries
//             slot_dim(sub, i) of phi(k), v and N = H^T phi(k) (float4 chunks interleaved
//             across the 8 lanes), and every lane holds the slot's z = s^T phi(k).
//   evictee   8 lanes hold s and the evictee's phi, v and N in the slot layout, so the
//             evictee is scored by exactly the arithmetic of a cached slot.
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
    static constexpr int NRG = kThreads / kWarp;  // H row groups, one per warp
    static constexpr int HR = D / NRG;            // H rows per thread
    static constexpr int HC = DV / kWarp;         // H columns per thread
    static constexpr int PD = D / kSG;            // phi entries per slot lane
    static constexpr int PV = DV / kSG;           // v / N entries per slot lane
    static_assert(D % NRG == 0 && HR % 4 == 0 && (HC == 2 || HC == 4) && PD % 4 == 0 && PV % 4 == 0, "shape");
};

__device__ __forceinline__ int slot_dim(int sub, int i) { return 4 * sub + 32 * (i >> 2) + (i & 3); }

// bfloat16 halves of a 32-bit word, widened to float32 (exact)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }


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
template <int HC>
__device__ __forceinline__ void h_vec_load(const float* src, float* out) {
    if constexpr (HC == 4) {
        const float4 f = *reinterpret_cast<const float4*>(src);
        out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
    } else {
        const float2 f = *reinterpret_cast<const float2*>(src);
        out[0] = f.x; out[1] = f.y;
    }
}
template <int HC>
__device__ __forceinline__ void h_vec_store(float* dst, const float* in) {
    if constexpr (HC == 4) *reinterpret_cast<float4*>(dst) = make_float4(in[0], in[1], in[2], in[3]);
    else *reinterpret_cast<float2*>(dst) = make_float2(in[0], in[1]);
}
// this thread's block of a row-major D x DV matrix (H in the state, a snapshot)
template <int D, int DV>
__device__ __forceinline__ void h_load(float* h, const float* Hm, int w, int l) {
    using S = Shape<D, DV>;
#pragma unroll
    for (int r = 0; r < S::HR; ++r) h_vec_load<S::HC>(Hm + (int64_t)(w * S::HR + r) * DV + l * S::HC, h + r * S::HC);
}
template <int D, int DV>
__device__ __forceinline__ void h_store(float* Hm, const float* h, int w, int l) {
    using S = Shape<D, DV>;
#pragma unroll
    for (int r = 0; r < S::HR; ++r) h_vec_store<S::HC>(Hm + (int64_t)(w * S::HR + r) * DV + l * S::HC, h + r * S::HC);
}
// the same block rounded to bf16 (round to nearest even)
template <int D, int DV>
__device__ __forceinline__ void h_store_bf16(__nv_bfloat16* Hm, const float* h, int w, int l) {
    using S = Shape<D, DV>;
#pragma unroll
    for (int r = 0; r < S::HR; ++r) {
        __nv_bfloat16* dst = Hm + (int64_t)(w * S::HR + r) * DV + l * S::HC;
        const float* x = h + r * S::HC;
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(x[0], x[1]);
        if constexpr (S::HC == 4) {
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(x[2], x[3]);
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
        } else {
            *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(&b0);
        }
    }
}
// this lane's HC entries of a value row (float32 or bfloat16, widened exactly)
template <int DV, typename T>
__device__ __forceinline__ void h_cols(const T* v, int l, float* out) {
    constexpr int HC = DV / kWarp;
    if constexpr (sizeof(T) == 4) {
        h_vec_load<HC>(reinterpret_cast<const float*>(v) + l * HC, out);
    } else if constexpr (HC == 4) {
        const uint2 x = *reinterpret_cast<const uint2*>(v + l * HC);
        out[0] = bf16_lo(x.x); out[1] = bf16_hi(x.x); out[2] = bf16_lo(x.y); out[3] = bf16_hi(x.y);
    } else {
        const uint32_t x = *reinterpret_cast<const uint32_t*>(v + l * HC);
        out[0] = bf16_lo(x); out[1] = bf16_hi(x);
    }
}
// H += phi_w v_w^T on this thread's block: per element fma(phi_r, v_c, H[r][c]), paired
// over columns with __ffma2_rn (two IEEE fmaf in one instruction)
template <int D, int DV>
__device__ __forceinline__ void h_update(float* h, const float* phi_w, const float* vw, int w) {
    using S = Shape<D, DV>;
    constexpr int HR = S::HR, HC2 = S::HC / 2;
    const float4* p4 = reinterpret_cast<const float4*>(phi_w + w * HR);
    float2* h2 = reinterpret_cast<float2*>(h);
#pragma unroll
    for (int r4 = 0; r4 < HR / 4; ++r4) {
        const float4 f = p4[r4];
        const float ph[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int cp = 0; cp < HC2; ++cp) {
                float2& x = h2[(4 * r4 + rr) * HC2 + cp];
                x = __ffma2_rn(make_float2(ph[rr], ph[rr]), make_float2(vw[2 * cp], vw[2 * cp + 1]), x);
            }
    }
}
// this warp's row-group partial of H^T phi for the lane's HC columns: even and odd rows
// accumulate separately (in row order), then add
template <int D, int DV>
__device__ __forceinline__ void h_partial(const float* phi, const float* h, int w, float* out) {
    using S = Shape<D, DV>;
    constexpr int HR = S::HR, HC2 = S::HC / 2;
    const float4* p4 = reinterpret_cast<const float4*>(phi + w * HR);
    const float2* h2 = reinterpret_cast<const float2*>(h);
    float2 a0[HC2], a1[HC2];
#pragma unroll
    for (int cp = 0; cp < HC2; ++cp) {
        a0[cp] = make_float2(0.f, 0.f);
        a1[cp] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int r4 = 0; r4 < HR / 4; ++r4) {
        const float4 f = p4[r4];
        const float ph[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int cp = 0; cp < HC2; ++cp) {
                float2& acc = (rr & 1) ? a1[cp] : a0[cp];
                acc = __ffma2_rn(make_float2(ph[rr], ph[rr]), h2[(4 * r4 + rr) * HC2 + cp], acc);
            }
    }
#pragma unroll
    for (int cp = 0; cp < HC2; ++cp) {
        out[2 * cp] = a0[cp].x + a1[cp].x;
        out[2 * cp + 1] = a0[cp].y + a1[cp].y;
    }
}
// the partial stored at red[w][l*HC ..] (red: [NRG][DV])
template <int D, int DV>
__device__ __forceinline__ void h_partial_store(float* red, const float* phi, const float* h, int w, int l) {
    using S = Shape<D, DV>;
    float out[S::HC];
    h_partial<D, DV>(phi, h, w, out);
    h_vec_store<S::HC>(red + w * DV + l * S::HC, out);
}
// ---- warp role (32 lanes, N/32 consecutive entries per lane): the evictee's gram with the
// written key, its z' = s^T phi and its SRE.  Fixed operation order: per lane in entry order,
// then a butterfly over xor 16, 8, 4, 2, 1; every lane gets the result. ----
template <int N>
__device__ __forceinline__ float warp_dot(const float* a, const float* b, int lane) {
    constexpr int E = N / kWarp;
    float x[E], y[E];
    h_vec_load<E>(a + lane * E, x);
    h_vec_load<E>(b + lane * E, y);
    float p = x[0] * y[0];
#pragma unroll
    for (int e = 1; e < E; ++e) p = __fmaf_rn(x[e], y[e], p);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(kFull, p, o);
    return p;
}
// SRE^2 from this lane's entries of N and v (the fallback vv when z = 0, as slot_sre2)
template <int DV>
__device__ __forceinline__ float warp_sre2(const float* Nl, float z, const float* vl, float vv) {
    constexpr int E = DV / kWarp;
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float d = __fmaf_rn(-z, vl[e], Nl[e]);
        ss = __fmaf_rn(d, d, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
    return z == 0.f ? vv : __fdividef(ss, z * z);
}

// N' = sum of the row-group partials in row-group order, one column j (any thread)
template <int D, int DV>
__device__ __forceinline__ float reduce_partials_col(const float* red, int j) {
    constexpr int NRG = Shape<D, DV>::NRG;
    float acc = red[j];
#pragma unroll
    for (int rg = 1; rg < NRG; ++rg) acc += red[rg * DV + j];
    return acc;
}

// ---- slot role (8 lanes per slot) ----
template <int D>
__device__ __forceinline__ float slot_gram(const float* wphi, const float* sphi, int sub) {
    constexpr int PD = D / kSG;
    const float2* s2 = reinterpret_cast<const float2*>(sphi);
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < PD / 4; ++c) {
        const float4 f = *reinterpret_cast<const float4*>(wphi + 32 * c + 4 * sub);
        a01 = __ffma2_rn(make_float2(f.x, f.y), s2[2 * c], a01);
        a23 = __ffma2_rn(make_float2(f.z, f.w), s2[2 * c + 1], a23);
    }
    float g = (a01.x + a01.y) + (a23.x + a23.y);
    g += __shfl_xor_sync(kFull, g, 1);
    g += __shfl_xor_sync(kFull, g, 2);
    g += __shfl_xor_sync(kFull, g, 4);
    return g;
}
template <int DV>
__device__ __forceinline__ void slot_axpy(float* sN, float g, const float* wv, int sub) {
    constexpr int PV = DV / kSG;
    float2* n2 = reinterpret_cast<float2*>(sN);
    const float2 g2 = make_float2(g, g);
#pragma unroll
    for (int c = 0; c < PV / 4; ++c) {
        const float4 f = *reinterpret_cast<const float4*>(wv + 32 * c + 4 * sub);
        n2[2 * c] = __ffma2_rn(g2, make_float2(f.x, f.y), n2[2 * c]);
        n2[2 * c + 1] = __ffma2_rn(g2, make_float2(f.z, f.w), n2[2 * c + 1]);
    }
}
template <int DV>
__device__ __forceinline__ float slot_sre2(const float* sN, float sz, const float* sv, float svv) {
    constexpr int PV = DV / kSG;
    const float2* n2 = reinterpret_cast<const float2*>(sN);
    const float2* v2 = reinterpret_cast<const float2*>(sv);
    const float2 mz = make_float2(-sz, -sz);
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < PV / 4; ++c) {
        const float2 d01 = __ffma2_rn(mz, v2[2 * c], n2[2 * c]);
        const float2 d23 = __ffma2_rn(mz, v2[2 * c + 1], n2[2 * c + 1]);
        a01 = __ffma2_rn(d01, d01, a01);
        a23 = __ffma2_rn(d23, d23, a23);
    }
    float ss = (a01.x + a01.y) + (a23.x + a23.y);
    ss += __shfl_xor_sync(kFull, ss, 1);
    ss += __shfl_xor_sync(kFull, ss, 2);
    ss += __shfl_xor_sync(kFull, ss, 4);
    // the fast reciprocal-multiply quotient (about 2 ulp): a decision is a comparison of
    // these keys, and prefill and decode form them with this same expression
    return sz == 0.f ? svv : __fdividef(ss, sz * sz);
}
template <int DV>
__device__ __forceinline__ float slot_vv(const float* sv) {
    constexpr int PV = DV / kSG;
    const float2* v2 = reinterpret_cast<const float2*>(sv);
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < PV / 4; ++c) {
        a01 = __ffma2_rn(v2[2 * c], v2[2 * c], a01);
        a23 = __ffma2_rn(v2[2 * c + 1], v2[2 * c + 1], a23);
    }
    float vv = (a01.x + a01.y) + (a23.x + a23.y);
    vv += __shfl_xor_sync(kFull, vv, 1);
    vv += __shfl_xor_sync(kFull, vv, 2);
    vv += __shfl_xor_sync(kFull, vv, 4);
    return vv;
}
// N' of the evictee in slot layout: the row-group partials red[rg][j] summed in order
template <int D, int DV>
__device__ __forceinline__ void slot_reduce_partials(const float* red, int sub, float* out) {
    constexpr int NRG = Shape<D, DV>::NRG, PV = DV / kSG;
#pragma unroll
    for (int c = 0; c < PV / 4; ++c) {
        float4 acc = *reinterpret_cast<const float4*>(red + 32 * c + 4 * sub);
#pragma unroll
        for (int rg = 1; rg < NRG; ++rg) {
            const float4 f = *reinterpret_cast<const float4*>(red + rg * DV + 32 * c + 4 * sub);
            acc.x += f.x;
            acc.y += f.y;
            acc.z += f.z;
            acc.w += f.w;
        }
        out[4 * c + 0] = acc.x;
        out[4 * c + 1] = acc.y;
        out[4 * c + 2] = acc.z;
        out[4 * c + 3] = acc.w;
    }
}
// load a slot-layout slice of a shared-memory vector
template <int N>
__device__ __forceinline__ void slot_load(const float* v, int sub, float* out) {
#pragma unroll
    for (int c = 0; c < N / kSG / 4; ++c) {
        const float4 f = *reinterpret_cast<const float4*>(v + 32 * c + 4 * sub);
        out[4 * c + 0] = f.x;
        out[4 * c + 1] = f.y;
        out[4 * c + 2] = f.z;
        out[4 * c + 3] = f.w;
    }
}
template <int N>
__device__ __forceinline__ void slot_store(float* v, int sub, const float* in) {
#pragma unroll
    for (int c = 0; c < N / kSG / 4; ++c)
        *reinterpret_cast<float4*>(v + 32 * c + 4 * sub) = make_float4(in[4 * c], in[4 * c + 1], in[4 * c + 2], in[4 * c + 3]);
}

// ---- value rows kept in the input type (bfloat16 rows are half the shared-memory
// traffic; widening a bfloat16 to float32 is exact, so the arithmetic is unchanged) ----

// slot-layout slice of a value row as raw 32-bit words (float: one value per word,
// bfloat16: two values per word)
template <int N, typename T>
struct SlotWords {
    static constexpr int kWords = (N / kSG) * (int)sizeof(T) / 4;
};
template <int N, typename T>
__device__ __forceinline__ void slot_load_words(const T* v, int sub, uint32_t* w) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int c = 0; c < N / kSG / 4; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(v + 32 * c + 4 * sub);
            w[4 * c + 0] = x.x;
            w[4 * c + 1] = x.y;
            w[4 * c + 2] = x.z;
            w[4 * c + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < N / kSG / 4; ++c) {
            const uint2 x = *reinterpret_cast<const uint2*>(v + 32 * c + 4 * sub);
            w[2 * c + 0] = x.x;
            w[2 * c + 1] = x.y;
        }
    }
}
template <int N, typename T>
__device__ __forceinline__ void slot_store_words(T* v, int sub, const uint32_t* w) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int c = 0; c < N / kSG / 4; ++c)
            *reinterpret_cast<uint4*>(v + 32 * c + 4 * sub) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    } else {
#pragma unroll
        for (int c = 0; c < N / kSG / 4; ++c)
            *reinterpret_cast<uint2*>(v + 32 * c + 4 * sub) = make_uint2(w[2 * c], w[2 * c + 1]);
    }
}
template <int N, typename T>
__device__ __forceinline__ void slot_widen(const uint32_t* w, float* out) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < N / kSG; ++i) out[i] = __uint_as_float(w[i]);
    } else {
#pragma unroll
        for (int i = 0; i < N / kSG / 2; ++i) {
            out[2 * i] = bf16_lo(w[i]);
            out[2 * i + 1] = bf16_hi(w[i]);
        }
    }
}
template <int N, typename T>
__device__ __forceinline__ void slot_load_io(const T* v, int sub, float* out) {
    uint32_t w[SlotWords<N, T>::kWords];
    slot_load_words<N, T>(v, sub, w);
    slot_widen<N, T>(w, out);
}
// slot_axpy with the written value row in the input type (same per-element FMA)
template <int DV, typename T>
__device__ __forceinline__ void slot_axpy_io(float* sN, float g, const T* wv, int sub) {
    constexpr int PV = DV / kSG;
    float v[PV];
    slot_load_io<DV, T>(wv, sub, v);
    float2* n2 = reinterpret_cast<float2*>(sN);
    const float2 g2 = make_float2(g, g);
#pragma unroll
    for (int c = 0; c < PV / 2; ++c) n2[c] = __ffma2_rn(g2, make_float2(v[2 * c], v[2 * c + 1]), n2[c]);
}

}  // namespace chain
}  // namespace lola
