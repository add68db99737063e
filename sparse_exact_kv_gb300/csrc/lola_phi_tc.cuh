// The feature map phi(x) = [softmax(W x), softmax(-W x)] of bf16 rows on the tensor cores
// (LoLA reading notes, section 2.2, Eq. 3, in the configured form), for d_k = D = 128.
//
// z = X W^T is a dense [128 rows x d_k] x [d_k x D/2] product.  The rows x are bf16 (exact);
// W is float32, so it is split exactly into three bf16 terms, W = W_hi + W_mid + W_lo (each
// the nearest bf16 to what the terms before it leave), and
//   z = X W_hi^T + X W_mid^T + X W_lo^T
// accumulates in float32 in TMEM: 3 * d_k / 16 tcgen05 MMAs of M = 128, N = D/2, K = 16, always
// issued in the same order (every product of two bf16 values is exact in float32).  Then, for
// each row and each half, one thread forms
//   g = z (first half) or -z (second half),  e_m = exp(g_m - max g),
//   sum = e_0 + e_1 + ... (in increasing m),  phi_m = e_m * (1 / sum)   (reciprocal rounded).
// max(-z) = -min(z) exactly, so the second half is exp(min z - z_m) as the definition has it.
//
// Every kernel that maps a bf16 row with a W shared by all heads (the prefill's feature map of
// K and Q, the decode step's feature map of the new token) runs exactly these functions on the
// same operands: a row's phi depends only on the row, so a decode step continues a prefill bit
// for bit.
#pragma once

#include "lola_internal.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace phitc {

constexpr int kDK = 128;                                  // d_k
constexpr int kD = 128;                                   // D
constexpr int kN = kD / 2;                                // z values per row
constexpr uint32_t kXAtom = 128u * 128;                   // one 64-column atom of a 128-row tile
constexpr uint32_t kXBytes = 128u * kDK * 2;              // a 128-row tile, K-major, 128-byte swizzle
constexpr uint32_t kWAtom = (uint32_t)kN * 128;           // one 64-column atom of a W term
constexpr uint32_t kWBytes = (uint32_t)kN * kDK * 2;      // one W term
constexpr uint32_t kWSplitBytes = 3 * kWBytes;            // the three terms

// W (float32 [D/2][d_k], row-major) as its three bf16 terms W_hi, W_mid, W_lo, each a K-major
// 128-byte-swizzled tile of D/2 rows, at sw, sw + kWBytes, sw + 2 kWBytes (sw 1024-aligned).
// Every load of the thread is issued before its first store.
template <int NT>
__device__ __forceinline__ void stage_w_split(uint8_t* sw, const float* W, int tid) {
    constexpr int N4 = kN * kDK / 4;                 // float4 chunks
    constexpr int PER = (N4 + NT - 1) / NT;
    float4 w[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int i = tid + u * NT;
        if (i < N4) w[u] = reinterpret_cast<const float4*>(W)[i];
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int i = tid + u * NT;
        if (i >= N4) break;
        const int r = (4 * i) / kDK, c = (4 * i) % kDK;   // four consecutive columns, one 16-byte chunk
        const float wv[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        __nv_bfloat16 t[3][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(wv[j]);
            const float r1 = wv[j] - __bfloat162float(hi);
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mid);
            t[0][j] = hi;
            t[1][j] = mid;
            t[2][j] = __float2bfloat16_rn(r2);
        }
        const uint32_t off = (uint32_t)(c >> 6) * kWAtom + tc::kmaj_chunk(r, (c & 63) >> 3) + (uint32_t)(c & 7) * 2;
#pragma unroll
        for (int s = 0; s < 3; ++s) *reinterpret_cast<uint2*>(sw + s * kWBytes + off) = *reinterpret_cast<const uint2*>(t[s]);
    }
}

// One thread: z = X W^T of the 128-row tile at shared address sx (two 64-column atoms, K-major,
// 128-byte swizzle) into TMEM columns [tmem, tmem + D/2).  The caller commits.
__device__ __forceinline__ void issue_mma(uint32_t tmem, uint32_t sx, uint32_t sw) {
    constexpr uint32_t id = tc::idesc_bf16(128, kN, 0);
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int k = 0; k < kDK / 16; ++k) {
            const uint32_t ao = (k >> 2) * kXAtom + (k & 3) * 32;
            const uint32_t bo = (uint32_t)s * kWBytes + (k >> 2) * kWAtom + (k & 3) * 32;
            tc::mma_bf16(tmem, tc::sdesc(sx + ao, 16, 1024), tc::sdesc(sw + bo, 16, 1024), id, (s > 0 || k > 0) ? 1 : 0);
        }
}

// z of the thread's row from TMEM (lane = row; taddr includes the warp's lane quarter).
// Warp-collective.
__device__ __forceinline__ void load_z(uint32_t taddr, float (&z)[kN]) {
#pragma unroll
    for (int c = 0; c < kN; c += 32) tc::tmem_ld32(taddr + c, z + c);
    tc::tmem_wait_ld();
}

// One half of the row's phi: neg = 0 gives entries 0 .. D/2 - 1 (softmax of z), neg = 1 the
// entries D/2 .. D - 1 (softmax of -z).
__device__ __forceinline__ void half_phi(const float (&z)[kN], bool neg, float (&e)[kN]) {
    const float sg = neg ? -1.f : 1.f;
    float g[kN];
#pragma unroll
    for (int m = 0; m < kN; ++m) g[m] = sg * z[m];
    float mx = g[0];
#pragma unroll
    for (int m = 1; m < kN; ++m) mx = fmaxf(mx, g[m]);
    float sum = 0.f;
#pragma unroll
    for (int m = 0; m < kN; ++m) {
        e[m] = expf(g[m] - mx);
        sum += e[m];
    }
    const float r = __frcp_rn(sum);
#pragma unroll
    for (int m = 0; m < kN; ++m) e[m] *= r;
}

}  // namespace phitc
}  // namespace lola
