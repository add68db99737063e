// K1: feature map phi(x) = [softmax(W x), softmax(-W x)] for every row of Q or K.
//
// LoLA reading notes (arXiv 2505.23666v3), section 2.2, Eq. 3: the linear branch
// approximates exp(q^T k / sqrt(d_k)) by phi(q)^T phi(k); the configured phi is the
// two-sided softmax of a (D/2) x d_k projection W, so phi is strictly positive and each
// half sums to one.
//
// One CTA handles kRowsPerCta consecutive rows of one head (so it loads that head's W
// once into shared memory); one warp computes one row at a time with phi_warp().  The
// work is 2 * D/2 * d_k FMAs and d_k * io + D * 4 bytes per row: HBM-bound on the output.
#include "lola_internal.cuh"

namespace lola {
namespace {

constexpr int kPhiThreads = 256;
constexpr int kRowsPerCta = 128;

constexpr int kRowsPerWarp = 8;

template <int DK, int D, typename T>
__global__ void __launch_bounds__(kPhiThreads) phi_kernel(const T* __restrict__ X, const float* __restrict__ W,
                                                          int64_t w_head_stride, int n, int Hh,
                                                          float* __restrict__ out,
                                                          __nv_bfloat16* __restrict__ out_bf16) {
    extern __shared__ __align__(16) float sm[];
    float* Ws = sm;                                           // [D/2][DK+4]
    float* xs = sm + (D / 2) * w_stride<DK>();                // [warps][kRowsPerWarp][DK]
    const int bh = blockIdx.y;
    const int h = bh % Hh;
    stage_w<DK, D, kPhiThreads>(Ws, W + (int64_t)h * w_head_stride, threadIdx.x);
    __syncthreads();
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    float* xw = xs + warp * kRowsPerWarp * DK;
    const int r0 = blockIdx.x * kRowsPerCta;
    const int r1 = min(n, r0 + kRowsPerCta);
    constexpr int kWarps = kPhiThreads / kWarp;
    for (int rb = r0 + warp * kRowsPerWarp; rb < r1; rb += kWarps * kRowsPerWarp) {
        const int64_t row = (int64_t)bh * n + rb;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int c = lane; c < DK; c += kWarp)
                xw[r * DK + c] = rb + r < r1 ? IO<T>::ld(X, (row + r) * DK + c) : 0.f;
        __syncwarp();
        float ph[kRowsPerWarp][D / 32];
        phi_rows<DK, D, kRowsPerWarp>(xw, Ws, lane, ph);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            if (rb + r >= r1) break;
            if (out) {
#pragma unroll
                for (int m = 0; m < D / 32; ++m) out[(row + r) * D + lane + 32 * m] = ph[r][m];
            }
            if (out_bf16) {
#pragma unroll
                for (int m = 0; m < D / 32; ++m) out_bf16[(row + r) * D + lane + 32 * m] = __float2bfloat16_rn(ph[r][m]);
            }
        }
        __syncwarp();
    }
}

template <int DK, int D, typename T>
cudaError_t launch_phi_t(const Dims& d, int n, const void* X, const float* W, int64_t ws, float* out,
                         __nv_bfloat16* outb, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((D / 2) * w_stride<DK>() + (kPhiThreads / kWarp) * kRowsPerWarp * DK);
    auto kern = phi_kernel<DK, D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((n + kRowsPerCta - 1) / kRowsPerCta, d.BH);
    kern<<<grid, kPhiThreads, smem, st>>>(static_cast<const T*>(X), W, ws, n, d.Hh, out, outb);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_phi(const Dims& d, int n, const void* X, const float* W, int64_t ws, float* out,
                       __nv_bfloat16* outb, cudaStream_t st) {
    const bool bf = d.dtype == LOLA_BF16;
    if (d.dk == 128 && d.D == 128)
        return bf ? launch_phi_t<128, 128, __nv_bfloat16>(d, n, X, W, ws, out, outb, st)
                  : launch_phi_t<128, 128, float>(d, n, X, W, ws, out, outb, st);
    if (d.dk == 64 && d.D == 64)
        return bf ? launch_phi_t<64, 64, __nv_bfloat16>(d, n, X, W, ws, out, outb, st)
                  : launch_phi_t<64, 64, float>(d, n, X, W, ws, out, outb, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
