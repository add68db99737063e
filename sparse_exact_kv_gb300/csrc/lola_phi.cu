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
//
// bf16 rows with d_k = D = 128 and one W for every head take the tensor cores instead
// (phi_tc_kernel, the arithmetic of lola_phi_tc.cuh): a persistent CTA per SM streams
// 128-row tiles through TMA loads, three split-W MMAs per 16 columns into a double-buffered
// TMEM accumulator, and a softmax epilogue whose rows leave by TMA stores.
#include <cuda.h>

#include "lola_internal.cuh"
#include "lola_phi_tc.cuh"

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

// ---------------------------------------------------------------------------------
// tensor-core path
//
// Roles (320 threads):
//   * warp 8 (one thread): per tile, the 128 x 128 bf16 row tile by two TMA boxes into one of
//     two stages (rows past n zero-filled);
//   * warp 9 (one thread): z = X W^T of the tile (24 MMAs) into one of two TMEM buffers,
//     committed to the epilogue and to the stage's release;
//   * warps 0-7 (epilogue): warp w reads z of rows 32 (w % 4) .. + 31 (its TMEM lane quarter)
//     and forms half w / 4 of their phi (thread = row), writes it into its own staging boxes
//     (128-byte swizzle, conflict-free) and stores them with TMA (rows past n clipped):
//     float32 phi and, when asked, its bf16 copy.
// Every wait is bounded by %globaltimer (1 s, then the head's status word gets the timeout
// bit and the launch's abort flag is set).
// ---------------------------------------------------------------------------------
namespace tcphi {
constexpr int kEpiWarps = 8, kLoadWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 10 * kWarp;
constexpr uint32_t SW = 0;                                    // W_hi, W_mid, W_lo
constexpr uint32_t SX = phitc::kWSplitBytes;                  // two row-tile stages
constexpr uint32_t SOUT = SX + 2 * phitc::kXBytes;            // per epilogue warp: 2 float32 boxes, 1 bf16 box
constexpr uint32_t kBox = 32 * 128;                           // 32 rows x 128 bytes
constexpr uint32_t kOutWarp = 3 * kBox;
constexpr uint32_t SEND = SOUT + kEpiWarps * kOutWarp;
constexpr uint64_t kWaitNs = 1000000000ull;
enum { B_XFULL = 0, B_XEMPTY = 2, B_TFULL = 4, B_TFREE = 6, B_N = 8 };
}  // namespace tcphi

struct PhiTcMaps {
    CUtensorMap x;      // bf16 [BH][n][d_k], boxes 64 x 128
    CUtensorMap out;    // float32 [BH][n][D], boxes 32 x 32
    CUtensorMap outb;   // bf16 [BH][n][D], boxes 64 x 32
};

struct PhiTcArgs {
    const float* W;
    int n, ntiles, tiles_per_head;
    int has_out, has_outb;
    char* state;        // per-head status words (timeouts)
    int64_t head_bytes;
    int* abort_flag;
};

__global__ void __launch_bounds__(tcphi::kThreads, 1) phi_tc_kernel(const __grid_constant__ PhiTcMaps maps,
                                                                  const PhiTcArgs a) {
    using namespace tcphi;
    using namespace tc;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    __shared__ __align__(8) uint64_t bars[B_N];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_sm;
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    auto tile_at = [&](int tile, int* bh, int* t0) {
        *bh = tile / a.tiles_per_head;
        *t0 = (tile % a.tiles_per_head) * 128;
    };

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_XFULL + s), 1);
            mbar_init(bar(B_XEMPTY + s), 1);
            mbar_init(bar(B_TFULL + s), 1);
            mbar_init(bar(B_TFREE + s), kEpiWarps);
        }
        abort_sm = 0;
    }
    if (warp == kMmaWarp) tmem_alloc<2 * phitc::kN>(smem_u32(&tmem_base));
    __syncthreads();
    // the first two row tiles are on their way while W is split
    if (warp == kLoadWarp && lane == 0) {
        for (int i = 0; i < 2; ++i) {
            const int tile = blockIdx.x + i * gridDim.x;
            if (tile >= a.ntiles) break;
            int bh, t0;
            tile_at(tile, &bh, &t0);
            mbar_expect(bar(B_XFULL + i), phitc::kXBytes);
            tma_load3(sb + SX + i * phitc::kXBytes, &maps.x, 0, t0, bh, bar(B_XFULL + i));
            tma_load3(sb + SX + i * phitc::kXBytes + phitc::kXAtom, &maps.x, 64, t0, bh, bar(B_XFULL + i));
        }
    }
    phitc::stage_w_split<kThreads>(sm + SW, a.W, tid);
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tb = tmem_base;

    // bounded wait on a barrier phase; gives up at once when another role has given up
    auto wait = [&](int i, uint32_t parity) -> bool {
        const uint32_t b = bar(i);
        uint64_t start = 0;
        for (int it = 0;; ++it) {
            uint32_t ok;
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}\n"
                : "=r"(ok)
                : "r"(b), "r"(parity)
                : "memory");
            if (ok) return true;
            if (*reinterpret_cast<volatile int*>(&abort_sm)) return false;
            const uint64_t now = globaltimer_ns();
            if (it == 0) start = now;
            else if (now - start > kWaitNs) {
                abort_sm = 1;
                return false;
            }
        }
    };

    if (warp == kLoadWarp) {
        // ================================ loads ================================
        if (lane == 0) {
            int last[2] = {-1, -1};
            int i = 0;
            for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++i) {
                const int s = i & 1;
                if (i >= 2) {
                    if (!wait(B_XEMPTY + s, ((i >> 1) & 1) ^ 1)) break;
                    int bh, t0;
                    tile_at(tile, &bh, &t0);
                    mbar_expect(bar(B_XFULL + s), phitc::kXBytes);
                    tma_load3(sb + SX + s * phitc::kXBytes, &maps.x, 0, t0, bh, bar(B_XFULL + s));
                    tma_load3(sb + SX + s * phitc::kXBytes + phitc::kXAtom, &maps.x, 64, t0, bh, bar(B_XFULL + s));
                }
                last[s] = i;
            }
            // no load may still be writing shared memory when the CTA ends
            for (int s = 0; s < 2; ++s)
                if (last[s] >= 0) mbar_wait(bar(B_XFULL + s), (uint32_t)(last[s] >> 1) & 1u, kWaitNs);
        }
    } else if (warp == kMmaWarp) {
        // ================================ MMA ================================
        if (lane == 0) {
            int i = 0, last = -1;
            for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++i) {
                const int s = i & 1;
                if (!wait(B_XFULL + s, (i >> 1) & 1)) break;
                if (!wait(B_TFREE + s, ((i >> 1) & 1) ^ 1)) break;
                fence_after();
                phitc::issue_mma(tb + s * phitc::kN, sb + SX + s * phitc::kXBytes, sb + SW);
                mma_commit(bar(B_TFULL + s));
                mma_commit(bar(B_XEMPTY + s));
                last = i;
            }
            // no MMA may still be running when TMEM is released
            if (last >= 0) mbar_wait(bar(B_TFULL + (last & 1)), (uint32_t)(last >> 1) & 1u, kWaitNs);
        }
    } else {
        // ================================ epilogue ================================
        const int quarter = warp & 3;
        const bool neg = warp >= 4;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint8_t* stg = sm + SOUT + warp * kOutWarp;
        const uint32_t stg_s = sb + SOUT + warp * kOutWarp;
        const int sw = lane & 7;
        int i = 0;
        for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++i) {
            const int s = i & 1;
            const bool ok = __all_sync(0xffffffffu, wait(B_TFULL + s, (i >> 1) & 1));
            if (!ok) break;
            fence_after();
            float z[phitc::kN];
            phitc::load_z(tb + lane_off + s * phitc::kN, z);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive1(bar(B_TFREE + s));
            float e[phitc::kN];
            phitc::half_phi(z, neg, e);
            // the staging boxes are free once this warp's previous stores have read them
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            if (a.has_out) {
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4*>(stg + b * kBox + lane * 128 + ((c ^ sw) << 4)) =
                            make_float4(e[32 * b + 4 * c], e[32 * b + 4 * c + 1], e[32 * b + 4 * c + 2],
                                        e[32 * b + 4 * c + 3]);
            }
            if (a.has_outb) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t pk[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __nv_bfloat162 v = __floats2bfloat162_rn(e[8 * c + 2 * q], e[8 * c + 2 * q + 1]);
                        pk[q] = *reinterpret_cast<const uint32_t*>(&v);
                    }
                    *reinterpret_cast<uint4*>(stg + 2 * kBox + lane * 128 + ((c ^ sw) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                int bh, t0;
                tile_at(tile, &bh, &t0);
                const int r0 = t0 + 32 * quarter;
                if (r0 < a.n) {
                    const int col = neg ? phitc::kN : 0;
                    if (a.has_out) {
                        tma_store3(&maps.out, col, r0, bh, stg_s);
                        tma_store3(&maps.out, col + 32, r0, bh, stg_s + kBox);
                    }
                    if (a.has_outb) tma_store3(&maps.outb, col, r0, bh, stg_s + 2 * kBox);
                }
                bulk_commit();
            }
        }
        if (lane == 0) bulk_wait0();
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (abort_sm && tid == 0) {
        int bh, t0;
        tile_at(blockIdx.x, &bh, &t0);
        atomicOr(reinterpret_cast<int32_t*>(a.state + (int64_t)bh * a.head_bytes) + HDR_STATUS, (int)ST_TIMEOUT);
        atomicExch(a.abort_flag, 1);
    }
    if (warp == kMmaWarp) tmem_dealloc<2 * phitc::kN>(tb);
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            n = v;
    }
    return n > 0 ? n : 1;
}

cudaError_t launch_phi_tc(const Dims& d, int n, const void* X, const float* W, float* out, __nv_bfloat16* outb,
                          char* state, int64_t head_bytes, int* abort_flag, cudaStream_t st) {
    PhiTcMaps maps;
    // a map over a missing output still needs a valid base: it is never used
    const void* ob = out ? static_cast<const void*>(out) : X;
    const void* obb = outb ? static_cast<const void*>(outb) : X;
    if (!tc::make_tmap3(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, phitc::kDK, n, d.BH, 64, 128) ||
        !tc::make_tmap3(&maps.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ob, phitc::kD, n, d.BH, 32, 32) ||
        !tc::make_tmap3(&maps.outb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, obb, phitc::kD, n, d.BH, 64, 32))
        return cudaErrorInvalidValue;
    PhiTcArgs a;
    a.W = W;
    a.n = n;
    a.tiles_per_head = (n + 127) / 128;
    a.ntiles = a.tiles_per_head * d.BH;
    a.has_out = out != nullptr;
    a.has_outb = outb != nullptr;
    a.state = state;
    a.head_bytes = head_bytes;
    a.abort_flag = abort_flag;
    const size_t smem = tcphi::SEND + 1024;
    cudaError_t e = cudaFuncSetAttribute(phi_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = a.ntiles < sm_count() ? a.ntiles : sm_count();
    phi_tc_kernel<<<grid, tcphi::kThreads, smem, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace

bool phi_uses_tc(const Dims& d, int64_t w_head_stride) {
    return d.dtype == LOLA_BF16 && d.dk == phitc::kDK && d.D == phitc::kD && w_head_stride == 0;
}

cudaError_t launch_phi(const Dims& d, int n, const void* X, const float* W, int64_t ws, float* out,
                       __nv_bfloat16* outb, char* state, int64_t head_bytes, int* abort_flag, cudaStream_t st) {
    if (phi_uses_tc(d, ws)) return launch_phi_tc(d, n, X, W, out, outb, state, head_bytes, abort_flag, st);
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
