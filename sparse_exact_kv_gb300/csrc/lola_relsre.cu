// The relative SRE map (LoLA reading notes, appendix G, Fig. 10, Eq. 26): for every key the
// linear memory holds at a snapshot, its SRE against that memory minus its SRE against the
// first memory that held it -- a difference, the drift of the key's recall since its write.
//
// The baseline of key j, written at step w_j, is its SRE against the memory right after
// that write: the keys written at or before w_j (in chunk-granular allocation that includes
// every key written at the same chunk start).  With the prefill's snapshots (the memory
// before step cP, every P = max(C, 128) steps) that memory is the snapshot of j's interval
// plus the keys of the same interval written at or before w_j:
//   N_j = H_c^T phi_j + sum_{i: cP <= w_i <= w_j} (phi_i . phi_j) v_i,   z_j likewise with s_c,
//   base_j = | N_j / z_j - v_j |   (|v_j| when z_j = 0: the empty memory predicts 0).
//
// relsre_base_kernel: CTA (interval c, head) gathers the keys written in [cP, cP + P) in
// position order (a ballot scan of the per-key write steps) and gives one warp per key.
// relsre_sub_kernel: out[c][j] -= base_j wherever snapshot c holds key j (0 <= w_j < cP),
// after the absolute map (lola_sre_map's kernel) has filled `out`.
#include "lola_internal.cuh"

namespace lola {
namespace {

constexpr int kRsThreads = 512;
constexpr int kRsMaxKeys = 256;   // keys written per interval: P <= 256 and at most one per step
                                  // (per token) or C per chunk start (chunk-granular)

struct RelArgs {
    int n, snap, nck;
    const float* phiK;            // [BH][n][D]
    const void* V;                // io [BH][n][DV]
    const int32_t* wstep;         // [BH][n]
    const float* snapH;           // [BH][nck][D*DV] float32, or
    const __nv_bfloat16* snapHb;  // the same in bf16 (the tensor-core path keeps these)
    const float* snapS;           // [BH][nck][D]
    float* base;                  // [BH][n] out: SRE at first write, 0 for keys never written
    float* out;                   // [BH][nck][n] the absolute map, made relative in place
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kRsThreads, 1) relsre_base_kernel(const RelArgs a) {
    extern __shared__ __align__(16) float rsm[];
    float* Hs = rsm;                         // [D][DV] the interval's snapshot of H
    float* ss = Hs + D * DV;                 // [D]     and of s
    __shared__ int keys[kRsMaxKeys];
    __shared__ int nkeys;
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int c = blockIdx.x, bh = blockIdx.y, n = a.n;
    const int64_t row0 = (int64_t)bh * n, sc = (int64_t)bh * a.nck + c;
    const int lo = c * a.snap, hi = min(n, (c + 1) * a.snap);
    const int32_t* ws = a.wstep + row0;
    for (int i = tid; i < D * DV; i += kRsThreads)
        Hs[i] = a.snapHb ? __bfloat162float(a.snapHb[sc * D * DV + i]) : a.snapH[sc * D * DV + i];
    for (int i = tid; i < D; i += kRsThreads) ss[i] = a.snapS[sc * D + i];
    if (warp == 0) {
        // a key written at step w has position <= w, so every key of the interval is below hi
        int cnt = 0;
        for (int i0 = 0; i0 < hi; i0 += kWarp) {
            const int i = i0 + lane;
            const bool in = i < hi && ws[i] >= lo && ws[i] < hi;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (in) {
                const int slot = cnt + __popc(m & ((1u << lane) - 1u));
                if (slot < kRsMaxKeys) keys[slot] = i;
            }
            cnt += __popc(m);
        }
        if (lane == 0) nkeys = min(cnt, kRsMaxKeys);
    }
    __syncthreads();
    const T* Vin = static_cast<const T*>(a.V) + row0 * DV;
    const float* PK = a.phiK + row0 * D;
    constexpr int LC = DV / kWarp;
    for (int kk = warp; kk < nkeys; kk += kRsThreads / kWarp) {
        const int j = keys[kk], wj = ws[j];
        const float* pj = PK + (int64_t)j * D;
        // N = H_c^T phi_j (lane: columns lane*LC ..), z = s_c^T phi_j
        float N[LC];
#pragma unroll
        for (int q = 0; q < LC; ++q) N[q] = 0.f;
        float z = 0.f;
        for (int r = 0; r < D; ++r) {
            const float f = pj[r];
#pragma unroll
            for (int q = 0; q < LC; ++q) N[q] = fmaf(f, Hs[r * DV + lane * LC + q], N[q]);
        }
        for (int r = lane; r < D; r += kWarp) z = fmaf(pj[r], ss[r], z);
        z = warp_sum(z);
        // the interval's keys written at or before w_j (j itself included)
        for (int m = 0; m < nkeys; ++m) {
            const int i = keys[m];
            if (ws[i] > wj) continue;
            const float* pi = PK + (int64_t)i * D;
            float g = 0.f;
            for (int r = lane; r < D; r += kWarp) g = fmaf(pi[r], pj[r], g);
            g = warp_sum(g);
            z += g;
#pragma unroll
            for (int q = 0; q < LC; ++q) N[q] = fmaf(g, IO<T>::ld(Vin, (int64_t)i * DV + lane * LC + q), N[q]);
        }
        float dd = 0.f, vv = 0.f;
#pragma unroll
        for (int q = 0; q < LC; ++q) {
            const float vq = IO<T>::ld(Vin, (int64_t)j * DV + lane * LC + q);
            const float d = z == 0.f ? 0.f : N[q] / z - vq;
            dd = fmaf(d, d, dd);
            vv = fmaf(vq, vq, vv);
        }
        dd = warp_sum(dd);
        vv = warp_sum(vv);
        if (lane == 0) a.base[row0 + j] = sqrtf(z == 0.f ? vv : dd);
    }
}

__global__ void relsre_sub_kernel(const RelArgs a) {
    const int c = blockIdx.y % a.nck, bh = blockIdx.y / a.nck, n = a.n;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const int64_t row0 = (int64_t)bh * n;
    const int w = a.wstep[row0 + j];
    if (w >= 0 && w < c * a.snap) a.out[((int64_t)bh * a.nck + c) * n + j] -= a.base[row0 + j];
}

template <int D, int DV, typename T>
cudaError_t launch_relsre_t(const Dims& d, int n, const RelArgs& a, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(a.base, 0, sizeof(float) * (size_t)d.BH * n, st);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(float) * ((size_t)D * DV + D);
    auto k = relsre_base_kernel<D, DV, T>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    k<<<dim3(a.nck, d.BH), kRsThreads, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    relsre_sub_kernel<<<dim3((n + 255) / 256, a.nck * d.BH), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sre_map_relative(const Dims& d, int n, const Workspace& ws, const void* V, float* out,
                                    float* base, cudaStream_t st) {
    if (ws.snap_interval > kRsMaxKeys) return cudaErrorInvalidValue;
    cudaError_t e = launch_sre_map(d, n, ws, V, out, st);
    if (e != cudaSuccess) return e;
    RelArgs a;
    a.n = n;
    a.snap = ws.snap_interval;
    a.nck = ws.nck;
    a.phiK = ws.phiK;
    a.V = V;
    a.wstep = ws.wstep;
    a.snapH = ws.snapH;
    a.snapHb = ws.snapHb;
    a.snapS = ws.snapS;
    a.base = base;
    a.out = out;
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_relsre_t<128, 128, __nv_bfloat16>(d, n, a, st) : launch_relsre_t<128, 128, float>(d, n, a, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_relsre_t<64, 64, __nv_bfloat16>(d, n, a, st) : launch_relsre_t<64, 64, float>(d, n, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
