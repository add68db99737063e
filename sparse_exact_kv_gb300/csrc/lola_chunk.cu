// K2c: chunk-granular allocation of LoLA prefill -- the notes' own prefill schedule.
//
// LoLA reading notes (arXiv 2505.23666v3), section 2.6, Eq. 15: the sequence is cut into
// chunks of C tokens that share the memory they begin with; once a chunk is done, the
// oldest window chunk is scored together with the sparse cache (about C + lambda
// candidates, SRE of section 2.3, Eq. 10, against the current state), the lambda highest
// stay exact and the rest are written into (H, s) at once.  Readings taken (the notes
// call the window / chunk mapping ambiguous): the window is the last eta / C chunks, the
// current one included; the scoring happens as the next chunk begins (so the memory after
// the last token is not evicted from); the lowest SRE is written first and the older
// position first among equal ones; the empty memory predicts 0 (SRE = ||v||).  With C = 1
// this is the per-token rule.
//
// One CTA of 512 threads per head walks its chunks.  At every chunk start c0: the snapshot for
// the output pass when c0 is a multiple of its interval (the memory before this start's writes,
// as in the per-token chain); then the candidates -- the cache, then the chunk leaving the
// window -- are scored, ranked by (SRE^2, position), and the lowest P - lambda are added to H
// and s.  Every written key's step is recorded as c0 (the first query that reads it through
// the state), which is the rule the output kernels apply: key j is exact for query t iff
// j <= t < w_j, linear iff w_j <= t.
//
// Two builds.  bfloat16 io with D = d_v = 128: both contractions on the tensor cores
// (tcgen05), H in TMEM (float32) for the whole launch -- the candidates' N = Phi H from
// bfloat16 hi/lo splits of both operands, the written keys' H += Phi^T V from the split Phi
// and the (exact) bfloat16 values.  Otherwise (float32 io, or D = 64): CUDA cores, H in shared
// memory, the candidates scored 64 at a time (a 64 x d_v product of their phi, staged
// transposed, with H; each warp a 16-key x d_v/4-column tile of it) and the written keys
// added in rank order by rank-1 FMAs, so that the float32 decisions match an exact-arithmetic
// reference wherever their SREs differ at float32 resolution.
#include "lola_chain.cuh"
#include "lola_tc.cuh"

namespace lola {
namespace {

using chain::Shape;

constexpr int kCkThreads = 512;
constexpr int kCkWarps = kCkThreads / kWarp;
constexpr int kG = 64;                 // candidates per scoring group, 4 per warp
static_assert(kG == 4 * kCkWarps, "four candidates per warp");
constexpr int kTS = kG + 4;            // row stride of the transposed phi tile (floats)
// tensor-core scoring (bfloat16 io, D = d_v = 128): candidates per MMA group (M), TMEM
// columns (the fp32 N tile), the halves of the split operands, the completion wait limit
constexpr int kGT = 128;
constexpr int kGW = 64;                // written keys per H-update product group (K)
constexpr int kTmemCols = 256;         // [0, 128): the scoring tile N; [128, 256): H (float32)
constexpr uint32_t kTH = 128;
constexpr uint32_t kAhalf = 2u * kGT * 128, kBhalf = 2u * 128 * 128, kAWhalf = 2u * kGW * 128;
constexpr uint64_t kCkWaitNs = 1000000000ull;

struct ChunkArgs {
    int n, eta, lam, C, nwc, snap, nck;
    const float* phiK;         // [BH][n][D] float32
    const void* K;             // io [BH][n][D]
    const void* V;             // io [BH][n][DV]
    int32_t* wstep;            // [BH][n]: chunk start at which key j was written, -1 never
    int32_t* wpos;             // [BH][n] (the caller's log, nullable): the same per key
    float* snapH;              // [BH][nck][D*DV] float32, or
    __nv_bfloat16* snapHb;     // the same in bf16
    float* snapS;              // [BH][nck][D]
    int32_t* snapC;            // [BH][nck][lam]
    char* state;
    Layout L;
};

__host__ __device__ constexpr size_t a16c(size_t x) { return (x + 15) / 16 * 16; }

// shared-memory plan (bytes), from the runtime lambda and C; with TC the offsets are from a
// 1024-byte aligned base (the swizzled operand tiles) and `total` includes the slack
template <int D, int DV, bool TC>
struct CkPlan {
    size_t A, B, H, tile, red, s, cpos, cand, keys, wlist, klist, total;
    __host__ __device__ CkPlan(int lam, int C) {
        const size_t P = (size_t)lam + C;
        // scoring on CUDA cores: phi transposed [D][kTS] + v [kG][DV]; writing: phi [kG][D] +
        // v [kG][DV] (float32)
        const size_t tile_b = 4ull * (D * kTS > kG * D ? D * kTS : kG * D) + 4ull * kG * DV;
        if (TC) {
            // A: the candidates' phi as bf16 hi and lo parts (K-major [kGT][D] each), B: H
            // likewise (MN-major [D][DV] each); the write phase's operands reuse A; H itself
            // lives in TMEM
            A = 0;
            B = A + 2ull * kAhalf;
            H = 0;
            tile = 0;
            red = B + 2ull * kBhalf;             // z and the column blocks' partials
            s = a16c(red + 4ull * 9 * kGT);
        } else {
            A = B = 0;
            H = 0;
            tile = H + 4ull * D * DV;
            red = a16c(tile + tile_b);           // tile_sre2's z and column-block partials
            s = a16c(red + 4ull * 9 * kG);
        }
        cpos = a16c(s + 4ull * D);
        cand = a16c(cpos + 4ull * (lam > 0 ? lam : 1));
        keys = a16c(cand + 4 * P);
        wlist = a16c(keys + 8 * P);
        klist = a16c(wlist + 4 * P);
        total = a16c(klist + 4ull * (lam > 0 ? lam : 1)) + (TC ? 1024 : 0);
    }
};

// eight float32 as bfloat16 hi parts and the bfloat16 of the remainders (x - hi is exact)
__device__ __forceinline__ void split8(const float4& a, const float4& b, uint4& hi, uint4& lo) {
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        const float2 hf = __bfloat1622float2(hh);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
        h[e] = *reinterpret_cast<const uint32_t*>(&hh);
        l[e] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// kG rows of phi (float32, D wide) and of v (input type, DV wide, widened exactly) for the
// keys at positions pos(j), j < cnt (zero rows beyond), all loads issued before any store.
// phi moves as float4 into phi_at(j, r) (four consecutive r); with JM the 32 lanes of a
// warp take 32 consecutive keys (conflict-free stores into a transposed tile), else 32
// consecutive float4 of one row.  v moves 16 bytes at a time into vt[j * DV + q].
template <int D, int DV, typename T, bool JM, typename Pos, typename PhiAt>
__device__ __forceinline__ void stage_rows(const float* phiK, const T* Vin, int cnt, Pos pos, PhiAt phi_at, float* vt,
                                           int tid) {
    constexpr int F4 = kG * D / 4 / kCkThreads;           // float4 of phi per thread
    constexpr int VE = 16 / (int)sizeof(T);               // values per 16-byte chunk of v
    constexpr int V4 = kG * DV / VE / kCkThreads;         // chunks of v per thread
    static_assert(F4 * 4 * kCkThreads == kG * D && V4 * VE * kCkThreads == kG * DV, "staging split");
    float4 f[F4];
    uint4 vr[V4];
#pragma unroll
    for (int u = 0; u < F4; ++u) {
        const int i = tid + u * kCkThreads;
        const int j = JM ? i % kG : i / (D / 4), r4 = JM ? i / kG : i % (D / 4);
        f[u] = j < cnt ? *reinterpret_cast<const float4*>(phiK + (int64_t)pos(j) * D + 4 * r4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < V4; ++u) {
        const int i = tid + u * kCkThreads, j = i / (DV / VE), c = i % (DV / VE);
        vr[u] = j < cnt ? *reinterpret_cast<const uint4*>(Vin + (int64_t)pos(j) * DV + VE * c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < F4; ++u) {
        const int i = tid + u * kCkThreads;
        const int j = JM ? i % kG : i / (D / 4), r4 = JM ? i / kG : i % (D / 4);
        phi_at(j, 4 * r4 + 0) = f[u].x;
        phi_at(j, 4 * r4 + 1) = f[u].y;
        phi_at(j, 4 * r4 + 2) = f[u].z;
        phi_at(j, 4 * r4 + 3) = f[u].w;
    }
#pragma unroll
    for (int u = 0; u < V4; ++u) {
        const int i = tid + u * kCkThreads, j = i / (DV / VE), c = i % (DV / VE);
        float* dst = vt + j * DV + VE * c;
        if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(vr[u].x), __uint_as_float(vr[u].y),
                                                          __uint_as_float(vr[u].z), __uint_as_float(vr[u].w));
        } else {
            const uint32_t w4[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dst[2 * k] = chain::bf16_lo(w4[k]);
                dst[2 * k + 1] = chain::bf16_hi(w4[k]);
            }
        }
    }
}

// SRE^2 of the kG keys staged in the tile (phi transposed [D][kTS], values [kG][DV]) against
// (H, s) in shared memory, for keys j < nvalid.  N = H^T phi is a [kG x DV] product over the D
// rows: warp w takes keys 16 (w % 4) .. + 15 and value columns (w / 4) * 8 LC .. (LC = DV / 32),
// lane l four of those keys (4 (l / 8) ..) and LC columns ((l % 8) LC ..), so that a row costs
// the warp one shared-memory wavefront of phi and one of H.  z = s^T phi is formed first (warp w
// for keys 4w .. 4w + 3, lane-strided rows, then a warp sum) and shared through red[0 .. kG);
// each warp's |N - z v|^2 and |v|^2 over its columns go to red[kG ..], and thread j < kG adds the
// four column blocks in order: SRE^2 = |N - z v|^2 / z^2, or |v|^2 when z = 0 (the empty memory
// predicts 0).  Thread j hands (j, SRE^2) to emit.  red holds kG + 2 * 4 * kG floats; contains
// two block-wide barriers, so every thread of the CTA calls it.
template <int D, int DV, typename Emit>
__device__ __forceinline__ void tile_sre2(const float* Hs, const float* ss, const float* tile, const float* vts,
                                          float* red, int nvalid, int warp, int lane, Emit emit) {
    constexpr int LC = DV / kWarp, LC2 = LC / 2, NCB = 4;   // columns per lane, column blocks
    static_assert(LC % 2 == 0 && kG == 16 * 4 && kCkWarps == 4 * NCB && DV == NCB * 8 * LC, "warp tiling");
    float* zs = red;
    float* part = red + kG;   // [NCB][kG][2]
    // z = s^T phi(k) for keys 4w .. 4w + 3: lane l takes rows l, l + 32, ...
    {
        float z4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = lane; r < D; r += kWarp) {
            const float4 f = *reinterpret_cast<const float4*>(tile + r * kTS + 4 * warp);
            const float sr = ss[r];
            z4[0] = fmaf(f.x, sr, z4[0]);
            z4[1] = fmaf(f.y, sr, z4[1]);
            z4[2] = fmaf(f.z, sr, z4[2]);
            z4[3] = fmaf(f.w, sr, z4[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float z = warp_sum(z4[i]);
            if (lane == 0) zs[4 * warp + i] = z;
        }
    }
    const int cb = warp % 4, colb = warp / 4;
    const int j0 = 16 * cb + 4 * (lane / 8);                 // this lane's four keys
    const int c0 = colb * 8 * LC + (lane % 8) * LC;          // and LC columns
    // column pairs in float2: one paired FMA per two products, each rounded as a single fmaf;
    // every element takes the rows in order
    float2 acc2[4][LC2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < LC2; ++q) acc2[i][q] = make_float2(0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < D; ++r) {
        float h[LC];
        chain::h_vec_load<LC>(Hs + r * DV + c0, h);
        const float4 f = *reinterpret_cast<const float4*>(tile + r * kTS + j0);
        const float fi[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int q = 0; q < LC2; ++q)
                acc2[i][q] = __ffma2_rn(make_float2(fi[i], fi[i]), make_float2(h[2 * q], h[2 * q + 1]), acc2[i][q]);
    }
    __syncthreads();   // zs complete
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = j0 + i;
        const float z = zs[j];
        float v[LC];
        chain::h_vec_load<LC>(vts + j * DV + c0, v);
        float dd = 0.f, vv = 0.f;
#pragma unroll
        for (int q = 0; q < LC2; ++q) {
            const float d0 = fmaf(-z, v[2 * q], acc2[i][q].x), d1 = fmaf(-z, v[2 * q + 1], acc2[i][q].y);
            dd = fmaf(d0, d0, dd);
            dd = fmaf(d1, d1, dd);
            vv = fmaf(v[2 * q], v[2 * q], vv);
            vv = fmaf(v[2 * q + 1], v[2 * q + 1], vv);
        }
        // the eight lanes of this key group hold the warp's column block
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            dd += __shfl_xor_sync(0xffffffffu, dd, o);
            vv += __shfl_xor_sync(0xffffffffu, vv, o);
        }
        if (lane % 8 == 0) {
            part[(colb * kG + j) * 2] = dd;
            part[(colb * kG + j) * 2 + 1] = vv;
        }
    }
    __syncthreads();   // the column blocks' partials
    const int j = warp * kWarp + lane;
    if (j < kG && j < nvalid) {
        float dd = 0.f, vv = 0.f;
#pragma unroll
        for (int b = 0; b < NCB; ++b) {
            dd += part[(b * kG + j) * 2];
            vv += part[(b * kG + j) * 2 + 1];
        }
        const float z = zs[j];
        emit(j, z == 0.f ? vv : dd / (z * z));
    }
}

// TC: the scoring runs on the tensor cores (bfloat16 io, D = d_v = 128 only).  N = Phi H is
// formed from bfloat16 hi/lo splits of both operands, Phi_hi H_hi + Phi_hi H_lo + Phi_lo H_hi,
// accumulated in float32 in TMEM (relative error about 2^-16; the lo x lo term is dropped),
// kGT candidates per group (M = kGT, N = d_v, K = D; A K-major, B MN-major, 128-byte
// swizzle).  z = s^T phi stays float32 on the CUDA cores, formed while A is staged; the
// epilogue reads N from TMEM (warp w: TMEM lanes 32 (w % 4) .., columns 32 (w / 4) ..).
template <int D, int DV, typename T, bool TC>
__global__ void __launch_bounds__(kCkThreads, 1) chunk_select_kernel(const ChunkArgs a) {
    using S = Shape<D, DV>;
    constexpr int HR = S::HR, HC = S::HC;
    static_assert(kCkThreads == chain::kThreads, "H blocks of the chain layout");
    static_assert(!TC || (D == 128 && DV == 128 && sizeof(T) == 2), "tensor-core scoring: bf16, D = d_v = 128");
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = TC ? reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023))
                           : smraw;
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_base;
    const CkPlan<D, DV, TC> pl(a.lam, a.C);
    float* Hs = reinterpret_cast<float*>(sm + pl.H);
    float* tile = reinterpret_cast<float*>(sm + pl.tile);
    float* red = reinterpret_cast<float*>(sm + pl.red);
    float* ss = reinterpret_cast<float*>(sm + pl.s);
    int* cpos = reinterpret_cast<int*>(sm + pl.cpos);
    int* cand = reinterpret_cast<int*>(sm + pl.cand);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(sm + pl.keys);
    int* wlist = reinterpret_cast<int*>(sm + pl.wlist);
    int* klist = reinterpret_cast<int*>(sm + pl.klist);

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int bh = blockIdx.x;
    const int n = a.n, lam = a.lam, C = a.C;
    const int64_t row0 = (int64_t)bh * n;
    const float* phiK = a.phiK + row0 * D;
    const T* Vin = static_cast<const T*>(a.V) + row0 * DV;
    int32_t* wst = a.wstep + row0;
    int32_t* wps = a.wpos ? a.wpos + row0 : nullptr;

    if constexpr (!TC)
        for (int i = tid; i < D * DV; i += kCkThreads) Hs[i] = 0.f;
    for (int i = tid; i < D; i += kCkThreads) ss[i] = 0.f;
    for (int i = tid; i < n; i += kCkThreads) {
        wst[i] = -1;
        if (wps) wps[i] = -1;
    }
    int nc = 0, nwritten = 0;   // (uniform)
    uint32_t tb = 0, phase = 0;
    bool timed_out = false;     // (uniform)
    if constexpr (TC) {
        if (tid == 0) tc::mbar_init(tc::smem_u32(&mbar), 1);
        if (warp == 0) tc::tmem_alloc<kTmemCols>(tc::smem_u32(&tmem_base));
        tc::fence_before();
    }
    __syncthreads();
    // TC: thread (warp w, lane l) reads and writes H row 32 (w % 4) + l, columns 32 (w / 4) ..
    // (its TMEM lane quarter and column block)
    const uint32_t lane_q = (uint32_t)(32 * (warp & 3)) << 16;
    const int hrow = 32 * (warp & 3) + lane, hcol = 32 * (warp >> 2);
    if constexpr (TC) {
        tc::fence_after();
        tb = tmem_base;
        float zero[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) zero[i] = 0.f;
        tc::tmem_st32(tb + lane_q + kTH + hcol, zero);   // H = 0
        tc::tmem_wait_st();
    }

    const int nch = (n + C - 1) / C;
    for (int c = 0; c < nch; ++c) {
        const int c0 = c * C;
        // ---- the output pass's snapshot: the memory the chunk begins with, before this
        //      start's writes ----
        if (c0 % a.snap == 0) {
            const int64_t sc = (int64_t)bh * a.nck + c0 / a.snap;
            if constexpr (TC) {
                float hv[32];
                tc::tmem_ld32(tb + lane_q + kTH + hcol, hv);
                tc::tmem_wait_ld();
                const int64_t o = sc * D * DV + (int64_t)hrow * DV + hcol;
                if (a.snapHb) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 b = __floats2bfloat162_rn(hv[8 * q + 2 * e], hv[8 * q + 2 * e + 1]);
                            w[e] = *reinterpret_cast<const uint32_t*>(&b);
                        }
                        *reinterpret_cast<uint4*>(a.snapHb + o + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<float4*>(a.snapH + o + 4 * q) =
                            make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
                }
            } else if (a.snapHb) {
                for (int i = tid; i < D * DV; i += kCkThreads) a.snapHb[sc * D * DV + i] = __float2bfloat16_rn(Hs[i]);
            } else {
                for (int i = tid; i < D * DV; i += kCkThreads) a.snapH[sc * D * DV + i] = Hs[i];
            }
            for (int i = tid; i < D; i += kCkThreads) a.snapS[sc * D + i] = ss[i];
            for (int i = tid; i < lam; i += kCkThreads) a.snapC[sc * lam + i] = i < nc ? cpos[i] : -1;
        }
        const int e = c - a.nwc;   // the chunk that leaves the window now
        if (e < 0) continue;
        const int P = nc + C;
        for (int i = tid; i < P; i += kCkThreads) cand[i] = i < nc ? cpos[i] : e * C + (i - nc);
        __syncthreads();
        if (P <= lam) {             // room for every candidate
            for (int i = tid; i < C; i += kCkThreads) cpos[nc + i] = e * C + i;
            nc = P;
            __syncthreads();
            continue;
        }

        // ---- SRE^2 of every candidate against the current (H, s) ----
        if constexpr (TC) {
            unsigned char* Ab = sm + pl.A;
            unsigned char* Bb = sm + pl.B;
            float* zs = red;              // [kGT]
            float* part = red + kGT;      // [4][kGT][2]
            // B = H as bf16 hi and lo (MN-major), once per scoring chunk start, from TMEM
            {
                float hv[32];
                tc::tmem_ld32(tb + lane_q + kTH + hcol, hv);
                tc::tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 hi, lo;
                    split8(make_float4(hv[8 * q], hv[8 * q + 1], hv[8 * q + 2], hv[8 * q + 3]),
                           make_float4(hv[8 * q + 4], hv[8 * q + 5], hv[8 * q + 6], hv[8 * q + 7]), hi, lo);
                    const uint32_t off = tc::mnmaj_chunk(hrow, hcol + 8 * q, D);
                    *reinterpret_cast<uint4*>(Bb + off) = hi;
                    *reinterpret_cast<uint4*>(Bb + kBhalf + off) = lo;
                }
            }
            for (int g0 = 0; g0 < P; g0 += kGT) {
                const int cnt = min(kGT, P - g0);
                // A = the group's phi rows split (K-major; rows >= cnt zero); thread tid takes
                // the 16-byte chunk c16 = tid % 16 of rows tid / 16 + 32 u, u < 4, and z of
                // those rows is summed over the 16 lanes that hold a row
                {
                    constexpr int U = kGT * (D / 8) / kCkThreads;
                    static_assert(U * kCkThreads == kGT * (D / 8) && D / 8 == 16, "A staging split");
                    const int c16 = tid & 15;
                    float4 f[U][2];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int r = (tid >> 4) + 32 * u;
                        if (r < cnt) {
                            const float* src = phiK + (int64_t)cand[g0 + r] * D + c16 * 8;
                            f[u][0] = *reinterpret_cast<const float4*>(src);
                            f[u][1] = *reinterpret_cast<const float4*>(src + 4);
                        } else {
                            f[u][0] = f[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    const float4 s0 = *reinterpret_cast<const float4*>(ss + c16 * 8);
                    const float4 s1 = *reinterpret_cast<const float4*>(ss + c16 * 8 + 4);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int r = (tid >> 4) + 32 * u;
                        uint4 hi, lo;
                        split8(f[u][0], f[u][1], hi, lo);
                        const uint32_t off = (c16 >> 3) * 16384 + tc::kmaj_chunk(r, c16 & 7);
                        *reinterpret_cast<uint4*>(Ab + off) = hi;
                        *reinterpret_cast<uint4*>(Ab + kAhalf + off) = lo;
                        float z = 0.f;
                        z = fmaf(f[u][0].x, s0.x, z);
                        z = fmaf(f[u][0].y, s0.y, z);
                        z = fmaf(f[u][0].z, s0.z, z);
                        z = fmaf(f[u][0].w, s0.w, z);
                        z = fmaf(f[u][1].x, s1.x, z);
                        z = fmaf(f[u][1].y, s1.y, z);
                        z = fmaf(f[u][1].z, s1.z, z);
                        z = fmaf(f[u][1].w, s1.w, z);
#pragma unroll
                        for (int o = 1; o < 16; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                        if (c16 == 0) zs[r] = z;
                    }
                }
                tc::fence_async_smem();
                tc::fence_before();
                __syncthreads();
                tc::fence_after();
                if (tid == 0) {
                    constexpr uint32_t id = tc::idesc_bf16(kGT, DV, 1);
                    const uint32_t sa = tc::smem_u32(Ab), sb = tc::smem_u32(Bb);
#pragma unroll 1
                    for (int pass = 0; pass < 3; ++pass) {   // hi x hi, hi x lo, lo x hi
                        const uint32_t ao = pass == 2 ? kAhalf : 0u, bo = pass == 1 ? kBhalf : 0u;
#pragma unroll
                        for (int k = 0; k < D / 16; ++k) {
                            const uint64_t ad = tc::sdesc(sa + ao + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
                            const uint64_t bd = tc::sdesc(sb + bo + k * 2048, 16384, 1024);
                            tc::mma_bf16(tb, ad, bd, id, (pass | k) != 0);
                        }
                    }
                    tc::mma_commit(tc::smem_u32(&mbar));
                }
                // the epilogue's values, loaded while the products run
                const int ql = warp & 3, colb = warp >> 2, j = 32 * ql + lane;
                uint4 vr[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) vr[q] = make_uint4(0, 0, 0, 0);
                if (j < cnt) {
                    const uint4* src = reinterpret_cast<const uint4*>(Vin + (int64_t)cand[g0 + j] * DV + 32 * colb);
#pragma unroll
                    for (int q = 0; q < 4; ++q) vr[q] = src[q];
                }
                const bool ok = tc::mbar_wait(tc::smem_u32(&mbar), phase, kCkWaitNs);
                phase ^= 1u;
                tc::fence_after();
                if (__syncthreads_or(!ok)) {
                    timed_out = true;
                    break;
                }
                float nv[32];
                tc::tmem_ld32(tb + ((uint32_t)(32 * ql) << 16) + 32 * colb, nv);
                tc::tmem_wait_ld();
                const float z = zs[j];
                float dd = 0.f, vv = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t w4[4] = {vr[q].x, vr[q].y, vr[q].z, vr[q].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float v0 = chain::bf16_lo(w4[e]), v1 = chain::bf16_hi(w4[e]);
                        const float d0 = fmaf(-z, v0, nv[8 * q + 2 * e]), d1 = fmaf(-z, v1, nv[8 * q + 2 * e + 1]);
                        dd = fmaf(d0, d0, dd);
                        dd = fmaf(d1, d1, dd);
                        vv = fmaf(v0, v0, vv);
                        vv = fmaf(v1, v1, vv);
                    }
                }
                part[(colb * kGT + j) * 2] = dd;
                part[(colb * kGT + j) * 2 + 1] = vv;
                tc::fence_before();
                __syncthreads();
                if (tid < cnt) {
                    float d2 = 0.f, v2 = 0.f;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        d2 += part[(b * kGT + tid) * 2];
                        v2 += part[(b * kGT + tid) * 2 + 1];
                    }
                    const float zt = zs[tid];
                    const float sre2 = zt == 0.f ? v2 : d2 / (zt * zt);
                    keys[g0 + tid] = ((unsigned long long)__float_as_uint(sre2) << 32) | (unsigned)cand[g0 + tid];
                }
                __syncthreads();   // A, z and the partials are restaged; TMEM is read
            }
            if (timed_out) break;
        } else {
            // on the CUDA cores, kG candidates at a time
            float* vts = tile + D * kTS;   // [kG][DV] the group's values (float32)
            for (int g0 = 0; g0 < P; g0 += kG) {
                const int cnt = min(kG, P - g0);
                stage_rows<D, DV, T, true>(phiK, Vin, cnt, [&](int j) { return cand[g0 + j]; },
                                           [&](int j, int r) -> float& { return tile[r * kTS + j]; }, vts, tid);
                __syncthreads();
                tile_sre2<D, DV>(Hs, ss, tile, vts, red, cnt, warp, lane, [&](int j, float sre2) {
                    keys[g0 + j] = ((unsigned long long)__float_as_uint(sre2) << 32) | (unsigned)cand[g0 + j];
                });
                __syncthreads();   // the tile is restaged
            }
        }

        // ---- rank by (SRE^2, position): the lowest P - lambda are written ----
        // (four consecutive lanes per candidate, each counting a quarter of the keys)
        const int nwr = P - lam;
        for (int base = 0; base < P; base += kCkThreads / 4) {
            const int i = base + tid / 4, part = tid % 4;
            const unsigned long long k = i < P ? keys[i] : 0ull;
            int r = 0;
            if (i < P)
                for (int j = part; j < P; j += 4) r += keys[j] < k ? 1 : 0;
            r += __shfl_xor_sync(0xffffffffu, r, 1);
            r += __shfl_xor_sync(0xffffffffu, r, 2);
            if (i < P && part == 0) {
                const int p = (int)(k & 0xffffffffu);
                if (r < nwr) wlist[r] = p;
                else klist[r - nwr] = p;
            }
        }
        __syncthreads();

        // ---- H += sum phi(k) v^T and s += sum phi(k) over the written keys ----
        if constexpr (TC) {
            // on the tensor cores, into H in TMEM: kGW keys per group, A = their phi split
            // into bf16 hi and lo, B = their values (both MN-major [keys][D]); two passes,
            // Phi_hi^T V + Phi_lo^T V.  s in float32 on the CUDA cores from the staged rows:
            // each thread adds its two keys, the two lanes holding one column block add, the
            // 16 warps' partials go to spart (the scoring B tile, idle here) and thread r < D
            // adds them in warp order while the products run
            unsigned char* AW = sm + pl.A;
            unsigned char* VW = sm + pl.A + 2 * kAWhalf;
            float* spart = reinterpret_cast<float*>(sm + pl.B);   // [kCkWarps][D]
            float sreg = tid < D ? ss[tid] : 0.f;
            for (int w0 = 0; w0 < nwr; w0 += kGW) {
                const int cnt = min(kGW, nwr - w0);
                constexpr int U = kGW * (D / 8) / kCkThreads;
                static_assert(U * kCkThreads == kGW * (D / 8) && D == DV, "write staging split");
                const int c16 = tid & 15;
                float4 f[U][2];
                uint4 vr[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = (tid >> 4) + 32 * u;
                    if (k < cnt) {
                        const int p = wlist[w0 + k];
                        const float* src = phiK + (int64_t)p * D + c16 * 8;
                        f[u][0] = *reinterpret_cast<const float4*>(src);
                        f[u][1] = *reinterpret_cast<const float4*>(src + 4);
                        vr[u] = *reinterpret_cast<const uint4*>(Vin + (int64_t)p * DV + c16 * 8);
                    } else {
                        f[u][0] = f[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                        vr[u] = make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = (tid >> 4) + 32 * u;
                    uint4 hi, lo;
                    split8(f[u][0], f[u][1], hi, lo);
                    const uint32_t off = tc::mnmaj_chunk(k, c16 * 8, kGW);
                    *reinterpret_cast<uint4*>(AW + off) = hi;
                    *reinterpret_cast<uint4*>(AW + kAWhalf + off) = lo;
                    *reinterpret_cast<uint4*>(VW + off) = vr[u];
                }
                {
                    static_assert(U == 2, "two keys per thread");
                    float sp[8] = {f[0][0].x + f[1][0].x, f[0][0].y + f[1][0].y, f[0][0].z + f[1][0].z,
                                   f[0][0].w + f[1][0].w, f[0][1].x + f[1][1].x, f[0][1].y + f[1][1].y,
                                   f[0][1].z + f[1][1].z, f[0][1].w + f[1][1].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) sp[e] += __shfl_xor_sync(0xffffffffu, sp[e], 16);
                    if (lane < 16) {
                        float* dst = spart + warp * D + c16 * 8;
                        *reinterpret_cast<float4*>(dst) = make_float4(sp[0], sp[1], sp[2], sp[3]);
                        *reinterpret_cast<float4*>(dst + 4) = make_float4(sp[4], sp[5], sp[6], sp[7]);
                    }
                }
                tc::fence_async_smem();
                tc::fence_before();
                __syncthreads();
                tc::fence_after();
                if (tid == 0) {
                    constexpr uint32_t id = tc::idesc_bf16(D, DV, 1) | (1u << 15);   // A MN-major too
                    const uint32_t sa = tc::smem_u32(AW), sv = tc::smem_u32(VW);
#pragma unroll
                    for (int pass = 0; pass < 2; ++pass)
#pragma unroll
                        for (int k = 0; k < kGW / 16; ++k) {
                            const uint64_t ad = tc::sdesc(sa + pass * kAWhalf + k * 2048, (kGW / 8) * 1024, 1024);
                            const uint64_t bd = tc::sdesc(sv + k * 2048, (kGW / 8) * 1024, 1024);
                            tc::mma_bf16(tb + kTH, ad, bd, id, 1);
                        }
                    tc::mma_commit(tc::smem_u32(&mbar));
                }
                if (tid < D) {
                    float inc = 0.f;
#pragma unroll
                    for (int w = 0; w < kCkWarps; ++w) inc += spart[w * D + tid];
                    sreg += inc;
                }
                const bool ok = tc::mbar_wait(tc::smem_u32(&mbar), phase, kCkWaitNs);
                phase ^= 1u;
                tc::fence_after();
                if (__syncthreads_or(!ok)) {   // (also: this group's operands and spart are consumed)
                    timed_out = true;
                    break;
                }
            }
            if (timed_out) break;
            if (tid < D) ss[tid] = sreg;
        } else {
            // on the CUDA cores, in rank order: thread (warp w, lane l) owns rows w*HR .. and
            // columns l*HC .. of H
            float hreg[HR * HC];
            chain::h_load<D, DV>(hreg, Hs, warp, lane);
            float sreg = tid < D ? ss[tid] : 0.f;
            float* tphi = tile;              // [kG][D]
            float* tv = tile + D * kTS;      // [kG][DV]
            for (int w0 = 0; w0 < nwr; w0 += kG) {
                const int cnt = min(kG, nwr - w0);
                stage_rows<D, DV, T, false>(phiK, Vin, cnt, [&](int j) { return wlist[w0 + j]; },
                                     [&](int j, int r) -> float& { return tphi[j * D + r]; }, tv, tid);
                __syncthreads();
                // (unrolled so that the next keys' loads overlap this key's products; every
                //  element still takes the keys one after another, in rank order)
#pragma unroll 4
                for (int j = 0; j < cnt; ++j) {
                    float vh[HC];
                    chain::h_vec_load<HC>(tv + j * DV + lane * HC, vh);
                    chain::h_update<D, DV>(hreg, tphi + j * D, vh, warp);
                }
                if (tid < D)
                    for (int j = 0; j < cnt; ++j) sreg += tphi[j * D + tid];
                __syncthreads();
            }
            chain::h_store<D, DV>(Hs, hreg, warp, lane);
            if (tid < D) ss[tid] = sreg;
        }
        for (int i = tid; i < nwr; i += kCkThreads) {
            wst[wlist[i]] = c0;
            if (wps) wps[wlist[i]] = c0;
        }
        for (int i = tid; i < lam; i += kCkThreads) cpos[i] = klist[i];
        nc = lam;
        nwritten += nwr;
        __syncthreads();
    }

    char* rec = a.state + (int64_t)bh * a.L.head_bytes;
    float* Hg = reinterpret_cast<float*>(rec + a.L.H);
    if constexpr (TC) {
        if (!timed_out) {
            float hv[32];
            tc::tmem_ld32(tb + lane_q + kTH + hcol, hv);
            tc::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(Hg + (int64_t)hrow * DV + hcol + 4 * q) =
                    make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        if (warp == 0) tc::tmem_dealloc<kTmemCols>(tb);
        if (timed_out) {   // a product group did not complete: report it, export nothing
            if (tid == 0) reinterpret_cast<int32_t*>(rec)[HDR_STATUS] = ST_TIMEOUT;
            return;
        }
    }

    // ---- export: header, H, s, the cache (positions and rows) and the window ring ----
    if (tid == 0) {
        int32_t* hdr = reinterpret_cast<int32_t*>(rec);
        hdr[HDR_T] = n;
        hdr[HDR_NCACHE] = nc;
        hdr[HDR_NWRITTEN] = nwritten;
        hdr[HDR_STATUS] = 0;
    }
    if constexpr (!TC)
        for (int i = tid; i < D * DV; i += kCkThreads) Hg[i] = Hs[i];
    float* sg = reinterpret_cast<float*>(rec + a.L.s);
    for (int i = tid; i < D; i += kCkThreads) sg[i] = ss[i];
    const T* Kin = static_cast<const T*>(a.K) + row0 * D;
    int32_t* cp = reinterpret_cast<int32_t*>(rec + a.L.c_pos);
    T* ck = reinterpret_cast<T*>(rec + a.L.c_k);
    T* cv = reinterpret_cast<T*>(rec + a.L.c_v);
    float* cph = reinterpret_cast<float*>(rec + a.L.c_phi);
    for (int i = tid; i < nc; i += kCkThreads) cp[i] = cpos[i];
    for (int i = tid; i < nc * D; i += kCkThreads) {
        const int sl = i / D, r = i % D;
        ck[(int64_t)sl * D + r] = Kin[(int64_t)cpos[sl] * D + r];
        cph[(int64_t)sl * D + r] = phiK[(int64_t)cpos[sl] * D + r];
    }
    for (int i = tid; i < nc * DV; i += kCkThreads) {
        const int sl = i / DV, q = i % DV;
        cv[(int64_t)sl * DV + q] = Vin[(int64_t)cpos[sl] * DV + q];
    }
    // the window after the last token: positions [(nch - nwc) C, n), entry p % eta
    const int wlo = max(0, (nch - a.nwc) * C);
    int32_t* wp = reinterpret_cast<int32_t*>(rec + a.L.win_pos);
    T* wk = reinterpret_cast<T*>(rec + a.L.win_k);
    T* wv = reinterpret_cast<T*>(rec + a.L.win_v);
    float* wph = reinterpret_cast<float*>(rec + a.L.win_phi);
    for (int p = wlo + tid; p < n; p += kCkThreads) {
        const int e = p % a.eta;
        wp[e] = p;
        for (int r = 0; r < D; ++r) {
            wk[(int64_t)e * D + r] = Kin[(int64_t)p * D + r];
            wph[(int64_t)e * D + r] = phiK[(int64_t)p * D + r];
        }
        for (int q = 0; q < DV; ++q) wv[(int64_t)e * DV + q] = Vin[(int64_t)p * DV + q];
    }
}

template <int D, int DV, typename T>
cudaError_t launch_chunk_t(const Dims& d, int n, const Workspace& ws, const void* K, const void* V, char* state,
                           const Layout& L, cudaStream_t st) {
    ChunkArgs a;
    a.n = n;
    a.eta = d.eta;
    a.lam = d.lam;
    a.C = d.chunk;
    a.nwc = d.eta / d.chunk;
    a.snap = ws.snap_interval;
    a.nck = ws.nck;
    a.phiK = ws.phiK;
    a.K = K;
    a.V = V;
    a.wstep = ws.wstep;
    a.wpos = ws.wpos;
    a.snapH = ws.snapH;
    a.snapHb = ws.snapHb;
    a.snapS = ws.snapS;
    a.snapC = ws.snapC;
    a.state = state;
    a.L = L;
    constexpr bool TC = sizeof(T) == 2 && D == 128 && DV == 128;
    const size_t smem = CkPlan<D, DV, TC>(d.lam, d.chunk).total;
    auto kern = chunk_select_kernel<D, DV, T, TC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<d.BH, kCkThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// SRE map (the notes' Fig. 3 diagnostic, section 4.4): CTA (c, bh) takes the memory the
// prefill snapshotted before step c * snap and the SRE of every key it holds (written
// before that step); the keys it does not hold read 0.  Same scoring routine as above.
// ---------------------------------------------------------------------------------
struct SreArgs {
    int n, snap, nck;
    const float* phiK;          // [BH][n][D]
    const void* V;              // io [BH][n][DV]
    const int32_t* wstep;       // [BH][n]
    const float* snapH;         // [BH][nck][D*DV] float32, or
    const __nv_bfloat16* snapHb;
    const float* snapS;         // [BH][nck][D]
    float* out;                 // [BH][nck][n]
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kCkThreads, 1) sre_map_kernel(const SreArgs a) {
    extern __shared__ __align__(16) unsigned char sm[];
    float* Hs = reinterpret_cast<float*>(sm);                           // [D][DV]
    float* tile = Hs + D * DV;                                           // [D][kTS]
    float* vts = tile + D * kTS;                                         // [kG][DV]
    float* ss = vts + kG * DV;                                           // [D]
    float* red = ss + D;                                                 // [9 kG]
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int n = a.n, tc = c * a.snap;
    const int64_t row0 = (int64_t)bh * n, sc = (int64_t)bh * a.nck + c;
    const float* phiK = a.phiK + row0 * D;
    const T* Vin = static_cast<const T*>(a.V) + row0 * DV;
    const int32_t* wst = a.wstep + row0;
    float* out = a.out + sc * n;
    for (int i = tid; i < D * DV; i += kCkThreads)
        Hs[i] = a.snapHb ? __bfloat162float(a.snapHb[sc * D * DV + i]) : a.snapH[sc * D * DV + i];
    for (int i = tid; i < D; i += kCkThreads) ss[i] = a.snapS[sc * D + i];
    for (int j = tc + tid; j < n; j += kCkThreads) out[j] = 0.f;   // not seen before step tc
    for (int j0 = 0; j0 < tc; j0 += kG) {
        const int cnt = min(kG, tc - j0);
        __syncthreads();   // H and s staged; the previous tile is consumed
        stage_rows<D, DV, T, true>(phiK, Vin, cnt, [&](int j) { return j0 + j; },
                                   [&](int j, int r) -> float& { return tile[r * kTS + j]; }, vts, tid);
        __syncthreads();
        tile_sre2<D, DV>(Hs, ss, tile, vts, red, cnt, warp, lane, [&](int j, float sre2) {
            const int w = wst[j0 + j];
            out[j0 + j] = (w >= 0 && w < tc) ? sqrtf(sre2) : 0.f;   // held by the memory, else 0
        });
    }
}

template <int D, int DV, typename T>
cudaError_t launch_sre_map_t(const Dims& d, int n, const Workspace& ws, const void* V, float* out, cudaStream_t st) {
    SreArgs a;
    a.n = n;
    a.snap = ws.snap_interval;
    a.nck = ws.nck;
    a.phiK = ws.phiK;
    a.V = V;
    a.wstep = ws.wstep;
    a.snapH = ws.snapH;
    a.snapHb = ws.snapHb;
    a.snapS = ws.snapS;
    a.out = out;
    const size_t smem = sizeof(float) * ((size_t)D * DV + D * kTS + kG * DV + D + 9 * kG);
    auto kern = sre_map_kernel<D, DV, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(ws.nck, d.BH), kCkThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sre_map(const Dims& d, int n, const Workspace& ws, const void* V, float* out, cudaStream_t st) {
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_sre_map_t<128, 128, __nv_bfloat16>(d, n, ws, V, out, st)
                  : launch_sre_map_t<128, 128, float>(d, n, ws, V, out, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_sre_map_t<64, 64, __nv_bfloat16>(d, n, ws, V, out, st)
                  : launch_sre_map_t<64, 64, float>(d, n, ws, V, out, st);
    return cudaErrorInvalidValue;
}

bool chunk_mode_fits(const Dims& d) {
    const bool bf = d.dtype == LOLA_BF16;
    const size_t smem = d.D == 128 ? (bf ? CkPlan<128, 128, true>(d.lam, d.chunk).total
                                         : CkPlan<128, 128, false>(d.lam, d.chunk).total)
                                   : CkPlan<64, 64, false>(d.lam, d.chunk).total;
    return smem <= 227 * 1024;
}

cudaError_t launch_chunk_select(const Dims& d, int n, const Workspace& ws, const void* K, const void* V,
                                char* state, const Layout& L, cudaStream_t st) {
    const bool bf = d.dtype == LOLA_BF16;
    if (d.D == 128 && d.dv == 128)
        return bf ? launch_chunk_t<128, 128, __nv_bfloat16>(d, n, ws, K, V, state, L, st)
                  : launch_chunk_t<128, 128, float>(d, n, ws, K, V, state, L, st);
    if (d.D == 64 && d.dv == 64)
        return bf ? launch_chunk_t<64, 64, __nv_bfloat16>(d, n, ws, K, V, state, L, st)
                  : launch_chunk_t<64, 64, float>(d, n, ws, K, V, state, L, st);
    return cudaErrorInvalidValue;
}

}  // namespace lola
