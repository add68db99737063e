/* lola.h -- C ABI of the GB300 LoLA hybrid-attention library (liblola.so).
 *
 * The library computes, per attention head, the LoLA memory of "LoLA: Low-Rank Linear
 * Attention With Sparse Caching" (arXiv 2505.23666v3), reading notes sections 2.1-2.7:
 *   - a feature map phi(x) = [softmax(W x), softmax(-W x)], W of shape (D/2, d_k)
 *     (section 2.2, Eq. 3, in the configured form);
 *   - a linear memory H (D x d_v) and s (D) fed by H += phi(k) v^T, s += phi(k)
 *     (section 2.2, Eqs. 3-5) with only the KV assigned to it;
 *   - a sliding window of the eta most recent KV (the current token included) and a
 *     sparse cache of at most lambda exact KV;
 *   - per token: the KV leaving the window joins the cache as a candidate; when the
 *     candidates exceed lambda, the one with the smallest self-recall error
 *     SRE(k, v | H, s) = || H^T phi(k) / (phi(k)^T s) - v ||_2 (section 2.3, Eq. 10),
 *     scored against the memory before this step's write (section 2.4, Eqs. 11-13), is
 *     written into (H, s) and leaves the exact memory for good; ties go to the older
 *     token; an empty memory predicts 0, so SRE = ||v|| while s = 0;
 *   - the output y_t = (H^T phi(q) + sum_{G ∪ W} a v) / (phi(q)^T s + sum_{G ∪ W} a)
 *     with a = exp(q^T k / sqrt(d_k)), read after this step's write (section 2.5, Eq. 14).
 * The prefill chunk length only schedules the work: it never changes which KV are kept
 * (the per-token rule above is the definition).
 *
 * Conventions for every call:
 *   - Pointers marked "device" point to memory on the current CUDA device; "host" to
 *     host memory.  The library never allocates device memory in these calls: the caller
 *     owns every buffer (state, workspace, inputs, outputs).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  Host-side validation failures return at once
 *     with nothing enqueued.
 *   - Return values are lola_status codes.  LOLA_ERR_CUDA means a CUDA runtime call
 *     failed while enqueueing; the CUDA error text is available from
 *     lola_last_cuda_error().  Device-side anomalies (a chain whose bookkeeping went out
 *     of its bounds) are recorded in the per-head status word of the state and read
 *     with lola_read_status(); the kernels never trap.
 *   - Calls on distinct states may run concurrently; calls on one state must not overlap.
 *   - Tensors are dense row-major: Q, K, V and Y are [B, Hh, n, d] with d the innermost
 *     axis; per-head data of head (b, h) is at head index b * Hh + h.
 */
#ifndef LOLA_H
#define LOLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LOLA_OK = 0,
    LOLA_ERR_INVALID_ARG = -1,   /* null pointer, non-positive size, misaligned buffer */
    LOLA_ERR_UNSUPPORTED = -2,   /* valid but outside the shapes this build compiles */
    LOLA_ERR_WORKSPACE = -3,     /* workspace smaller than lola_prefill_workspace_bytes() */
    LOLA_ERR_CUDA = -4,          /* a CUDA runtime call failed */
    LOLA_ERR_DEVICE = -5         /* lola_read_status(): a head reported a device-side error */
} lola_status;

typedef enum {
    LOLA_F32 = 0,                /* Q, K, V, Y and the exact KV in float32 */
    LOLA_BF16 = 1                /* ... in bfloat16; H, s and all scores stay float32 */
} lola_dtype;

typedef struct {
    int32_t B;          /* batch */
    int32_t Hh;         /* heads per layer; every (b, h) is an independent memory */
    int32_t d_k;        /* query/key width */
    int32_t d_v;        /* value width */
    int32_t D;          /* feature width of phi; W has D/2 rows */
    int32_t eta;        /* window length (>= 0) */
    int32_t lambda;     /* sparse-cache capacity (>= 0) */
    int32_t chunk;      /* prefill schedule granularity C; no effect on results */
    int32_t dtype;      /* lola_dtype */
    int32_t read_mask;  /* 0, or lola_read_flags: memories left out of every query's read */
    int32_t alloc;      /* lola_alloc: LOLA_ALLOC_TOKEN (0, the default) or LOLA_ALLOC_CHUNK */
    int32_t score;      /* lola_score: LOLA_SCORE_SRE (0, the default) or a query-dependent score */
} lola_config;

/* Allocation granularity.  LOLA_ALLOC_TOKEN: the per-token rule (sections 2.3-2.4); the
 * chunk length only schedules the work.  LOLA_ALLOC_CHUNK (section 2.6, Eq. 15, the notes'
 * own prefill): the window is the last eta / chunk chunks, the current one included; each
 * chunk's queries read the state and cache it began with; as a chunk begins, the oldest
 * chunk of the previous window joins the cache, every candidate is scored against the
 * current state, the lambda highest-SRE stay and the rest are written at once.  Needs eta
 * a positive multiple of chunk and read_mask = 0; lola_prefill only (lola_decode_step
 * returns LOLA_ERR_UNSUPPORTED), and its write_pos log is per key: the chunk start at which
 * key j was written, -1 if never.  The exported state holds H, s, the cache positions and
 * rows and the window ring; the per-slot N, z and the next evictee's record stay zero.
 * Precision: with bfloat16 io at D = d_v = 128 the candidates' H^T phi and the written keys'
 * phi v^T are tensor-core products of bfloat16 hi + lo splits of the float32 operands (about
 * 2^-16 relative; H, s and z = s^T phi accumulate in float32), so a decision can differ from
 * an exact-arithmetic one only between candidates whose SREs agree to about that; float32 io
 * and D = 64 score and write in float32 on the CUDA cores. */
typedef enum { LOLA_ALLOC_TOKEN = 0, LOLA_ALLOC_CHUNK = 1 } lola_alloc;

/* Read mask (appendix I, Table 12: a read-time ablation).  The cache and the state are
 * updated exactly as with read_mask = 0 (same decisions, same memory); only the output
 * leaves out H^T phi(q), phi(q)^T s (HIDE_STATE) and/or the cached keys (HIDE_CACHE).  The
 * window is always read; a nonzero mask needs eta >= 1 (LOLA_ERR_INVALID_ARG otherwise). */
typedef enum { LOLA_READ_HIDE_STATE = 1, LOLA_READ_HIDE_CACHE = 2 } lola_read_flags;

/* Cache score (section 4.4, Table 4: the scoring ablation).  LOLA_SCORE_SRE: the self-recall
 * error, scored against the current memory at every eviction (sections 2.3-2.4).  The others
 * are query-dependent scores that a key collects while it is in the window: with
 * e = exp(q_t . k_j / sqrt(d_k)) and l = phi(q_t) . phi(k_j), summed over the eta queries of the
 * steps t = j .. j + eta - 1 -- (e - l)^2 (KERNEL_SQ), |e - l| (KERNEL_ABS), l / e
 * (KERNEL_RATIO), e (ATTENTION).  The score is complete when the key leaves the window and is
 * never updated: when the candidates exceed lambda the lowest (score, position) is written
 * (the older among equal scores), so the cache is the lambda highest-scored evicted keys.
 * Needs eta >= 1 and alloc = LOLA_ALLOC_TOKEN (else LOLA_ERR_INVALID_ARG); lola_prefill only
 * (lola_decode_step returns LOLA_ERR_UNSUPPORTED: the state keeps no window scores).  Scores
 * are summed in float32.  The exported state holds H, s, the cache positions and rows and the
 * window ring; the per-slot N, z and the next evictee's record stay zero. */
typedef enum {
    LOLA_SCORE_SRE = 0,
    LOLA_SCORE_KERNEL_SQ = 1,
    LOLA_SCORE_KERNEL_ABS = 2,
    LOLA_SCORE_KERNEL_RATIO = 3,
    LOLA_SCORE_ATTENTION = 4
} lola_score;

/* Supported by this build: d_k = d_v = D in {64, 128}; lambda <= 1024; eta <= 8192;
 * chunk a power of two in [16, 256]; B * Hh >= 1. */

/* ---- per-head state layout (the public "checkpoint" format) -----------------------
 * lola_state_bytes(cfg) = B * Hh * lola_head_state_bytes(cfg).  Head i's record starts
 * at byte i * lola_head_state_bytes(cfg).  Offsets below are from the record start and
 * are multiples of 256 bytes; io = float32 or bf16 per cfg->dtype.
 *   [0]        int32 header[16]: t (tokens consumed), n_cache (live cache entries),
 *              n_written, status (0 ok; nonzero = device-side error bits), rest 0
 *   H          float32 [D][d_v]          linear memory
 *   s          float32 [D]               normaliser
 *   win_pos    int32   [eta]             window ring: position p sits in entry p % eta
 *   win_k      io      [eta][d_k]
 *   win_v      io      [eta][d_v]
 *   win_phi    float32 [eta][D]          phi(k) of each window entry
 *   c_pos      int32   [lambda]          cache slots, -1 = empty; after lola_prefill the
 *                                        live slots come first, sorted by position;
 *                                        lola_decode_step reuses slots in place
 *   c_k        io      [lambda][d_k]
 *   c_v        io      [lambda][d_v]
 *   c_phi      float32 [lambda][D]       phi(k) of each cached key
 *   c_N        float32 [lambda][d_v]     H^T phi(k) kept current for each cached key
 *   c_z        float32 [lambda]          s^T phi(k) kept current for each cached key
 *   ev         float32 [d_v + 4]         the next evictee (token t - eta, eta > 0): its
 *                                        H^T phi(k) in [0, d_v) and s^T phi(k) at [d_v],
 *                                        both against the memory after token t - 1
 *   tok_phi    float32 [2][D]            scratch of lola_decode_step: phi(q), phi(k) of the
 *                                        token being decoded (no meaning between calls)
 * The appendix-B element count (eta + lambda)(d_k + d_v) + D d_v + D is the window,
 * cache, H and s above; win_phi, c_phi, c_N, c_z, ev, positions and the header are the
 * bookkeeping that lets a decode step score the cache without recomputing H^T phi(k). */

typedef struct {
    int64_t head_bytes;
    int64_t H, s, win_pos, win_k, win_v, win_phi, c_pos, c_k, c_v, c_phi, c_N, c_z, ev, tok_phi;
} lola_state_layout;

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t lola_version(void);

/* Static text for a lola_status value. */
const char* lola_status_string(int32_t status);

/* Text of the last CUDA error seen by the calling thread in this library ("" if none). */
const char* lola_last_cuda_error(void);

/* LOLA_OK if cfg is valid and supported, else LOLA_ERR_INVALID_ARG / LOLA_ERR_UNSUPPORTED. */
int32_t lola_check_config(const lola_config* cfg);

/* Fills *out with the per-head state layout (host). */
int32_t lola_state_layout_of(const lola_config* cfg, lola_state_layout* out);

/* Bytes of the whole state buffer (all B * Hh heads); 0 if cfg is invalid. */
size_t lola_state_bytes(const lola_config* cfg);

/* Bytes of device workspace lola_prefill needs for n tokens; 0 if invalid. */
size_t lola_prefill_workspace_bytes(const lola_config* cfg, int32_t n);

/* Resets every head of `state` (device, lola_state_bytes) to the empty memory: t = 0,
 * H = 0, s = 0, window and cache empty.  Stream-ordered. */
int32_t lola_state_init(const lola_config* cfg, void* state, void* stream);

/* Prefill: runs the per-token rule over n tokens of every head from the empty memory
 * (section 2.4, Eqs. 11-13; output section 2.5, Eq. 14).
 *   Q, K  device io [B, Hh, n, d_k];  V device io [B, Hh, n, d_v]
 *   W     device float32 [D/2, d_k] shared by all heads when w_head_stride == 0, else head
 *         h uses W + h * w_head_stride (elements; a multiple of 4, so that every head's W
 *         starts on a 16-byte boundary, else LOLA_ERR_INVALID_ARG)
 *   Y     device io [B, Hh, n, d_v]: the outputs y_0 .. y_{n-1}
 *   state device, lola_state_bytes(cfg): overwritten with the memory after token n-1,
 *         ready for lola_decode_step
 *   write_pos  nullable device int32 [B, Hh, n]: the position written into (H, s) at each
 *         step, or -1 when the step wrote nothing (the decision log)
 *   workspace  device, >= lola_prefill_workspace_bytes(cfg, n), 256-byte aligned
 * n >= 1.  Every device pointer must be 16-byte aligned.
 * Stream-ordered on `stream`: the call forks the feature map of the queries onto the
 * library's lower-priority side stream (it runs beside the selection chain) and joins it
 * back before the output pass, so all of the call's work precedes later work on `stream`.
 * The first call on a device (with that device current) creates that side stream and two
 * events, held until the process exits; make it before any stream capture starts. */
int32_t lola_prefill(const lola_config* cfg, int32_t n, const void* Q, const void* K,
                     const void* V, const float* W, int64_t w_head_stride, void* Y, void* state,
                     int32_t* write_pos, void* workspace, size_t workspace_bytes, void* stream);

/* One decode step for every head: token t = state.t with q, k, v (device io [B, Hh, d])
 * goes through the same rule as one prefill step; y (device io [B, Hh, d_v]) receives
 * its output; written_pos (nullable device int32 [B, Hh]) receives the position written
 * this step or -1.  W as in lola_prefill.  The state advances by one token.
 * For 1 <= eta <= 128, lambda <= 64 (and not float32 I/O at D = 128) the step is two kernels
 * on `stream`: the token's feature map (into the state's tok_phi scratch; traced as
 * LOLA_KERNEL_PHI), then the step itself as its programmatic dependent launch. */
int32_t lola_decode_step(const lola_config* cfg, void* state, const float* W,
                         int64_t w_head_stride, const void* q, const void* k, const void* v,
                         void* y, int32_t* written_pos, void* stream);

/* Synchronises `stream`, then copies the per-head status words into host_status (host
 * int32 [B * Hh], nullable).  Returns LOLA_OK if every head is 0, else LOLA_ERR_DEVICE. */
int32_t lola_read_status(const lola_config* cfg, const void* state, int32_t* host_status,
                         void* stream);

/* ---- prefill without a workspace argument ---------------------------------------------
 * No counterpart in the LoLA paper: this is an integration convenience of the library.
 *
 * For callers that cannot allocate device memory when they call in -- code hosted by a
 * runtime that owns the device allocator and fixes its budget at start-up, or a
 * latency-critical path that must not call cudaMalloc/cudaFree, which can synchronise the
 * whole device.  It computes exactly what lola_prefill computes, but its scratch memory is
 * a fixed array of LOLA_NOALLOC_SCRATCH_BYTES bytes inside the library's device image:
 *   - every device that loads the library holds that array until the process exits;
 *   - the call allocates nothing (no cudaMalloc, cudaFree or allocating library routine);
 *   - the first call on a device (with that device current) looks up the array's device
 *     address with cudaGetSymbolAddress and caches it, and (as lola_prefill's first call)
 *     creates the side stream and its two events; make that first call before any stream
 *     capture starts.  Both stay cached until the process exits, so cudaDeviceReset on that
 *     device after the first call is not supported;
 *   - all calls on a device share the one array and it keeps the last call's contents, so
 *     calls that overlap on the GPU (different streams, or different host threads, on the
 *     same device) race with each other: serialise them;
 *   - returns LOLA_ERR_WORKSPACE, with nothing enqueued, when
 *     lola_prefill_workspace_bytes(cfg, n) > LOLA_NOALLOC_SCRATCH_BYTES.
 * Arguments, outputs and errors are otherwise those of lola_prefill. */
#define LOLA_NOALLOC_SCRATCH_BYTES (32u << 20)

int32_t lola_prefill_noalloc(const lola_config* cfg, int32_t n, const void* Q, const void* K,
                             const void* V, const float* W, int64_t w_head_stride, void* Y,
                             void* state, int32_t* write_pos, void* stream);

/* ---- tracing: per-kernel device time of the library's own launches --------------------
 * When enabled, every kernel launch of lola_prefill / lola_decode_step / lola_state_init is
 * bracketed by two CUDA events on the stream it runs on (the call's stream; the side stream
 * for the queries' feature map, LOLA_KERNEL_PHI_Q, whose time then includes sharing the GPU
 * with the selection chain); a few microseconds of overhead per launch, no device memory.  Kernel ids: */
typedef enum {
    LOLA_KERNEL_STATE_INIT = 0,  /* state reset */
    LOLA_KERNEL_PHI = 1,         /* prefill: feature map of K; decode step: of the token's q, k */
    LOLA_KERNEL_SELECT = 2,      /* allocation chain: SRE scoring, argmin, (H, s) write */
    LOLA_KERNEL_OUTPUT = 3,      /* co-normalised output of every query */
    LOLA_KERNEL_DECODE = 4,      /* one decode step */
    LOLA_KERNEL_PHI_Q = 5,       /* prefill: feature map of Q (on the side stream) */
    LOLA_KERNEL_HOLA_PREP = 6,   /* write-magnitude cache layer: unit q, k tiles, RMS-scaled rows */
    LOLA_KERNEL_HOLA_STATE = 7,  /* ... the delta-rule state path (chunked, tensor cores), scores */
    LOLA_KERNEL_HOLA_CACHE = 8,  /* ... the persistent cache at every chunk start */
    LOLA_KERNEL_HOLA_READ = 9,   /* ... the cache read and the gated sum */
    LOLA_KERNEL_COUNT = 10
} lola_kernel_id;

/* enable != 0: clear the totals and start recording (process-wide); 0: stop recording. */
int32_t lola_kernel_timing(int32_t enable);

/* Waits for the recorded events of kernel `id`, then returns in *total_ms and *launches
 * the summed device time and number of launches recorded since lola_kernel_timing(1).
 * Either output may be NULL. */
int32_t lola_kernel_time(int32_t id, double* total_ms, int64_t* launches);

/* Static name of a kernel id ("" if out of range). */
const char* lola_kernel_name(int32_t id);

/* ---- SRE diagnostics ---------------------------------------------------------------------
 * Section 4.4 (the notes' Fig. 3): the self-recall error of every key the linear memory
 * holds, over state time.  Reads the snapshots that the last lola_prefill(cfg, n, ...) left
 * in `workspace` (same cfg and n, nothing written to it since): snapshot c is the memory
 * (H, s) before step c * P, P = max(chunk, 128), c < nck = ceil(n / P).
 *   V    device io [B, Hh, n, d_v]: the values given to that prefill
 *   out  device float32 [B, Hh, nck, n]: out[b, h, c, j] = SRE(k_j, v_j | H, s of snapshot
 *        c) = || H^T phi(k_j) / phi(k_j)^T s - v_j || if key j was written before step c * P,
 *        else 0 (the key is still exact, or not seen yet).  On the bf16 tensor-core path the
 *        snapshots of H are bf16 (rounded to nearest even), so the map carries that rounding.
 * Stream-ordered; validation errors return before anything is enqueued. */
int32_t lola_sre_map(const lola_config* cfg, int32_t n, const void* V, const void* workspace,
                     size_t workspace_bytes, float* out, void* stream);

/* The relative SRE map (appendix G, Fig. 10, Eq. 26): for each key a snapshot's memory holds,
 * its SRE against that memory minus its SRE against the first memory that held it.  Reads
 * the same workspace, cfg and n as lola_sre_map.
 *   out   device float32 [B, Hh, nck, n]: out[b, h, c, j] = SRE_c(j) - base[b, h, j] if key j
 *         was written before step c * P, else 0
 *   base  device float32 [B, Hh, n]: base[b, h, j] = SRE of key j against the memory right
 *         after its write step w_j (the sums over the keys written at or before w_j; in
 *         chunk-granular allocation every key written at that chunk start is included); 0 for
 *         keys never written.  Formed from the snapshot before j's interval plus the
 *         interval's writes up to w_j, so on the bf16 tensor-core path it carries the bf16
 *         rounding of that snapshot, like the map.
 * Stream-ordered; validation errors return before anything is enqueued. */
int32_t lola_sre_map_relative(const lola_config* cfg, int32_t n, const void* V, const void* workspace,
                              size_t workspace_bytes, float* out, float* base, void* stream);

/* ---- the write-magnitude exact cache on a gated delta-rule state --------------------------
 * "A Hippocampus for Linear Attention" (arXiv 2607.02303v1), reading notes, method sections
 * 3.1-3.5.  A sibling of the LoLA layer above with its own state: per head (b, h), S (d_k x d_v,
 * float32) starts at 0 and for t = 0 .. n-1
 *   k^ = k_t / ||k_t||, q^ = q_t / ||q_t||                          (state path: unit rows)
 *   e_t = v_t - alpha_t S^T k^,   S <- alpha_t S + beta_t k^ e_t^T    (Eq. 1, gated form of 3.5)
 *   m_t = beta_t ||e_t||                                             (Eqs. 5-6: write magnitude,
 *                                                                     fixed at the write)
 * The persistent cache of chunk c (queries [cC, cC + C)) is the w tokens j < cC with the
 * highest m_j (ties: the older token stays); the query reads it with its chunk's tokens up to
 * t and a null sink (logit sink[h], value 0):
 *   q~ = gamma_q * q / rms(q), k~ = gamma_k * k / rms(k), rms(x) = sqrt(mean(x^2) + 1e-6),
 *   o_t = softmax over {cache, chunk tokens <= t, sink} of q~ . k~ / sqrt(d_k), times v  (Eq. 7)
 *   y_t = S_t^T q^ + gate[h] * o_t                                   (section 3.2, Eq. 3)
 * Shapes this build compiles: bf16 Q, K, V, d_k = d_v = 128, 0 <= w <= 128, chunk a positive
 * multiple of 128 (at most 1024); else LOLA_ERR_UNSUPPORTED. */
typedef struct {
    int32_t B;       /* sequences */
    int32_t Hh;      /* heads per sequence */
    int32_t d_k;
    int32_t d_v;
    int32_t w;       /* persistent cache capacity */
    int32_t chunk;   /* C: the cache changes at multiples of C */
    int32_t dtype;   /* LOLA_BF16 */
} lola_hola_config;

/* Workspace bytes of one lola_hola_prefill over n tokens (negative: an invalid or
 * unsupported cfg, the lola_status code). */
int64_t lola_hola_workspace_bytes(const lola_hola_config* cfg, int32_t n);

/* One layer over n tokens of every head.  Device pointers, 16-byte aligned, caller-owned:
 *   Q, K, V   bf16 [B, Hh, n, d]            alpha, beta  float32 [B, Hh, n]  (decay in (0, 1],
 *                                                        write strength in [0, 1]; a decay
 *                                                        below 2^-100 is taken as 2^-100)
 *   gamma_q, gamma_k  float32 [d_k]         sink, gate   float32 [Hh]
 *   Y         bf16 [B, Hh, n, d_v] (out)
 *   S_out     float32 [B, Hh, d_k, d_v] (out, nullable): the state after token n - 1
 *   scores    float32 [B, Hh, n] (out, nullable): m_t
 *   cache     int32 [B, Hh, ceil(n / C), w] (out, nullable): the persistent cache's positions
 *             at every chunk start (unordered, -1 for empty entries)
 *   workspace at least lola_hola_workspace_bytes(cfg, n) bytes (it holds the same scores and
 *             cache lists when those outputs are null, and the per-head status words).
 * Stream-ordered on `stream`; validation errors return before anything is enqueued.  A bounded
 * wait of the state or read kernel that gives up sets ST-timeout bits readable with
 * lola_hola_status. */
int32_t lola_hola_prefill(const lola_hola_config* cfg, int32_t n, const void* Q, const void* K, const void* V,
                          const float* alpha, const float* beta, const float* gamma_q, const float* gamma_k,
                          const float* sink, const float* gate, void* Y, float* S_out, float* scores,
                          int32_t* cache, void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream` and copies the per-head status words of the last lola_hola_prefill
 * in `workspace` (same cfg, n) to host_status (int32 [B * Hh], nullable).  LOLA_OK if every
 * head is 0, else LOLA_ERR_DEVICE. */
int32_t lola_hola_status(const lola_hola_config* cfg, int32_t n, const void* workspace, int32_t* host_status,
                         void* stream);

/* ---- self-test of the bounded waits -----------------------------------------------------
 * No counterpart in the LoLA paper.  Every wait of the library's kernels on an mbarrier (the
 * decode step's burst, the output pass's MMA groups) gives up after a time limit, records a
 * status bit and returns, so that the CUDA context stays usable.  This call runs that same
 * wait on an mbarrier that nothing completes: one thread waits limit_ns nanoseconds
 * (1 .. 10^9) and *host_elapsed_ns (host, nullable) receives how long it waited.  Synchronises
 * `stream`; not for concurrent use.  Returns LOLA_ERR_DEVICE when the wait gave up as designed,
 * LOLA_OK if it returned without giving up (a defect), LOLA_ERR_INVALID_ARG for a limit outside
 * the range (before anything is enqueued), LOLA_ERR_CUDA on a CUDA failure. */
int32_t lola_selftest_bounded_wait(int64_t limit_ns, int64_t* host_elapsed_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LOLA_H */
