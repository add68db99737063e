/* Seeded synthetic inputs: SplitMix64 counter stream + Box-Muller normals.
 *
 * Number drawing only; none of the attention method's arithmetic lives here.
 * The word stream is the same as synth/generate.py's uniform_bits(): word i of
 * stream (seed, stream) is mix(key + (i + 1) * GOLDEN) with key derived from
 * (seed, stream).  Normal pair p uses words 2p and 2p + 1.
 *
 * Build: gcc -O2 -shared -fPIC -pthread synth_gen.c -o libsynth_gen.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * 0x100000001B3ULL + stream * 0x5851F42D4C957F2DULL + GOLDEN);
}

uint64_t synth_word(uint64_t seed, uint64_t stream, uint64_t i) {
    return mix64((i + 1) * GOLDEN + stream_key(seed, stream));
}

/* float32 -> bf16 word, round to nearest even (finite inputs) */
static inline uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += ((u >> 16) & 1u) + 0x7FFFu;
    return (uint16_t)(u >> 16);
}

typedef struct {
    uint64_t key;
    int64_t p0, p1;        /* pair range */
    int64_t count;         /* total values */
    double scale;
    int mode;              /* 0: double out, 1: float out, 2: bf16 out */
    void* out;
} job_t;

static void* run_job(void* arg) {
    job_t* j = (job_t*)arg;
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t p = j->p0; p < j->p1; ++p) {
        uint64_t a = mix64((uint64_t)(2 * p + 1) * GOLDEN + j->key);
        uint64_t b = mix64((uint64_t)(2 * p + 2) * GOLDEN + j->key);
        double u1 = ((double)(a >> 11) + 1.0) * (1.0 / 9007199254740992.0);
        double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
        double r = sqrt(-2.0 * log(u1));
        double ang = two_pi * u2;
        double z[2] = {r * cos(ang) * j->scale, r * sin(ang) * j->scale};
        for (int e = 0; e < 2; ++e) {
            int64_t idx = 2 * p + e;
            if (idx >= j->count) break;
            if (j->mode == 0) ((double*)j->out)[idx] = z[e];
            else if (j->mode == 1) ((float*)j->out)[idx] = (float)z[e];
            else ((uint16_t*)j->out)[idx] = f32_to_bf16((float)z[e]);
        }
    }
    return 0;
}

/* count normals of stream (seed, stream) times `scale`, written as double (mode 0),
 * float (mode 1) or bf16 words (mode 2), on up to nthreads threads. */
void synth_normal(uint64_t seed, uint64_t stream, int64_t count, double scale, int mode,
                  void* out, int nthreads) {
    if (count <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    int64_t npairs = (count + 1) / 2;
    if (npairs < 65536) nthreads = 1;
    pthread_t th[64];
    job_t jobs[64];
    uint64_t key = stream_key(seed, stream);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].key = key;
        jobs[t].p0 = npairs * t / nthreads;
        jobs[t].p1 = npairs * (t + 1) / nthreads;
        jobs[t].count = count;
        jobs[t].scale = scale;
        jobs[t].mode = mode;
        jobs[t].out = out;
        if (t > 0) pthread_create(&th[t], 0, run_job, &jobs[t]);
    }
    run_job(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], 0);
}

/* float32 array -> bf16 words (round to nearest even) */
void synth_to_bf16(const float* x, uint16_t* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = f32_to_bf16(x[i]);
}

/* Per-channel AR(1): x[r,0,c] = e[r,0,c];  x[r,t,c] = rho x[r,t-1,c] + sqrt(1-rho^2) e[r,t,c],
 * with e the normal stream (seed, stream) in row-major (rows, n, d) order.  The
 * recursion runs in double; the output is float32 (rows, n, d). */
typedef struct {
    uint64_t key;
    int64_t r0, r1, n, d;
    double rho;
    float* out;
} ar1_job_t;

static double normal_at(uint64_t key, int64_t idx) {
    const double two_pi = 6.283185307179586476925286766559;
    int64_t p = idx >> 1;
    uint64_t a = mix64((uint64_t)(2 * p + 1) * GOLDEN + key);
    uint64_t b = mix64((uint64_t)(2 * p + 2) * GOLDEN + key);
    double u1 = ((double)(a >> 11) + 1.0) * (1.0 / 9007199254740992.0);
    double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
    double r = sqrt(-2.0 * log(u1));
    return (idx & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static void* run_ar1(void* arg) {
    ar1_job_t* j = (ar1_job_t*)arg;
    double c = sqrt(1.0 - j->rho * j->rho);
    double x[1024];
    for (int64_t r = j->r0; r < j->r1; ++r) {
        for (int64_t t = 0; t < j->n; ++t) {
            int64_t base = (r * j->n + t) * j->d;
            for (int64_t ch = 0; ch < j->d; ++ch) {
                double e = normal_at(j->key, base + ch);
                x[ch] = (t == 0) ? e : j->rho * x[ch] + c * e;
                j->out[base + ch] = (float)x[ch];
            }
        }
    }
    return 0;
}

/* d <= 1024 */
void synth_ar1(uint64_t seed, uint64_t stream, int64_t rows, int64_t n, int64_t d, double rho,
               float* out, int nthreads) {
    if (rows <= 0 || n <= 0 || d <= 0 || d > 1024) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int)rows;
    if (nthreads > 64) nthreads = 64;
    pthread_t th[64];
    ar1_job_t jobs[64];
    uint64_t key = stream_key(seed, stream);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].key = key;
        jobs[t].r0 = rows * t / nthreads;
        jobs[t].r1 = rows * (t + 1) / nthreads;
        jobs[t].n = n;
        jobs[t].d = d;
        jobs[t].rho = rho;
        jobs[t].out = out;
        if (t > 0) pthread_create(&th[t], 0, run_ar1, &jobs[t]);
    }
    run_ar1(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], 0);
}
