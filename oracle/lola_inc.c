/* CPU float64 oracle for LoLA hybrid attention, incremental form.
 * TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU-baseline
 * leg call it; the CUDA library never does and shares no code with it.
 *
 * Source: "LoLA: Low-Rank Linear Attention With Sparse Caching" (arXiv 2505.23666v3),
 * reading notes sections 2.2-2.5 (Eqs. 3-5, 10, 11-13, 14).  The rule executed per
 * token t of one head is the one stated in oracle/lola_ref.py:
 *   1. phi(q_t); the window gains t; if it holds more than eta tokens, t - eta leaves
 *      and joins the candidate set E = G ∪ {t - eta} (for eta = 0, t itself);
 *   2. if |E| <= lambda all candidates stay in the cache G; otherwise each candidate's
 *      SRE is taken against (H, s) before this step's write, the smallest (ties: the
 *      older position) is written H += phi(k)v^T, s += phi(k), and the rest stay;
 *   3. y_t is the co-normalised read over window, cache and (H, s) after the write.
 *      The read mask (the notes' appendix I ablation, Table 12: the cache and the state
 *      are updated as always, only what the query reads is restricted) drops the state's
 *      terms (bit 0) and/or the cache's keys (bit 1) from the read; the window is always
 *      read.
 *
 * Incremental form: instead of recomputing H^T phi(k_c) for every candidate c at every
 * step, each cached candidate keeps N_c = H^T phi(k_c) and z_c = s^T phi(k_c), set when
 * it enters the candidate set and moved with every later write w by
 *   g = phi(k_w)^T phi(k_c),  N_c += g v_w,  z_c += g,
 * which is exact in real arithmetic because each write changes H by the rank-1 term
 * phi(k_w) v_w^T.  SRE_c^2 = || N_c / z_c - v_c ||^2, or ||v_c||^2 when z_c = 0 (the
 * empty-memory reading).
 *
 * Replay: given the position written at every step by some other implementation, the
 * oracle follows those writes, checks that each is a candidate and that writes happen
 * exactly at the due steps, and records the relative SRE gap of each decision to its
 * own best candidate.
 *
 * Build: gcc -O2 -shared -fPIC -pthread lola_inc.c -o liblola_oracle.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { IN_F32 = 0, IN_BF16 = 1 };

typedef struct {
    int BH, n, dk, dv, D, eta, lam, in_dtype;
    const void *Q, *K, *V;       /* [BH, n, dk|dv] float32 or bf16 words */
    const float* W;              /* [D/2, dk] */
    const int32_t* replay;       /* nullable [BH, n] */
    double* Y;                   /* [BH, n, dv] */
    int32_t* write_pos;          /* [BH, n] */
    int32_t* write_step;         /* [BH, n] */
    double* H_out;               /* nullable [BH, D*dv] */
    double* s_out;               /* nullable [BH, D] */
    int32_t* cache_out;          /* nullable [BH, lam] sorted, -1 padded */
    double* stats;               /* [BH, 4]: min_gap, max_gap, mismatches, status */
    int next;                    /* work counter */
    int read_mask;               /* bit 0: the state is not read; bit 1: the cache is not read */
} job_t;

static double widen(const void* base, int dtype, size_t idx) {
    if (dtype == IN_BF16) {
        uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* phi(x) = [softmax(Wx), softmax(-Wx)], max-subtracted, float64 */
static void feature(const double* x, const double* W, int dk, int D, double* out, double* z) {
    int h = D / 2;
    for (int r = 0; r < h; ++r) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += W[(size_t)r * dk + c] * x[c];
        z[r] = acc;
    }
    for (int sign = 0; sign < 2; ++sign) {
        double mx = -INFINITY, sum = 0.0;
        for (int r = 0; r < h; ++r) {
            double zz = sign ? -z[r] : z[r];
            if (zz > mx) mx = zz;
        }
        for (int r = 0; r < h; ++r) {
            double zz = sign ? -z[r] : z[r];
            double e = exp(zz - mx);
            out[sign * h + r] = e;
            sum += e;
        }
        for (int r = 0; r < h; ++r) out[sign * h + r] /= sum;
    }
}

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

static void run_chain(job_t* J, int bh) {
    const int n = J->n, dk = J->dk, dv = J->dv, D = J->D, eta = J->eta, lam = J->lam;
    const int cap = lam + 1;
    const double scale = 1.0 / sqrt((double)dk);
    double* W = malloc(sizeof(double) * (size_t)(D / 2) * dk);
    for (size_t i = 0; i < (size_t)(D / 2) * dk; ++i) W[i] = J->W[i];
    double* H = calloc((size_t)D * dv, sizeof(double));
    double* s = calloc(D, sizeof(double));
    int32_t* cpos = malloc(sizeof(int32_t) * cap);
    double* cN = malloc(sizeof(double) * (size_t)cap * dv);
    double* cz = malloc(sizeof(double) * cap);
    double* cphi = malloc(sizeof(double) * (size_t)cap * D);
    double* cv = malloc(sizeof(double) * (size_t)cap * dv);
    double* sq = malloc(sizeof(double) * cap);
    double *x = malloc(sizeof(double) * dk), *z = malloc(sizeof(double) * D);
    double *phiq = malloc(sizeof(double) * D), *hq = malloc(sizeof(double) * dv);
    double* num = malloc(sizeof(double) * dv);
    double* ascore = malloc(sizeof(double) * (size_t)(eta + cap));
    int count = 0;
    double min_gap = INFINITY, max_gap = 0.0, mismatches = 0.0, status = 0.0;
    const size_t base_k = (size_t)bh * n * dk, base_v = (size_t)bh * n * dv;
    int32_t* wpos = J->write_pos + (size_t)bh * n;
    int32_t* wstep = J->write_step + (size_t)bh * n;
    const int32_t* rep = J->replay ? J->replay + (size_t)bh * n : NULL;
    for (int t = 0; t < n; ++t) wpos[t] = wstep[t] = -1;

    for (int t = 0; t < n && status == 0.0; ++t) {
        /* 1. the evictee (if any) joins the candidates with N = H^T phi, z = s^T phi */
        if (t >= eta) {
            int e = t - eta;
            for (int c = 0; c < dk; ++c) x[c] = widen(J->K, J->in_dtype, base_k + (size_t)e * dk + c);
            double* ph = cphi + (size_t)count * D;
            feature(x, W, dk, D, ph, z);
            double* Ne = cN + (size_t)count * dv;
            for (int j = 0; j < dv; ++j) Ne[j] = 0.0;
            double ze = 0.0;
            for (int r = 0; r < D; ++r) {
                const double* Hr = H + (size_t)r * dv;
                for (int j = 0; j < dv; ++j) Ne[j] += ph[r] * Hr[j];
                ze += ph[r] * s[r];
            }
            cz[count] = ze;
            for (int j = 0; j < dv; ++j) cv[(size_t)count * dv + j] = widen(J->V, J->in_dtype, base_v + (size_t)e * dv + j);
            cpos[count] = e;
            count++;
        }
        /* 2. decision when the candidates exceed the cache capacity */
        if (count > lam) {
            int best = -1, second = -1;
            for (int i = 0; i < count; ++i) {
                const double* vi = cv + (size_t)i * dv;
                double acc = 0.0;
                if (cz[i] == 0.0) {
                    for (int j = 0; j < dv; ++j) acc += vi[j] * vi[j];
                } else {
                    const double* Ni = cN + (size_t)i * dv;
                    for (int j = 0; j < dv; ++j) {
                        double r = Ni[j] / cz[i] - vi[j];
                        acc += r * r;
                    }
                }
                sq[i] = acc;
            }
            for (int i = 0; i < count; ++i)
                if (best < 0 || sq[i] < sq[best] || (sq[i] == sq[best] && cpos[i] < cpos[best])) best = i;
            for (int i = 0; i < count; ++i)
                if (i != best && (second < 0 || sq[i] < sq[second] || (sq[i] == sq[second] && cpos[i] < cpos[second])))
                    second = i;
            if (second >= 0) {
                double sb = sqrt(sq[best]), s2 = sqrt(sq[second]);
                double gap = sb > 0 ? (s2 - sb) / sb : (s2 > 0 ? INFINITY : 0.0);
                if (gap < min_gap) min_gap = gap;
            }
            int w = best;
            if (rep) {
                w = -1;
                for (int i = 0; i < count; ++i)
                    if (cpos[i] == rep[t]) w = i;
                if (w < 0) { status = 1.0; break; }   /* replayed write is not a candidate */
                if (w != best) {
                    mismatches += 1.0;
                    double sb = sqrt(sq[best]), sw = sqrt(sq[w]);
                    double gap = sb > 0 ? (sw - sb) / sb : (sw > 0 ? INFINITY : 0.0);
                    if (gap > max_gap) max_gap = gap;
                }
            }
            const double* pw = cphi + (size_t)w * D;
            const double* vw = cv + (size_t)w * dv;
            for (int r = 0; r < D; ++r) {
                double* Hr = H + (size_t)r * dv;
                for (int j = 0; j < dv; ++j) Hr[j] += pw[r] * vw[j];
                s[r] += pw[r];
            }
            for (int i = 0; i < count; ++i) {
                if (i == w) continue;
                const double* pi = cphi + (size_t)i * D;
                double g = 0.0;
                for (int r = 0; r < D; ++r) g += pw[r] * pi[r];
                double* Ni = cN + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) Ni[j] += g * vw[j];
                cz[i] += g;
            }
            wpos[t] = cpos[w];
            wstep[cpos[w]] = t;
            /* remove w: move the last candidate into its place */
            int last = count - 1;
            if (w != last) {
                cpos[w] = cpos[last];
                cz[w] = cz[last];
                memcpy(cN + (size_t)w * dv, cN + (size_t)last * dv, sizeof(double) * dv);
                memcpy(cv + (size_t)w * dv, cv + (size_t)last * dv, sizeof(double) * dv);
                memcpy(cphi + (size_t)w * D, cphi + (size_t)last * D, sizeof(double) * D);
            }
            count--;
        } else if (rep && rep[t] != -1) {
            status = 2.0;    /* replay writes when no write is due */
            break;
        }
        /* 3. co-normalised output over window ∪ cache ∪ (H, s), less what the read mask hides */
        const int ncache_read = (J->read_mask & 2) ? 0 : count;
        const int read_state = !(J->read_mask & 1);
        for (int c = 0; c < dk; ++c) x[c] = widen(J->Q, J->in_dtype, base_k + (size_t)t * dk + c);
        feature(x, W, dk, D, phiq, z);
        int w0 = t - eta + 1 < 0 ? 0 : t - eta + 1;
        int nex = 0;
        double m = -INFINITY;
        for (int pass = 0; pass < 2; ++pass) {
            int cnt = pass == 0 ? (t - w0 + 1) : ncache_read;
            for (int i = 0; i < cnt; ++i) {
                int p = pass == 0 ? w0 + i : cpos[i];
                double a = 0.0;
                for (int c = 0; c < dk; ++c) a += x[c] * widen(J->K, J->in_dtype, base_k + (size_t)p * dk + c);
                a *= scale;
                ascore[nex++] = a;
                if (a > m) m = a;
            }
        }
        for (int j = 0; j < dv; ++j) hq[j] = 0.0;
        double dl = 0.0;
        for (int r = 0; r < D; ++r) {
            const double* Hr = H + (size_t)r * dv;
            for (int j = 0; j < dv; ++j) hq[j] += phiq[r] * Hr[j];
            dl += phiq[r] * s[r];
        }
        double em = nex > 0 ? exp(-m) : 1.0, den = read_state ? em * dl : 0.0;
        for (int j = 0; j < dv; ++j) num[j] = read_state ? em * hq[j] : 0.0;
        nex = 0;
        for (int pass = 0; pass < 2; ++pass) {
            int cnt = pass == 0 ? (t - w0 + 1) : ncache_read;
            for (int i = 0; i < cnt; ++i) {
                int p = pass == 0 ? w0 + i : cpos[i];
                double wgt = exp(ascore[nex++] - m);
                den += wgt;
                for (int j = 0; j < dv; ++j) num[j] += wgt * widen(J->V, J->in_dtype, base_v + (size_t)p * dv + j);
            }
        }
        double* y = J->Y + base_v + (size_t)t * dv;
        for (int j = 0; j < dv; ++j) y[j] = num[j] / den;
    }
    if (J->H_out) memcpy(J->H_out + (size_t)bh * D * dv, H, sizeof(double) * (size_t)D * dv);
    if (J->s_out) memcpy(J->s_out + (size_t)bh * D, s, sizeof(double) * D);
    if (J->cache_out) {
        int32_t* co = J->cache_out + (size_t)bh * lam;
        for (int i = 0; i < lam; ++i) co[i] = i < count ? cpos[i] : -1;
        qsort(co, count < lam ? count : lam, sizeof(int32_t), cmp_i32);
    }
    J->stats[(size_t)bh * 4 + 0] = min_gap;
    J->stats[(size_t)bh * 4 + 1] = max_gap;
    J->stats[(size_t)bh * 4 + 2] = mismatches;
    J->stats[(size_t)bh * 4 + 3] = status;
    free(W); free(H); free(s); free(cpos); free(cN); free(cz); free(cphi); free(cv); free(sq);
    free(x); free(z); free(phiq); free(hq); free(num); free(ascore);
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    for (;;) {
        int bh = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (bh >= J->BH) break;
        run_chain(J, bh);
    }
    return 0;
}

/* Runs BH independent heads.  Returns 0, or -1 on invalid sizes or a read mask that
 * leaves nothing to read (any nonzero mask needs eta >= 1: the window then always holds
 * the current token). */
int lola_oracle_run(int BH, int n, int dk, int dv, int D, int eta, int lam, int in_dtype,
                    const void* Q, const void* K, const void* V, const float* W,
                    const int32_t* replay, double* Y, int32_t* write_pos, int32_t* write_step,
                    double* H_out, double* s_out, int32_t* cache_out, double* stats, int nthreads,
                    int read_mask) {
    if (BH < 0 || n < 0 || dk <= 0 || dv <= 0 || D <= 0 || (D & 1) || eta < 0 || lam < 0) return -1;
    if (read_mask < 0 || read_mask > 3 || (read_mask != 0 && eta < 1)) return -1;
    job_t J = {BH, n, dk, dv, D, eta, lam, in_dtype, Q, K, V, W, replay, Y, write_pos, write_step,
               H_out, s_out, cache_out, stats, 0, read_mask};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > BH) nthreads = BH > 0 ? BH : 1;
    pthread_t th[256];
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], 0, worker, &J);
    worker(&J);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], 0);
    return 0;
}
