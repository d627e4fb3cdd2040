/*
 * dspark_oracle.c -- plain CPU oracle for one DSpark decoding cycle.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no
 * code, header or table with the CUDA library.
 *
 * Every step is written in the order the pages give it, in double precision,
 * with no blocking or fusion.  The only parallelism is across requests,
 * which the method treats independently.
 *
 * Readings taken where the pages leave a step open:
 *  - temperature T divides both the draft logits (U + B) and the target
 *    logits P; T = 0 means greedy (argmax, lowest index on ties);
 *  - the draft samples by Gumbel-max with G = -ln(-ln u);
 *  - the residual and the bonus token are drawn by inverse CDF taken level by
 *    level down a binary sum tree over the vocabulary, one fresh uniform per
 *    level (each level is a two-way inverse CDF);
 *  - acceptance is u < p(x)/q(x) (so ratio >= 1 always accepts);
 *  - an empty residual (possible only through rounding) falls back to p.
 */
#include "dspark_oracle.h"

/* Width of the chunks of the draft's two-level Gumbel-max. */
#define ORACLE_DRAFT_CHUNK 256

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11, section 3.3 and Table 2).       */
/* ------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;   /* round multipliers */
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;   /* Weyl key increments */
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * (uint64_t)x0;
        uint64_t p1 = (uint64_t)M1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double oracle_uniform(uint32_t w) {
    return ((double)w + 0.5) * (1.0 / 4294967296.0);   /* (w + 1/2) 2^-32 */
}

/* Counter (v/4, request, position, stream), key (seed lo, seed hi); the
 * uniform for index v is output word v mod 4. */
double oracle_rng_uniform(uint64_t seed, uint32_t req, uint32_t pos, uint32_t stream, uint32_t v) {
    uint32_t ctr[4] = {v >> 2, req, pos, stream};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return oracle_uniform(out[v & 3u]);
}

/* ------------------------------------------------------------------ */
/* Input widening.                                                      */
/* ------------------------------------------------------------------ */
static double ld(const void* p, int dtype, size_t i) {
    if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Explainer section 05: acceptance and residual.                        */
/* ------------------------------------------------------------------ */
double oracle_accept_prob(double px, double qx) {
    double ratio = px / qx;
    return ratio < 1.0 ? ratio : 1.0;
}

void oracle_residual_weights(const double* p, const double* q, int V, double* w) {
    for (int v = 0; v < V; ++v) {
        double d = p[v] - q[v];
        w[v] = d > 0.0 ? d : 0.0;
    }
}

static int ceil_log2(int V) {
    int L = 0;
    while ((1 << L) < V) ++L;
    return L;
}

static double range_sum(const double* w, int V, long lo, long hi) {
    double s = 0.0;
    if (hi > V) hi = V;
    for (long v = lo; v < hi; ++v) s += w[v];
    return s;
}

int oracle_tree_sample(const double* w, int V, uint64_t seed, uint32_t req, uint32_t pos, double* min_gap) {
    int L = ceil_log2(V);
    long lo = 0;
    double gap = INFINITY;
    for (int d = 0; d < L; ++d) {
        long half = 1L << (L - d - 1);
        long mid = lo + half;
        double mL = range_sum(w, V, lo, mid);
        double mR = range_sum(w, V, mid, mid + half);
        double u = oracle_rng_uniform(seed, req, pos, 2u, (uint32_t)d);
        double thr = mL / (mL + mR);
        double g = fabs(u - thr);
        if (g < gap) gap = g;
        if (u * (mL + mR) < mL) {
            /* left child: lo stays */
        } else {
            lo = mid;
        }
    }
    if (min_gap) *min_gap = gap;
    return (int)lo;
}

/* ------------------------------------------------------------------ */
/* Drafting: the sequential stage (blog section 3.2).                    */
/* ------------------------------------------------------------------ */
typedef struct {
    /* shared read-only inputs */
    const void *U, *W1, *W2, *Wgco, *H;
    int u_dtype, w_dtype, h_dtype;
    const int32_t* anchor;
    int R, gamma, V, r, d, rnn;
    uint64_t seed;
    const uint32_t* req_ids;
    double T;
    /* outputs */
    int32_t* tokens;
    double *qx, *lse, *code, *margin, *state_out;
    /* work split */
    int r_begin, r_end;
    int status;
} draft_job;

/* One position of the draft for one request: logits z = (U_k + B_k)/T,
 * log-sum-exp, Gumbel-max sample (or argmax at T = 0). */
static void draft_position(const draft_job* J, int ri, int k, const double* B,
                           double* z, int32_t* x_out, double* qx_out, double* lse_out, double* margin_out) {
    const int V = J->V;
    const size_t urow = ((size_t)ri * J->gamma + (size_t)(k - 1)) * (size_t)V;
    uint32_t req = J->req_ids ? J->req_ids[ri] : (uint32_t)ri;
    if (J->T > 0.0) {
        for (int v = 0; v < V; ++v) z[v] = (ld(J->U, J->u_dtype, urow + v) + B[v]) / J->T;
        double m = -INFINITY;
        for (int v = 0; v < V; ++v) if (z[v] > m) m = z[v];
        double s = 0.0;
        for (int v = 0; v < V; ++v) s += exp(z[v] - m);
        double lse = m + log(s);
        /* Gumbel-max in two levels (an exact sampler of softmax(z)):
         * (1) over the chunks of 256 consecutive indices, with key
         *     ln(sum_{v in c} e^{z_v}) + G_c (stream 3, index c);
         * (2) inside the chosen chunk, with key z_v + G_v (stream 0, index v).
         * G = -ln(-ln u).  Ties go to the lowest index at both levels. */
        const int C = ORACLE_DRAFT_CHUNK;
        const int nC = (V + C - 1) / C;
        uint32_t key[2] = {(uint32_t)(J->seed & 0xFFFFFFFFu), (uint32_t)(J->seed >> 32)};
        double cbest = -INFINITY, csecond = -INFINITY;
        int carg = 0;
        for (int c = 0; c < nC; ++c) {
            double mass = 0.0;
            int hi = (c + 1) * C < V ? (c + 1) * C : V;
            for (int v = c * C; v < hi; ++v) mass += exp(z[v] - m);
            double u = oracle_rng_uniform(J->seed, req, (uint32_t)k, 3u, (uint32_t)c);
            double kc = (log(mass) + m) - log(-log(u));
            if (kc > cbest) { csecond = cbest; cbest = kc; carg = c; }
            else if (kc > csecond) { csecond = kc; }
        }
        double best = -INFINITY, second = -INFINITY;
        int arg = -1;
        uint32_t words[4];
        int hi = (carg + 1) * C < V ? (carg + 1) * C : V;
        for (int v = carg * C; v < hi; ++v) {
            if ((v & 3) == 0) {
                uint32_t ctr[4] = {(uint32_t)v >> 2, req, (uint32_t)k, 0u};
                oracle_philox4x32_10(ctr, key, words);
            }
            double u = oracle_uniform(words[v & 3]);
            double g = -log(-log(u));
            double kv = z[v] + g;
            if (kv > best) { second = best; best = kv; arg = v; }
            else if (kv > second) { second = kv; }
        }
        *x_out = arg;
        *qx_out = exp(z[arg] - lse);
        *lse_out = lse;
        double m1 = cbest - csecond, m2 = best - second;
        *margin_out = m1 < m2 ? m1 : m2;
    } else {
        double best = -INFINITY, second = -INFINITY;
        int arg = -1;
        for (int v = 0; v < V; ++v) {
            double y = ld(J->U, J->u_dtype, urow + v) + B[v];
            if (y > best) { second = best; best = y; arg = v; }
            else if (y > second) { second = y; }
        }
        *x_out = arg;
        *qx_out = 1.0;          /* the greedy draft is a point mass */
        *lse_out = 0.0;
        *margin_out = best - second;
    }
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void* draft_worker(void* arg) {
    draft_job* J = (draft_job*)arg;
    const int V = J->V, r = J->r, gamma = J->gamma;
    double* B = (double*)malloc(sizeof(double) * (size_t)V);
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* e = (double*)malloc(sizeof(double) * (size_t)r);
    double* s = (double*)calloc((size_t)r, sizeof(double));
    double* zin = NULL;
    double* G = NULL;
    if (J->rnn) {
        zin = (double*)malloc(sizeof(double) * (size_t)(2 * r + J->d));
        G = (double*)malloc(sizeof(double) * (size_t)(3 * r));
    }
    if (!B || !z || !e || !s || (J->rnn && (!zin || !G))) { J->status = -1; goto done; }
    for (int ri = J->r_begin; ri < J->r_end; ++ri) {
        int prev = J->anchor[ri];                 /* x_0 = anchor */
        if (prev < 0 || prev >= V) { J->status = -6; goto done; }
        memset(s, 0, sizeof(double) * (size_t)r);  /* s_0 = 0 */
        for (int k = 1; k <= gamma; ++k) {
            if (!J->rnn) {
                /* Markov head: e = W1[x_{k-1}] */
                for (int i = 0; i < r; ++i) e[i] = ld(J->W1, J->w_dtype, (size_t)prev * r + i);
            } else {
                /* RNN head: z = [s_{k-1}, W1[x_{k-1}], h_k]; G = z Wgco;
                 * g = sigmoid(G_gate); s_k = g s_{k-1} + (1-g) tanh(G_cand);
                 * e = tanh(G_out). */
                const int D = J->d, Kin = 2 * r + D;
                for (int i = 0; i < r; ++i) zin[i] = s[i];
                for (int i = 0; i < r; ++i) zin[r + i] = ld(J->W1, J->w_dtype, (size_t)prev * r + i);
                for (int i = 0; i < D; ++i)
                    zin[2 * r + i] = ld(J->H, J->h_dtype, ((size_t)ri * gamma + (size_t)(k - 1)) * D + i);
                for (int j = 0; j < 3 * r; ++j) G[j] = 0.0;
                for (int i = 0; i < Kin; ++i) {
                    double zi = zin[i];
                    for (int j = 0; j < 3 * r; ++j) G[j] += zi * ld(J->Wgco, J->w_dtype, (size_t)i * 3 * r + j);
                }
                for (int i = 0; i < r; ++i) {
                    double g = sigmoid(G[i]);
                    s[i] = g * s[i] + (1.0 - g) * tanh(G[r + i]);
                    e[i] = tanh(G[2 * r + i]);
                }
            }
            /* B = e W2 (row i of W2 is scaled by e_i and accumulated). */
            for (int v = 0; v < V; ++v) B[v] = 0.0;
            for (int i = 0; i < r; ++i) {
                double ei = e[i];
                size_t row = (size_t)i * V;
                for (int v = 0; v < V; ++v) B[v] += ei * ld(J->W2, J->w_dtype, row + v);
            }
            size_t o = (size_t)ri * gamma + (size_t)(k - 1);
            int32_t x;
            draft_position(J, ri, k, B, z, &x, &J->qx[o], &J->lse[o], &J->margin[o]);
            J->tokens[o] = x;
            for (int i = 0; i < r; ++i) J->code[o * r + i] = e[i];
            prev = x;                               /* the next step sees x_k */
        }
        if (J->rnn && J->state_out)
            for (int i = 0; i < r; ++i) J->state_out[(size_t)ri * r + i] = s[i];
    }
done:
    free(B); free(z); free(e); free(s); free(zin); free(G);
    return NULL;
}

static int run_jobs(void* jobs, size_t job_size, int n, void* (*fn)(void*)) {
    if (n <= 1) {
        fn(jobs);
        return 0;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n);
    int* started = (int*)calloc((size_t)n, sizeof(int));
    if (!th || !started) { free(th); free(started); return -1; }
    for (int i = 0; i < n; ++i) {
        void* job = (char*)jobs + (size_t)i * job_size;
        if (pthread_create(&th[i], NULL, fn, job) == 0) started[i] = 1;
        else fn(job);
    }
    for (int i = 0; i < n; ++i) if (started[i]) pthread_join(th[i], NULL);
    free(th); free(started);
    return 0;
}

static int draft_common(draft_job* proto, int n_threads) {
    if (proto->R <= 0 || proto->gamma <= 0 || proto->V <= 0 || proto->r <= 0) return -3;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > proto->R) n_threads = proto->R;
    draft_job* jobs = (draft_job*)calloc((size_t)n_threads, sizeof(draft_job));
    if (!jobs) return -1;
    for (int t = 0; t < n_threads; ++t) {
        jobs[t] = *proto;
        jobs[t].r_begin = (int)((long)proto->R * t / n_threads);
        jobs[t].r_end = (int)((long)proto->R * (t + 1) / n_threads);
        jobs[t].status = 0;
    }
    run_jobs(jobs, sizeof(draft_job), n_threads, draft_worker);
    int st = 0;
    for (int t = 0; t < n_threads; ++t) if (jobs[t].status) st = jobs[t].status;
    free(jobs);
    return st;
}

int oracle_draft_markov(const void* U, int u_dtype, const int32_t* anchor,
                        const void* W1, const void* W2, int w_dtype,
                        int R, int gamma, int V, int r,
                        uint64_t seed, const uint32_t* req_ids, double T,
                        int32_t* tokens, double* qx, double* lse, double* code,
                        double* margin, int n_threads) {
    draft_job J;
    memset(&J, 0, sizeof J);
    J.U = U; J.W1 = W1; J.W2 = W2; J.u_dtype = u_dtype; J.w_dtype = w_dtype;
    J.anchor = anchor; J.R = R; J.gamma = gamma; J.V = V; J.r = r; J.rnn = 0;
    J.seed = seed; J.req_ids = req_ids; J.T = T;
    J.tokens = tokens; J.qx = qx; J.lse = lse; J.code = code; J.margin = margin;
    return draft_common(&J, n_threads);
}

int oracle_draft_rnn(const void* U, int u_dtype, const int32_t* anchor,
                     const void* W1, const void* W2, const void* Wgco, int w_dtype,
                     const void* H, int h_dtype,
                     int R, int gamma, int V, int r, int d,
                     uint64_t seed, const uint32_t* req_ids, double T,
                     int32_t* tokens, double* qx, double* lse, double* code,
                     double* margin, double* state_out, int n_threads) {
    if (d <= 0) return -3;
    draft_job J;
    memset(&J, 0, sizeof J);
    J.U = U; J.W1 = W1; J.W2 = W2; J.Wgco = Wgco; J.H = H;
    J.u_dtype = u_dtype; J.w_dtype = w_dtype; J.h_dtype = h_dtype;
    J.anchor = anchor; J.R = R; J.gamma = gamma; J.V = V; J.r = r; J.d = d; J.rnn = 1;
    J.seed = seed; J.req_ids = req_ids; J.T = T;
    J.tokens = tokens; J.qx = qx; J.lse = lse; J.code = code; J.margin = margin;
    J.state_out = state_out;
    return draft_common(&J, n_threads);
}

/* ------------------------------------------------------------------ */
/* Verification (explainer section 05; blog section 1).                 */
/* ------------------------------------------------------------------ */
typedef struct {
    const void *P, *U, *W2;
    int p_dtype, u_dtype, w_dtype;
    const int32_t* tokens;
    const double *qx, *lse, *code;
    const int32_t* verify_len;
    int R, gamma, V, r;
    uint64_t seed;
    const uint32_t* req_ids;
    double T;
    int32_t *out_tokens, *accept_len, *n_out, *gap_kind;
    double *px, *lse_p, *min_gap;
    int r_begin, r_end, status;
} verify_job;

/* p = softmax(P_row / T); returns lse of P_row / T. */
static double target_probs(const verify_job* J, int ri, int row, double* p) {
    const int V = J->V;
    size_t base = ((size_t)ri * (J->gamma + 1) + (size_t)row) * (size_t)V;
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        p[v] = ld(J->P, J->p_dtype, base + v) / J->T;
        if (p[v] > m) m = p[v];
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp(p[v] - m);
    double lse = m + log(s);
    for (int v = 0; v < V; ++v) p[v] = exp(p[v] - lse);
    return lse;
}

static int target_argmax(const verify_job* J, int ri, int row) {
    size_t base = ((size_t)ri * (J->gamma + 1) + (size_t)row) * (size_t)J->V;
    double best = -INFINITY;
    int arg = 0;
    for (int v = 0; v < J->V; ++v) {
        double y = ld(J->P, J->p_dtype, base + v);
        if (y > best) { best = y; arg = v; }
    }
    return arg;
}

static void* verify_worker(void* arg) {
    verify_job* J = (verify_job*)arg;
    const int V = J->V, gamma = J->gamma, r = J->r;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p || !q || !w) { J->status = -1; goto done; }
    for (int ri = J->r_begin; ri < J->r_end; ++ri) {
        uint32_t req = J->req_ids ? J->req_ids[ri] : (uint32_t)ri;
        int L = J->verify_len ? J->verify_len[ri] : gamma;
        if (L < 0 || L > gamma) { J->status = -3; goto done; }
        int32_t* out = J->out_tokens + (size_t)ri * (gamma + 1);
        for (int i = 0; i <= gamma; ++i) out[i] = -1;
        for (int k = 0; k < gamma; ++k) J->px[(size_t)ri * gamma + k] = NAN;
        for (int k = 0; k <= gamma; ++k) J->lse_p[(size_t)ri * (gamma + 1) + k] = NAN;
        double gap = INFINITY;
        int kind = 0;
        const int32_t* x = J->tokens + (size_t)ri * gamma;
        int j = 0;   /* first rejected position (1-based), 0 if none */
        if (J->T > 0.0) {
            for (int k = 1; k <= L; ++k) {
                double lp = target_probs(J, ri, k - 1, p);
                J->lse_p[(size_t)ri * (gamma + 1) + (k - 1)] = lp;
                double pxk = p[x[k - 1]];
                J->px[(size_t)ri * gamma + (k - 1)] = pxk;
                double qxk = J->qx[(size_t)ri * gamma + (k - 1)];
                double ratio = pxk / qxk;
                double u = oracle_rng_uniform(J->seed, req, (uint32_t)k, 1u, 0u);
                double g = fabs(u - ratio);
                if (g < gap) { gap = g; kind = 1; }
                if (u < ratio) {
                    out[k - 1] = x[k - 1];          /* accepted */
                } else {
                    j = k;                          /* first rejection */
                    break;
                }
            }
            if (j > 0) {
                /* Residual r(v) = max(p - q, 0) / Z at position j. */
                double lp = target_probs(J, ri, j - 1, p);
                (void)lp;
                const double* e = J->code + ((size_t)ri * gamma + (size_t)(j - 1)) * r;
                size_t urow = ((size_t)ri * gamma + (size_t)(j - 1)) * (size_t)V;
                for (int v = 0; v < V; ++v) q[v] = 0.0;
                for (int i = 0; i < r; ++i) {
                    double ei = e[i];
                    for (int v = 0; v < V; ++v) q[v] += ei * ld(J->W2, J->w_dtype, (size_t)i * V + v);
                }
                double lq = J->lse[(size_t)ri * gamma + (size_t)(j - 1)];
                for (int v = 0; v < V; ++v) q[v] = exp((ld(J->U, J->u_dtype, urow + v) + q[v]) / J->T - lq);
                oracle_residual_weights(p, q, V, w);
                double Z = 0.0;
                for (int v = 0; v < V; ++v) Z += w[v];
                const double* src = w;
                if (!(Z > 0.0)) { src = p; if (0.0 < gap) { gap = 0.0; kind = 3; } }
                double tg;
                int y = oracle_tree_sample(src, V, J->seed, req, (uint32_t)j, &tg);
                if (tg < gap) { gap = tg; kind = 2; }
                out[j - 1] = y;
                J->accept_len[ri] = j - 1;
            } else {
                /* Every verified draft accepted: bonus token from p_{L+1}. */
                double lp = target_probs(J, ri, L, p);
                J->lse_p[(size_t)ri * (gamma + 1) + L] = lp;
                double tg;
                int y = oracle_tree_sample(p, V, J->seed, req, (uint32_t)(L + 1), &tg);
                if (tg < gap) { gap = tg; kind = 2; }
                out[L] = y;
                J->accept_len[ri] = L;
            }
        } else {
            /* Greedy: exact-match prefix, the target's argmax replaces the
             * first mismatch, otherwise a bonus argmax. */
            for (int k = 1; k <= L; ++k) {
                int t = target_argmax(J, ri, k - 1);
                if (t == x[k - 1]) {
                    out[k - 1] = t;
                } else {
                    out[k - 1] = t;
                    j = k;
                    break;
                }
            }
            if (j > 0) {
                J->accept_len[ri] = j - 1;
            } else {
                out[L] = target_argmax(J, ri, L);
                J->accept_len[ri] = L;
            }
        }
        J->n_out[ri] = J->accept_len[ri] + 1;
        J->min_gap[ri] = gap;
        J->gap_kind[ri] = kind;
    }
done:
    free(p); free(q); free(w);
    return NULL;
}

int oracle_verify(const void* P, int p_dtype, const void* U, int u_dtype,
                  const void* W2, int w_dtype,
                  const int32_t* tokens, const double* qx, const double* lse,
                  const double* code, const int32_t* verify_len,
                  int R, int gamma, int V, int r,
                  uint64_t seed, const uint32_t* req_ids, double T,
                  int32_t* out_tokens, int32_t* accept_len, int32_t* n_out,
                  double* px, double* lse_p, double* min_gap, int32_t* gap_kind,
                  int n_threads) {
    if (R <= 0 || gamma <= 0 || V <= 0 || r <= 0) return -3;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > R) n_threads = R;
    verify_job* jobs = (verify_job*)calloc((size_t)n_threads, sizeof(verify_job));
    if (!jobs) return -1;
    for (int t = 0; t < n_threads; ++t) {
        verify_job* J = &jobs[t];
        J->P = P; J->U = U; J->W2 = W2; J->p_dtype = p_dtype; J->u_dtype = u_dtype; J->w_dtype = w_dtype;
        J->tokens = tokens; J->qx = qx; J->lse = lse; J->code = code; J->verify_len = verify_len;
        J->R = R; J->gamma = gamma; J->V = V; J->r = r; J->seed = seed; J->req_ids = req_ids; J->T = T;
        J->out_tokens = out_tokens; J->accept_len = accept_len; J->n_out = n_out;
        J->px = px; J->lse_p = lse_p; J->min_gap = min_gap; J->gap_kind = gap_kind;
        J->r_begin = (int)((long)R * t / n_threads);
        J->r_end = (int)((long)R * (t + 1) / n_threads);
    }
    run_jobs(jobs, sizeof(verify_job), n_threads, verify_worker);
    int st = 0;
    for (int t = 0; t < n_threads; ++t) if (jobs[t].status) st = jobs[t].status;
    free(jobs);
    return st;
}

/* ------------------------------------------------------------------ */
/* Confidence head (blog section 4.1, ConfidenceHead).                  */
/* ------------------------------------------------------------------ */
int oracle_confidence(const void* H, int h_dtype, const void* W1, int w_dtype, const float* w,
                      const int32_t* anchor, const int32_t* tokens,
                      int R, int gamma, int V, int d, int r, const double* temps, double* c) {
    if (R <= 0 || gamma <= 0 || V <= 0 || d < 0 || r <= 0) return -3;
    for (int ri = 0; ri < R; ++ri) {
        for (int k = 1; k <= gamma; ++k) {
            /* the token before position k: x_0 = anchor, x_{k-1} = draft k-1 */
            int prev = (k == 1) ? anchor[ri] : tokens[(size_t)ri * gamma + (size_t)(k - 2)];
            if (prev < 0 || prev >= V) return -6;
            /* logit = w . [h_k, W1[x_{k-1}]]: the first d weights meet h_k,
             * the last r meet the previous token's rank-r embedding */
            double t = 0.0;
            const size_t hrow = ((size_t)ri * gamma + (size_t)(k - 1)) * (size_t)d;
            for (int i = 0; i < d; ++i) t += (double)w[i] * ld(H, h_dtype, hrow + (size_t)i);
            for (int i = 0; i < r; ++i) t += (double)w[d + i] * ld(W1, w_dtype, (size_t)prev * r + (size_t)i);
            /* with sequential temperature scaling (section 4.2): sigmoid(t / t_k) */
            if (temps) t /= temps[k - 1];
            c[(size_t)ri * gamma + (size_t)(k - 1)] = sigmoid(t);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Scheduler (blog section 4.3; explainer section 04).                   */
/* ------------------------------------------------------------------ */
void oracle_prefix_survival(const float* c, int R, int gamma, float* a) {
    for (int ri = 0; ri < R; ++ri) {
        float prod = 1.0f;
        for (int j = 0; j < gamma; ++j) {
            prod = prod * c[(size_t)ri * gamma + j];
            a[(size_t)ri * gamma + j] = prod;
        }
    }
}

typedef struct { float a; int r, j; } cand_t;

/* Order: a descending, then request ascending, then position ascending. */
static int cand_cmp(const void* x, const void* y) {
    const cand_t* A = (const cand_t*)x;
    const cand_t* B = (const cand_t*)y;
    if (A->a > B->a) return -1;
    if (A->a < B->a) return 1;
    if (A->r != B->r) return A->r < B->r ? -1 : 1;
    if (A->j != B->j) return A->j < B->j ? -1 : 1;
    return 0;
}

static double sps_at(const double* sps, int n_sps, long B) {
    return (B >= 0 && B < n_sps) ? sps[B] : 0.0;   /* missing entries count as 0 */
}

static cand_t* sorted_candidates(const float* c, int R, int gamma, int* n_out) {
    float* a = (float*)malloc(sizeof(float) * (size_t)R * gamma);
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * ((size_t)R * gamma + 1));
    if (!a || !cand) { free(a); free(cand); return NULL; }
    oracle_prefix_survival(c, R, gamma, a);
    int n = 0;
    for (int ri = 0; ri < R; ++ri)
        for (int j = 0; j < gamma; ++j) {
            float av = a[(size_t)ri * gamma + j];
            if (av > 0.0f) { cand[n].a = av; cand[n].r = ri; cand[n].j = j; ++n; }
        }
    free(a);
    qsort(cand, (size_t)n, sizeof(cand_t), cand_cmp);
    *n_out = n;
    return cand;
}

int oracle_schedule_loop(const float* c, const double* sps, int n_sps, int R, int gamma,
                         int32_t* lengths, double* theta) {
    int n;
    cand_t* cand = sorted_candidates(c, R, gamma, &n);
    if (!cand) return -1;
    int32_t* cur = (int32_t*)calloc((size_t)R, sizeof(int32_t));
    if (!cur) { free(cand); return -1; }
    for (int ri = 0; ri < R; ++ri) lengths[ri] = 0;
    long B = R;                       /* every request sends its anchor */
    double tau = (double)R;
    double best = tau * sps_at(sps, n_sps, B);
    for (int i = 0; i < n; ++i) {
        if (cand[i].j != cur[cand[i].r]) continue;    /* prefix constraint */
        cur[cand[i].r] += 1;
        B += 1;
        tau += (double)cand[i].a;
        double th = tau * sps_at(sps, n_sps, B);
        if (th > best) {
            best = th;
            memcpy(lengths, cur, sizeof(int32_t) * (size_t)R);
        } else {
            break;                                    /* early stop */
        }
    }
    *theta = best;
    int nstar = 0;
    for (int ri = 0; ri < R; ++ri) nstar += lengths[ri];
    free(cur); free(cand);
    return nstar;
}

int oracle_schedule_closed(const float* c, const double* sps, int n_sps, int R, int gamma,
                           int32_t* lengths, double* theta, double* min_rel_gap) {
    int n;
    cand_t* cand = sorted_candidates(c, R, gamma, &n);
    if (!cand) return -1;
    double* th = (double*)malloc(sizeof(double) * ((size_t)n + 1));
    if (!th) { free(cand); return -1; }
    double tau = (double)R;
    th[0] = tau * sps_at(sps, n_sps, R);
    for (int i = 0; i < n; ++i) {
        tau += (double)cand[i].a;              /* tau_{i+1} = R + a_(1) + ... + a_(i+1) */
        th[i + 1] = tau * sps_at(sps, n_sps, (long)R + i + 1);
    }
    int nstar = n;
    for (int i = 0; i < n; ++i)
        if (!(th[i + 1] > th[i])) { nstar = i; break; }
    /* smallest relative gap over every comparison the stop rule made */
    double gap = INFINITY;
    int last = nstar < n ? nstar : n - 1;
    for (int i = 0; i <= last; ++i) {
        double den = fabs(th[i]) > 0.0 ? fabs(th[i]) : 1.0;
        double g = fabs(th[i + 1] - th[i]) / den;
        if (g < gap) gap = g;
    }
    if (min_rel_gap) *min_rel_gap = gap;
    for (int ri = 0; ri < R; ++ri) lengths[ri] = 0;
    for (int i = 0; i < nstar; ++i) lengths[cand[i].r] += 1;
    *theta = th[nstar];
    free(th); free(cand);
    return nstar;
}

/* Production-style scheduler (explainer section 04): the capacity comes
 * from the prediction made two steps back, and the current candidates are
 * ranked into it.  Reading: budget = the n* the synchronous rule gave two
 * steps earlier (negative: none yet, use this step's n*); the current
 * candidates, in the order of the synchronous scheduler, fill min(budget,
 * count) places; theta = tau * SPS at that batch.  *n_star receives this
 * step's own synchronous n*, the capacity for two steps later.  Returns the
 * number of places filled. */
int oracle_schedule_budget(const float* c, const double* sps, int n_sps, int R, int gamma, int budget,
                           int32_t* lengths, double* theta, int32_t* n_star) {
    int n;
    cand_t* cand = sorted_candidates(c, R, gamma, &n);
    if (!cand) return -1;
    double th_sync;
    const int ns = oracle_schedule_closed(c, sps, n_sps, R, gamma, lengths, &th_sync, NULL);
    if (ns < 0) { free(cand); return -1; }
    *n_star = ns;
    const int nb = budget < 0 ? ns : (budget < n ? budget : n);
    double tau = (double)R;
    for (int ri = 0; ri < R; ++ri) lengths[ri] = 0;
    for (int i = 0; i < nb; ++i) {
        lengths[cand[i].r] += 1;
        tau += (double)cand[i].a;
    }
    *theta = tau * sps_at(sps, n_sps, (long)R + nb);
    free(cand);
    return nb;
}

/* Threshold filter (blog section 4.3, the confidence-threshold sweep; the
 * explainer's section 04 contrasts it with the scheduler): every request
 * verifies its longest prefix whose confidence clears one fixed threshold.
 * mode 0: a_{r,j} = c_{r,1} ... c_{r,j} >= theta (float32 product in position
 * order, as the scheduler forms it); mode 1: c_{r,j} >= theta itself, up to
 * the first position that misses. */
int oracle_threshold_lengths(const float* c, int R, int gamma, float theta, int mode, int32_t* lengths) {
    if (R <= 0 || gamma <= 0 || (mode != 0 && mode != 1)) return -3;
    float* a = (float*)malloc(sizeof(float) * (size_t)R * (size_t)gamma);
    if (!a) return -1;
    oracle_prefix_survival(c, R, gamma, a);
    const float* score = mode == 0 ? a : c;
    for (int ri = 0; ri < R; ++ri) {
        int len = 0;
        while (len < gamma && score[(size_t)ri * gamma + (size_t)len] >= theta) ++len;
        lengths[ri] = len;
    }
    free(a);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Sequential Temperature Scaling (blog section 4.2).                   */
/* ------------------------------------------------------------------ */

/* Expected calibration error (Guo, Pleiss, Sun, Weinberger, "On
 * Calibration of Modern Neural Networks", ICML 2017, section 2): the
 * predictions fall into M equal-width bins over [0, 1] (bin b holds
 * b/M <= p < (b+1)/M; p = 1 goes to the last bin), and
 *   ECE = sum_b |B_b|/N * |mean of y over B_b - mean of p over B_b|. */
double oracle_ece(const double* pred, const int32_t* y, int N, int M) {
    if (N <= 0 || M <= 0) return 0.0;
    double* sp = (double*)calloc((size_t)M, sizeof(double));
    double* sy = (double*)calloc((size_t)M, sizeof(double));
    long* cnt = (long*)calloc((size_t)M, sizeof(long));
    if (!sp || !sy || !cnt) { free(sp); free(sy); free(cnt); return NAN; }
    for (int n = 0; n < N; ++n) {
        int b = (int)floor(pred[n] * (double)M);
        if (b < 0) b = 0;
        if (b > M - 1) b = M - 1;
        cnt[b] += 1;
        sp[b] += pred[n];
        sy[b] += (double)(y[n] != 0);
    }
    double ece = 0.0;
    for (int b = 0; b < M; ++b) {
        if (cnt[b] == 0) continue;
        const double acc = sy[b] / (double)cnt[b], conf = sp[b] / (double)cnt[b];
        ece += ((double)cnt[b] / (double)N) * fabs(acc - conf);
    }
    free(sp); free(sy); free(cnt);
    return ece;
}

/* Temperature scaling of one confidence: sigmoid(logit(c) / t), with
 * logit(c) = ln c - ln(1 - c) (c = 0 and c = 1 stay where they are). */
static double temper(double c, double t) {
    const double z = log(c) - log1p(-c);
    return sigmoid(z / t);
}

int oracle_sts_fit(const float* c, const int32_t* accept_len, int N, int gamma,
                   const double* grid, int G, int M,
                   double* t_out, int32_t* g_out, double* ece_out, double* gap_out) {
    if (N <= 0 || gamma <= 0 || G <= 0 || M <= 0) return -3;
    double* a_prev = (double*)malloc(sizeof(double) * (size_t)N);   /* prefix survival of positions < k */
    double* pred = (double*)malloc(sizeof(double) * (size_t)N);
    int32_t* y = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    if (!a_prev || !pred || !y) { free(a_prev); free(pred); free(y); return -1; }
    for (int n = 0; n < N; ++n) a_prev[n] = 1.0;
    for (int k = 1; k <= gamma; ++k) {
        /* outcome at position k: the first k drafts were all accepted */
        for (int n = 0; n < N; ++n) y[n] = accept_len[n] >= k;
        double best = INFINITY, second = INFINITY;
        int gbest = 0;
        for (int g = 0; g < G; ++g) {
            for (int n = 0; n < N; ++n)
                pred[n] = a_prev[n] * temper((double)c[(size_t)n * gamma + (size_t)(k - 1)], grid[g]);
            const double e = oracle_ece(pred, y, N, M);
            if (e < best) { second = best; best = e; gbest = g; }   /* ties keep the lowest index */
            else if (e < second) { second = e; }
        }
        t_out[k - 1] = grid[gbest];
        g_out[k - 1] = gbest;
        ece_out[k - 1] = best;
        gap_out[k - 1] = second - best;
        /* fix this position's temperature before the next one */
        for (int n = 0; n < N; ++n)
            a_prev[n] *= temper((double)c[(size_t)n * gamma + (size_t)(k - 1)], grid[gbest]);
    }
    free(a_prev); free(pred); free(y);
    return 0;
}

void oracle_sts_apply(const float* c, int N, int gamma, const double* t, double* c_out) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < gamma; ++k)
            c_out[(size_t)n * gamma + k] = temper((double)c[(size_t)n * gamma + k], t[k]);
}
