/*
 * dspark_oracle.h -- plain CPU oracle for one DSpark decoding cycle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this code; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code with the CUDA library.
 *
 * All arithmetic is double precision unless a function says otherwise.
 * Inputs are read in their storage type (float32, or bfloat16 given as
 * uint16 bit patterns) and widened to double exactly.
 *
 * Sources (the pages are cited by title and section):
 *  - "DSpark: DeepSeek 线上跑的投机解码" (blog), section 3.2: Markov head
 *    B_k = W1[x_{k-1}] W2, RNN head step, and the sequential stage loop;
 *    section 4.1: the confidence head; section 4.2: sequential temperature
 *    scaling; section 4.3: prefix survival, the
 *    hardware-aware scheduler and the confidence-threshold sweep.
 *  - "DSpark explainer", section 03: q_k = softmax(U_k + B_k);
 *    section 04: a_j = c_1 ... c_j, B, tau, Theta = tau * SPS(B);
 *    section 05: alpha(x) = min(1, p(x)/q(x)) and
 *    r(v) = max(p(v) - q(v), 0) / sum_u max(p(u) - q(u), 0).
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers:
 *    As Easy as 1, 2, 3", SC'11.
 *  - Expected calibration error: Guo, Pleiss, Sun, Weinberger, "On
 *    Calibration of Modern Neural Networks", ICML 2017, section 2.
 */
#ifndef DSPARK_ORACLE_H
#define DSPARK_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Philox4x32-10 block function. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* Uniform in (0,1) from one 32-bit word: (w + 1/2) * 2^-32 (exact in double). */
double oracle_uniform(uint32_t w);
/* The uniform for (seed, request id, position, stream, index v). */
double oracle_rng_uniform(uint64_t seed, uint32_t req, uint32_t pos, uint32_t stream, uint32_t v);

/* Elementwise helpers of the explainer's section 05, exposed for the pins. */
double oracle_accept_prob(double px, double qx);                 /* min(1, p/q) */
void oracle_residual_weights(const double* p, const double* q, int V, double* w); /* max(p-q,0) */
/* Draw from weights w[0..V) by the binary sum tree (one uniform per level;
 * stream 2 at position pos).  Returns the index, writes the smallest gap
 * |u_d - threshold_d| over the levels to *min_gap. */
int oracle_tree_sample(const double* w, int V, uint64_t seed, uint32_t req, uint32_t pos, double* min_gap);

/* Draft with the Markov head (blog section 3.2; explainer section 03).
 * x_k is drawn from softmax(z), z = (U_k + B_k)/T, by Gumbel-max in two
 * levels: over chunks of 256 indices with keys ln(chunk mass) + G (stream 3,
 * index = chunk), then inside the chosen chunk with keys z_v + G (stream 0,
 * index = v).  Outputs: tokens [R,gamma], qx [R,gamma] = q_k(x_k),
 * lse [R,gamma] of the tempered logits, code [R,gamma,r] = W1[x_{k-1}],
 * margin [R,gamma] = the smaller of the two levels' best-minus-second key
 * gaps (logit gap at T = 0).
 * req_ids may be NULL (request index).  Returns 0 or a negative error. */
int oracle_draft_markov(const void* U, int u_dtype, const int32_t* anchor,
                        const void* W1, const void* W2, int w_dtype,
                        int R, int gamma, int V, int r,
                        uint64_t seed, const uint32_t* req_ids, double T,
                        int32_t* tokens, double* qx, double* lse, double* code,
                        double* margin, int n_threads);

/* Draft with the RNN head (blog section 3.2 RNNHead.step).  H is [R,gamma,d]
 * in h_dtype, Wgco is [2r+d, 3r] in w_dtype with column blocks
 * (gate | candidate | output).  code[R,gamma,r] = tanh(output) and
 * state_out [R,r] (may be NULL) is s_gamma. */
int oracle_draft_rnn(const void* U, int u_dtype, const int32_t* anchor,
                     const void* W1, const void* W2, const void* Wgco, int w_dtype,
                     const void* H, int h_dtype,
                     int R, int gamma, int V, int r, int d,
                     uint64_t seed, const uint32_t* req_ids, double T,
                     int32_t* tokens, double* qx, double* lse, double* code,
                     double* margin, double* state_out, int n_threads);

/* Lossless verification (explainer section 05).  verify_len may be NULL
 * (verify all gamma).  Outputs: out_tokens [R,gamma+1] (-1 padded),
 * accept_len [R], n_out [R], px [R,gamma] (p_k(x_k) for the positions that
 * were tested, NaN otherwise), lse_p [R,gamma+1] (NaN for unread rows),
 * min_gap [R] = smallest |u - threshold| over every random decision taken
 * for the request (+inf if none), gap_kind [R] = 1 acceptance, 2 tree level,
 * 3 empty residual, 0 none. */
int oracle_verify(const void* P, int p_dtype, const void* U, int u_dtype,
                  const void* W2, int w_dtype,
                  const int32_t* tokens, const double* qx, const double* lse,
                  const double* code, const int32_t* verify_len,
                  int R, int gamma, int V, int r,
                  uint64_t seed, const uint32_t* req_ids, double T,
                  int32_t* out_tokens, int32_t* accept_len, int32_t* n_out,
                  double* px, double* lse_p, double* min_gap, int32_t* gap_kind,
                  int n_threads);

/* Confidence head (blog section 4.1): c[r,k-1] = sigmoid(w . [h_k, W1[x_{k-1}]])
 * with no bias, x_0 = anchor[r] and x_{k-1} = tokens[r,k-2] for k >= 2.
 * H is [R,gamma,d] in h_dtype, W1 [V,r] in w_dtype, w [d + r] float32 (the
 * first d entries weigh h_k, the last r the embedding).  c is [R,gamma].
 * temps [gamma] (may be NULL): per-position temperatures of section 4.2,
 * c = sigmoid(w . [h_k, W1[x_{k-1}]] / temps[k-1]).
 * Returns 0, or -6 for a token outside [0, V). */
int oracle_confidence(const void* H, int h_dtype, const void* W1, int w_dtype, const float* w,
                      const int32_t* anchor, const int32_t* tokens,
                      int R, int gamma, int V, int d, int r, const double* temps, double* c);

/* Threshold filter: lengths[r] = the longest prefix of positions whose score
 * is >= theta; score = a[r,j] (mode 0, float32 prefix product) or c[r,j]
 * (mode 1).  Returns 0 or a negative error. */
int oracle_threshold_lengths(const float* c, int R, int gamma, float theta, int mode, int32_t* lengths);

/* Prefix survival a[r,j] = c[r,0] * ... * c[r,j], float32 sequential
 * product (the decision precision of the scheduler's sort). */
void oracle_prefix_survival(const float* c, int R, int gamma, float* a);

/* Scheduler of the blog's section 4.3, written as the page's loop:
 * candidates sorted by (a desc, r asc, j asc), prefix violations skipped,
 * stop at the first non-improving Theta.  Returns n*. */
int oracle_schedule_loop(const float* c, const double* sps, int n_sps, int R, int gamma,
                         int32_t* lengths, double* theta);
/* Same scheduler in closed form: Theta(n) = tau_n * SPS[R+n] over the sorted
 * prefix sums; n* = first n with Theta(n+1) <= Theta(n).  min_rel_gap gets
 * the smallest relative gap |Theta(n+1) - Theta(n)| / Theta(n) over the
 * comparisons n = 0..n* the stop rule made (+inf if none).  Returns n*. */
int oracle_schedule_closed(const float* c, const double* sps, int n_sps, int R, int gamma,
                           int32_t* lengths, double* theta, double* min_rel_gap);

/* Production-style scheduler (explainer section 04): budget = the n* of two
 * steps back (negative: none yet, this step's n* is used); the candidates
 * in the scheduler's order fill min(budget, count) places; theta = tau *
 * SPS at that batch; *n_star = this step's synchronous n*.  Returns the
 * number of places filled. */
int oracle_schedule_budget(const float* c, const double* sps, int n_sps, int R, int gamma, int budget,
                           int32_t* lengths, double* theta, int32_t* n_star);

/* Expected calibration error (Guo et al., ICML 2017, section 2) of
 * predictions pred[N] against outcomes y[N] (nonzero = 1) over M
 * equal-width bins of [0, 1]; p = 1 falls in the last bin. */
double oracle_ece(const double* pred, const int32_t* y, int N, int M);

/* Sequential Temperature Scaling (blog section 4.2): per position k = 1..gamma,
 * left to right, the grid temperature t minimising the ECE of the calibrated
 * prefix survival a'_k = prod_{i<=k} sigmoid(logit(c_i) / t_i) (t_i fixed for
 * i < k, t_k = t) against the outcome accept_len >= k; ties keep the lowest
 * grid index.  c [N,gamma] float32 raw confidences, accept_len [N], grid [G].
 * Outputs per position: t_out, g_out (grid index), ece_out (the minimum) and
 * gap_out (second-smallest ECE minus the minimum, +inf if G = 1). */
int oracle_sts_fit(const float* c, const int32_t* accept_len, int N, int gamma,
                   const double* grid, int G, int M,
                   double* t_out, int32_t* g_out, double* ece_out, double* gap_out);

/* c_out[n,k] = sigmoid(logit(c[n,k]) / t[k]). */
void oracle_sts_apply(const float* c, int N, int gamma, const double* t, double* c_out);

#ifdef __cplusplus
}
#endif
#endif
