/*
 * dspark.h -- C ABI of the GB300 DSpark cycle library (libdspark.so).
 *
 * One DSpark decoding cycle has three data-parallel parts, each one entry
 * point here:
 *
 *   dspark_draft_markov / dspark_draft_rnn
 *       the sequential stage of the semi-autoregressive drafter: for
 *       k = 1..gamma, B_k is added to the parallel backbone's base logits
 *       U_k and x_k is sampled from q_k = softmax((U_k + B_k) / T)
 *       ("DSpark: DeepSeek 线上跑的投机解码" blog, section 3.2, MarkovHead,
 *       RNNHead and the sequential-stage loop; DSpark explainer, section 03,
 *       q_k = softmax(U_k + B_k) with B_k = W1[x_{k-1}] W2).
 *   dspark_verify
 *       lossless verification: accept x with min(1, p(x)/q(x)), on the first
 *       rejection resample from max(p - q, 0) normalised, emit a bonus token
 *       when every verified draft is accepted (DSpark explainer, section 05,
 *       alpha(x) and r(v); section 02 for the greedy T = 0 form).
 *   dspark_schedule
 *       the confidence scheduler: a_j = c_1 ... c_j, B = sum_r (1 + l_r),
 *       tau = sum_r (1 + sum_{j <= l_r} a_{r,j}), Theta = tau * SPS(B), and
 *       the greedy early stop over candidates sorted by a (blog section 4.3;
 *       explainer section 04, "algorithm details").
 *
 * Conventions for every entry point:
 *  - Tensor arguments are DEVICE pointers owned by the caller, row-major and
 *    contiguous.  The library never allocates device memory: all scratch
 *    lives in a caller-provided workspace whose size the matching
 *    dspark_*_workspace_size() returns (256-byte aligned pointer required).
 *  - Work is enqueued asynchronously on the caller's stream `stream`
 *    (a cudaStream_t passed as void*; NULL = legacy default stream).
 *  - dtype arguments take DSPARK_F32 or DSPARK_BF16 (bf16 = IEEE bfloat16).
 *  - U, P (and dspark_verify_staged's staging buffer), W2 and Wgco are read
 *    with 16-byte loads and tensor-map copies: they must start on a 16-byte
 *    boundary, else the call returns DSPARK_ERR_INVALID_ARG (cudaMalloc and
 *    PyTorch allocations always do; an offset view may not).
 *  - The return value is DSPARK_OK or a negative DSPARK_ERR_* code.  Host
 *    checks (null pointers, sizes, dtypes, workspace size) fail before any
 *    work is enqueued.  Conditions that only the device can see (a token id
 *    outside [0, V), a bounded wait that ran out) do not fault: the kernel
 *    skips the bad access, records the condition in a status word at the
 *    start of the workspace and finishes; dspark_workspace_status() reads
 *    and clears it.
 *  - U, W2 and Wgco must be device memory of the current device (the
 *    tensor-core kernels read them through tensor maps and share W2 tiles
 *    among the CTAs of a thread-block cluster, which is defined for this
 *    GPU's own memory only); a peer device's buffer, mapped host memory or
 *    managed memory returns DSPARK_ERR_INVALID_ARG before anything is
 *    enqueued.  P (the target logits) may be pinned host memory mapped for
 *    the device (dspark_host_pointer).
 *  - Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key
 *    (seed low 32 bits, seed high 32 bits) and counter
 *    (v / 4, request id, position, stream); index v takes output word v mod 4
 *    and becomes u = (w + 1/2) * 2^-32 in (0, 1).  Streams:
 *    0 = draft Gumbel noise of a column (v = vocabulary index, position k = 1..gamma),
 *    1 = acceptance uniform (v = 0, position k),
 *    2 = residual / bonus draw (v = tree level, position = the position sampled),
 *    3 = draft Gumbel noise of a 256-column chunk (v = chunk index, position k).
 *    The request id is req_ids[i] (device array) or i when req_ids is NULL.
 *    dspark_philox4x32_10 below evaluates the same block function on the
 *    device, for known-answer checks.
 *  - Nothing is thrown across the ABI.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum dspark_dtype { DSPARK_F32 = 0, DSPARK_BF16 = 1 };

enum dspark_status {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = -1,     /* null pointer, negative size, bad temperature */
    DSPARK_ERR_UNSUPPORTED_DTYPE = -2,
    DSPARK_ERR_SHAPE = -3,           /* sizes outside the supported range */
    DSPARK_ERR_CUDA = -4,            /* a CUDA runtime call failed */
    DSPARK_ERR_TIMEOUT = -5,         /* a bounded device wait ran out */
    DSPARK_ERR_BAD_TOKEN = -6,       /* a token id outside [0, V) reached a kernel */
    DSPARK_ERR_UNIMPLEMENTED = -7,
    DSPARK_ERR_WORKSPACE = -8        /* workspace null, misaligned or too small */
};

/* Text for a status code (static storage). */
const char* dspark_strerror(int status);
/* Library version string (static storage). */
const char* dspark_version(void);

/*
 * Synchronises `stream`, then reads and clears the device status word at the
 * start of workspace `ws` (any workspace this library was given).  Returns
 * DSPARK_OK, DSPARK_ERR_BAD_TOKEN, DSPARK_ERR_TIMEOUT or DSPARK_ERR_CUDA.
 */
int dspark_workspace_status(void* ws, void* stream);

/*
 * Bounded waits (no counterpart on the pages).  Every wait of a kernel on
 * another thread's progress (a pipeline stage, a peer CTA's copy) gives up
 * after a limit of SM cycles, records DSPARK_ERR_TIMEOUT in the workspace's
 * status word and winds the kernel down without faulting.  The limit is
 * 2^32 cycles (2 to 4 s at 2 to 1 GHz) unless set here for the calls that
 * use workspace `ws` (limit_cycles = 0 restores the default).
 * test_withhold = 1 is a test hook: the next draft call on `ws` that runs the
 * tensor-core sweep withholds the first U stage of its first step (no copy is
 * issued for it), so that the bounded wait on it runs out and the call ends
 * with DSPARK_ERR_TIMEOUT in the status word; set 0 to turn it off.  The
 * values live in the workspace header (a fresh zeroed workspace has the
 * defaults).  Synchronises `stream`.  Errors: INVALID_ARG for a null or
 * misaligned workspace or another test_withhold, CUDA for a failed copy.
 */
int dspark_workspace_set_wait(void* ws, uint64_t limit_cycles, int test_withhold, void* stream);

/*
 * The device-accessible address of a pinned (page-locked) host buffer, so
 * that kernels read it in place over the host link (zero copy).  The input
 * arrays of the calls below may be such addresses: verification, for
 * example, then fetches only the target rows its decisions need.  Returns
 * DSPARK_ERR_CUDA (and *device = NULL) for memory that is not pinned and
 * mapped.  Host-side only; nothing is enqueued.
 */
int dspark_host_pointer(const void* host, void** device);

/* ------------------------------------------------------------------ draft */

/*
 * Workspace bytes for dspark_draft_markov / dspark_draft_rnn (d = 0 for the
 * Markov head).  Returns 0 for unsupported sizes.
 */
size_t dspark_draft_workspace_size(int R, int gamma, int V, int r, int d);

/*
 * Markov-head drafting: the sequential stage with B_k = W1[x_{k-1}] W2
 * (blog section 3.2 MarkovHead; explainer section 03), x_0 = anchor.
 *
 *   U       [R, gamma, V]  u_dtype   base logits of the parallel backbone
 *   anchor  [R]            int32     x_0 per request, in [0, V)
 *   W1      [V, r]         w_dtype   rank-r embedding of the previous token
 *   W2      [r, V]         w_dtype   rank-r projection to the vocabulary
 *   seed, req_ids, temperature       RNG key, request ids (NULL = index),
 *                                    T > 0 samples, T = 0 takes the argmax
 * Outputs (device, caller-owned):
 *   tokens  [R, gamma]     int32     x_k
 *   q_tok   [R, gamma]     float     q_k(x_k) (1 at T = 0)
 *   lse     [R, gamma]     double    log sum_v exp((U_k + B_k)[v] / T) (0 at T = 0)
 *   code    [R, gamma, r]  float     e_k = W1[x_{k-1}], the rank-r code that
 *                                    gives B_k = e_k W2 (consumed by verify)
 * Sampling (T > 0), with z = (U_k + B_k) / T and Gumbel noise G = -ln(-ln u):
 * Gumbel-max in two levels, an exact sampler of softmax(z).  First a chunk c
 * of 256 consecutive columns (the last one may be shorter):
 *   c = argmax_c  ln(sum_{v in c} exp z_v) + G_c,  u_c from stream 3, index c;
 * then the column inside it:
 *   x_k = argmax_{v in c}  z_v + G_v,            u_v from stream 0, index v.
 * Ties go to the lowest index at both levels.  (A chunk is chosen with
 * probability equal to its share of the mass, the column with its share of
 * the chunk, so x_k ~ softmax(z); the realisation differs from a single
 * Gumbel-max over all V columns.)  T = 0 takes argmax_v (U_k + B_k)[v], the
 * lowest v on ties.  B_k and q_k are never written to memory.
 * Requirements: R >= 1, 1 <= gamma <= 64, V >= 2 with V % 8 == 0 for bf16 and
 * V % 4 == 0 for f32 storage, V <= 2^20, 1 <= r <= 1024, T >= 0 and finite.
 * A logit of -inf (in U here, in U or P for verification) masks its column:
 * the column has no mass and is never drawn; every row needs at least one
 * finite logit.  NaN and +inf logits are not supported.
 */
int dspark_draft_markov(const void* U, int u_dtype, const int32_t* anchor,
                        const void* W1, const void* W2, int w_dtype,
                        int R, int gamma, int V, int r,
                        uint64_t seed, const uint32_t* req_ids, float temperature,
                        int32_t* tokens, float* q_tok, double* lse, float* code,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * RNN-head drafting (blog section 3.2 RNNHead.step): per step
 *   z   = [s_{k-1}, W1[x_{k-1}], h_k]                    (2r + d)
 *   G   = z Wgco, split into gate | cand | out           (3r, columns in that order)
 *   s_k = sigmoid(gate) * s_{k-1} + (1 - sigmoid(gate)) * tanh(cand),  s_0 = 0
 *   e_k = tanh(out),  B_k = e_k W2
 * and the same sampling as dspark_draft_markov.
 *   H      [R, gamma, d]  bfloat16   backbone hidden states h_k
 *   Wgco   [2r + d, 3r]   w_dtype
 *   state_out [R, r]      float      s_gamma (may be NULL)
 * code receives e_k = tanh(out_k).  Requirements as for the Markov head plus
 * 1 <= d <= 16384.
 */
int dspark_draft_rnn(const void* U, int u_dtype, const int32_t* anchor,
                     const void* W1, const void* W2, const void* Wgco, int w_dtype,
                     const void* H, int d,
                     int R, int gamma, int V, int r,
                     uint64_t seed, const uint32_t* req_ids, float temperature,
                     int32_t* tokens, float* q_tok, double* lse, float* code,
                     float* state_out,
                     void* ws, size_t ws_bytes, void* stream);

/* -------------------------------------------------------- confidence head */

/*
 * Confidence head fused into drafting (blog section 4.1, ConfidenceHead):
 *   c_k = sigmoid(w . [h_k, W1[x_{k-1}]])        no bias, x_0 = anchor
 * evaluated inside draft step k from the h_k row and the W1 row that step
 * gathers anyway, so c [R, gamma] is ready for dspark_schedule when the
 * draft finishes.
 *   H  [R, gamma, d]  bfloat16  backbone hidden states h_k (device).  NULL
 *                               with the RNN head: the head's own H and d
 *                               (the d below is then ignored); NULL with the
 *                               Markov head requires d = 0.
 *   w  [d + r]        float     weights: w[0, d) meet h_k, w[d, d + r) meet
 *                               W1[x_{k-1}] (device)
 *   d                 int       0 <= d <= 16384
 *   c  [R, gamma]     float     output (device, caller-owned): the dot product
 *                               in float32 (fixed summation order, so reruns
 *                               agree bit for bit), then the sigmoid in float32
 * The struct itself is read on the host during the call.  A null conf
 * turns the head off (the plain entry points below pass null).  Errors:
 * INVALID_ARG for a null w or c (or Markov H = NULL with d > 0), SHAPE for d
 * outside [0, 16384].
 *   t  [gamma]        double    per-position temperatures of Sequential
 *                               Temperature Scaling (blog section 4.2; for
 *                               example dspark_sts_fit's t_out), device, may be
 *                               NULL: c_k = sigmoid(w . [h_k, W1[x_{k-1}]] / t_k)
 *                               (the division in float32 by (float)(1 / t_k))
 */
typedef struct {
    const void* H;
    const float* w;
    int d;
    float* c;
    const double* t;
} dspark_conf_t;

/* dspark_draft_markov with the confidence head. */
int dspark_draft_markov_conf(const void* U, int u_dtype, const int32_t* anchor,
                             const void* W1, const void* W2, int w_dtype,
                             int R, int gamma, int V, int r,
                             uint64_t seed, const uint32_t* req_ids, float temperature,
                             int32_t* tokens, float* q_tok, double* lse, float* code,
                             const dspark_conf_t* conf,
                             void* ws, size_t ws_bytes, void* stream);

/* dspark_draft_rnn with the confidence head. */
int dspark_draft_rnn_conf(const void* U, int u_dtype, const int32_t* anchor,
                          const void* W1, const void* W2, const void* Wgco, int w_dtype,
                          const void* H, int d,
                          int R, int gamma, int V, int r,
                          uint64_t seed, const uint32_t* req_ids, float temperature,
                          int32_t* tokens, float* q_tok, double* lse, float* code,
                          float* state_out, const dspark_conf_t* conf,
                          void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------- verify */

size_t dspark_verify_workspace_size(int R, int gamma, int V, int r);

/*
 * Lossless verification (explainer section 05; blog section 1).
 *
 *   P          [R, gamma + 1, V] p_dtype  target logits; row k-1 scores draft
 *                                         position k, row gamma is the bonus row
 *   U, W2, tokens, q_tok, lse, code       as produced by a draft call
 *   verify_len [R] int32 or NULL          l_r in [0, gamma]; NULL verifies all
 * For T > 0, with p_k = softmax(P_{k-1} / T), for k = 1..l_r:
 *   u_k from stream 1; accept x_k iff u_k < p_k(x_k) / q_k(x_k).
 * On the first rejection j: draw from r(v) = max(p_j - q_j, 0) / Z with
 * q_j(v) = exp((U_j + code_j W2)[v] / T - lse_j) rebuilt on the fly; if Z = 0
 * (rounding only) draw from p_j.  If all l_r drafts are accepted: draw the
 * bonus token from p_{l_r + 1}.  Both draws go down a binary sum tree over
 * the vocabulary (depth ceil(log2 V)), one stream-2 uniform per level: at a
 * node with child masses (mL, mR) go left iff u * (mL + mR) < mL.
 * For T = 0: accept iff x_k equals argmax P_{k-1} (lowest index); the first
 * mismatch emits that argmax; a fully accepted block emits argmax P_{l_r}.
 * Outputs:
 *   out_tokens [R, gamma + 1] int32  accepted drafts then the new token, -1 padded
 *   accept_len [R]            int32  accepted drafts
 *   n_out      [R]            int32  accept_len + 1
 *   p_tok      [R, gamma]     float  p_k(x_k) for tested positions (may be NULL)
 *   lse_p      [R, gamma + 1] double log-sum-exp of P_k / T for rows read (may be NULL)
 * Rows the request never reads hold NaN in p_tok / lse_p.  The target rows
 * are read in windows of rows [0, 1), [1, 3), [3, 7), [7, gamma + 1): a
 * request reads the windows up to the one that holds its first rejection
 * (or its bonus row) and no further.
 * Requirements as for drafting (V <= 2^20; larger vocabularies return
 * DSPARK_ERR_SHAPE before anything is enqueued).
 */
int dspark_verify(const void* P, int p_dtype, const void* U, int u_dtype,
                  const void* W2, int w_dtype,
                  const int32_t* tokens, const float* q_tok, const double* lse,
                  const float* code, const int32_t* verify_len,
                  int R, int gamma, int V, int r,
                  uint64_t seed, const uint32_t* req_ids, float temperature,
                  int32_t* out_tokens, int32_t* accept_len, int32_t* n_out,
                  float* p_tok, double* lse_p,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_verify with a staging buffer for P, for targets read in place from
 * host memory (dspark_host_pointer): pass 1 copies every target row it reads
 * into p_stage, a device array of P's shape and dtype, and the passes after it
 * (acceptance, residual, sampling) read the target rows there, so each needed
 * byte crosses the host link once.  With p_stage the windows are one row each
 * ([k, k + 1)), so a request reads exactly rows 0 .. accept_len: p_tok holds
 * positions 1 .. min(accept_len + 1, l_r) and lse_p rows 0 .. accept_len, NaN
 * elsewhere; the tokens and lengths are those of dspark_verify.  p_stage may be
 * NULL (the same as dspark_verify).  Rows verification does not read are left
 * untouched.
 */
int dspark_verify_staged(const void* P, int p_dtype, const void* U, int u_dtype,
                         const void* W2, int w_dtype,
                         const int32_t* tokens, const float* q_tok, const double* lse,
                         const float* code, const int32_t* verify_len,
                         int R, int gamma, int V, int r,
                         uint64_t seed, const uint32_t* req_ids, float temperature,
                         int32_t* out_tokens, int32_t* accept_len, int32_t* n_out,
                         float* p_tok, double* lse_p, void* p_stage,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_verify_noalloc -- dspark_verify for callers that cannot allocate
 * device memory (no counterpart on the pages: it changes where scratch lives,
 * not what is computed).  Some callers are handed only their input and output
 * buffers -- a plugin inside another framework, an engine whose memory
 * planner owns the whole device, a path that must not pay for or synchronise
 * on an allocation -- so they have no workspace to pass.  This entry point
 * takes the same arguments as dspark_verify except the workspace, runs the
 * same kernels, and allocates nothing: its scratch is an 8 MiB array built
 * into the library, which every GPU that loads the library keeps until the
 * process exits.
 *  - Sizes whose workspace (dspark_verify_workspace_size) exceeds 8 MiB are
 *    rejected with DSPARK_ERR_SHAPE before any work is enqueued (the 5-token,
 *    256-request, 151936-word case needs about 4.4 MiB).
 *  - The first call on a device looks up the array's device address; make it
 *    before capturing a stream into a graph.
 *  - All calls share the array and leave their contents in it.  Calls whose
 *    work overlaps on the GPU race: order them (one stream, or events).
 *  - Each call clears the array's status word; device-side conditions
 *    (token ids outside [0, V)) are not reported by this variant.
 *  - `stream` must belong to the current device (the array's address is
 *    that device's); a stream of another device returns
 *    DSPARK_ERR_INVALID_ARG.
 */
int dspark_verify_noalloc(const void* P, int p_dtype, const void* U, int u_dtype,
                          const void* W2, int w_dtype,
                          const int32_t* tokens, const float* q_tok, const double* lse,
                          const float* code, const int32_t* verify_len,
                          int R, int gamma, int V, int r,
                          uint64_t seed, const uint32_t* req_ids, float temperature,
                          int32_t* out_tokens, int32_t* accept_len, int32_t* n_out,
                          float* p_tok, double* lse_p, void* stream);

/* --------------------------------------------------------------- schedule */

size_t dspark_schedule_workspace_size(int R, int gamma);

/*
 * Confidence scheduler (blog section 4.3; explainer section 04).
 *   c        [R, gamma]  float   calibrated confidences c_{r,j} in [0, 1]
 *   sps      [n_sps]     double  steps per second at token batch B = index;
 *                                entries past the table count as 0
 * a_{r,j} = c_{r,1} ... c_{r,j} (float32 product in position order).  The
 * candidates (r, j) with a > 0 are ordered by a descending, then r, then j
 * ascending; tau_n = R + a_(1) + ... + a_(n) (double), Theta(n) =
 * tau_n * SPS[R + n]; n* is the first n with Theta(n + 1) <= Theta(n)
 * (all candidates if none); l_r counts request r among the first n*.
 * Inputs are c and SPS only: the schedule never sees the target or the RNG.
 * Outputs: verify_len [R] int32, theta [1] double = Theta(n*), n_star [1] int32.
 * Requirements: 1 <= R, 1 <= gamma <= 64, R * gamma <= 8192, n_sps >= 1.
 */
int dspark_schedule(const float* c, const double* sps, int n_sps, int R, int gamma,
                    int32_t* verify_len, double* theta, int32_t* n_star,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * Production-style scheduler (explainer section 04: the capacity comes from
 * the predictions of two steps back, and the current candidates are ranked
 * into it, so a pipelined server never waits on the current step's stopping
 * rule).  Same inputs and ordering as dspark_schedule, plus
 *   budget  [1]  int32  (device) the capacity: the n_star that this call (or
 *                dspark_schedule) wrote two steps earlier; a negative value
 *                means no history yet and this step's own n* is used.
 * The candidates fill min(budget, number of candidates with a > 0) places:
 * verify_len counts each request's places, theta = tau * SPS[R + places],
 * and n_star receives this step's own synchronous n* (the capacity for two
 * steps later).  A caller keeps three n_star buffers in rotation and passes
 * the one of step t - 2 as the budget of step t: everything stays on the
 * device.  Errors as dspark_schedule; INVALID_ARG for a null budget.
 */
int dspark_schedule_async(const float* c, const double* sps, int n_sps, int R, int gamma,
                          const int32_t* budget, int32_t* verify_len, double* theta, int32_t* n_star,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * Threshold filter (blog section 4.3, the confidence-threshold sweep; the
 * explainer's section 04 sets the scheduler against one fixed threshold for
 * every request): request r verifies its longest prefix of positions whose
 * score is >= theta,
 *   mode 0: score a_{r,j} = c_{r,1} ... c_{r,j} (float32 product in position
 *           order, the scheduler's prefix survival)
 *   mode 1: score c_{r,j}
 * stopping at the first position that misses (a NaN score misses).
 *   c          [R, gamma]  float   (device)
 *   verify_len [R]         int32   output (device, caller-owned)
 * No workspace.  Requirements: R >= 1, 1 <= gamma <= 64, mode 0 or 1
 * (INVALID_ARG otherwise, or for a null pointer; SHAPE for the sizes).
 */
int dspark_schedule_threshold(const float* c, int R, int gamma, float theta, int mode,
                              int32_t* verify_len, void* stream);

/* -------------------------------------------------------------------- STS */

/*
 * Sequential Temperature Scaling (blog section 4.2): fit one temperature per
 * draft position on a calibration set, left to right.  The calibrated
 * confidence is c' = sigmoid(logit(c) / t_k), logit(c) = ln c - ln(1 - c).
 * Position k takes, from the grid, the t whose calibrated prefix survival
 * a'_{n,k} = c'_{n,1} ... c'_{n,k} (t_1 .. t_{k-1} already fixed) has the
 * smallest expected calibration error against the outcome accept_len[n] >= k
 * (Guo et al., ICML 2017, section 2: M equal-width bins over [0, 1], p = 1 in
 * the last bin, ECE = sum_b |B_b|/N |mean y - mean a'|); ties keep the lowest
 * grid index.
 *   c          [N, gamma]  float   raw confidences in [0, 1] (device)
 *   accept_len [N]         int32   accepted drafts of each calibration block
 *                                  (verification of all gamma positions)
 *   grid       [G]         double  candidate temperatures, positive (device)
 * Outputs (device, caller-owned), per position: t_out [gamma] double,
 * g_out [gamma] int32 (grid index), ece_out [gamma] double (the minimum),
 * gap_out [gamma] double (second-smallest ECE minus the minimum; +inf if G = 1).
 * Precision: the calibrated prefix survival is formed in float32, except that
 * a value within 1e-4 bin widths of a bin edge is formed again in double
 * (which bin it joins is decided as in double arithmetic); the prefix
 * survival carried between positions is double; per-bin sums are exact
 * (sums of p as integers of 2^-32).  The ECE values are accurate to about
 * 1e-7; a position whose gap is below that may pick either neighbour.
 * Requirements: 1 <= N <= 2^24, 1 <= gamma <= 64, 1 <= G <= 4096, 1 <= M <= 32
 * (SHAPE otherwise), workspace of dspark_sts_workspace_size bytes (256-byte
 * aligned).
 */
size_t dspark_sts_workspace_size(int N, int gamma, int G, int M);
int dspark_sts_fit(const float* c, const int32_t* accept_len, int N, int gamma,
                   const double* grid, int G, int M,
                   double* t_out, int32_t* g_out, double* ece_out, double* gap_out,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * Apply per-position temperatures: out[n,k] = sigmoid(logit(c[n,k]) / t[k])
 * in float32 (c = 0 and c = 1 stay put).  c, out [N, gamma] float, t [gamma]
 * double, all device.  No workspace.
 */
int dspark_sts_apply(const float* c, int N, int gamma, const double* t, float* out, void* stream);

/* ---------------------------------------------------------------- random */

/*
 * The device's Philox4x32-10 block function (Salmon et al., SC'11, the
 * generator every random decision above draws from), for known-answer
 * checks of the copy the kernels use.  For i < n:
 *   out[4i .. 4i+3] = Philox4x32-10(counter ctr[4i .. 4i+3], key key[2i .. 2i+1])
 * ctr [n, 4], key [n, 2] and out [n, 4] are uint32 device arrays
 * (caller-owned; ctr and out 16-byte aligned, key 8-byte aligned); the work
 * is enqueued on `stream`.  Errors: SHAPE for n < 1, INVALID_ARG for a null
 * or misaligned pointer, CUDA if the launch fails.
 */
int dspark_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int n, void* stream);

/* -------------------------------------------------------------- profiling */

/*
 * Kernel timing for benchmarks (no counterpart on the pages).  While enabled
 * (on != 0), every kernel the library launches is bracketed by two CUDA
 * events recorded on the caller's stream; dspark_profile_collect()
 * synchronises those events and returns, per launch in issue order, a kernel
 * name id and its device time in milliseconds (at most `cap` entries; the
 * return value is the number of launches recorded, which may exceed `cap`),
 * then forgets them.  dspark_profile_kernel_name() maps an id to its name.
 * Disabled by default; costs two event records per launch when enabled.
 * Host-side state, not thread-safe.
 */
int dspark_profile_enable(int on);
int dspark_profile_collect(int32_t* name_ids, float* ms, int cap);
const char* dspark_profile_kernel_name(int name_id);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H */
