// verify.cu -- lossless rejection-sampling verification.
//
// DSpark explainer, section 05: with p the target distribution and q the
// draft distribution actually used (including the sequential head's bias),
// x ~ q is accepted with alpha(x) = min(1, p(x)/q(x)); on rejection the new
// token comes from r(v) = max(p(v) - q(v), 0) / sum_u max(p(u) - q(u), 0).
// Blog section 1 and explainer section 02: everything after the first
// rejection is discarded, and a fully accepted block earns one bonus token
// from the target; the greedy teaching version (T = 0) accepts on exact match
// and replaces the first mismatch by the target's argmax.
//
// Kernels (one stream):
//   pass1     stream every target row the request verifies (rows 0..l_r)
//             once, 1024-wide chunks: (max, sum exp) of P/T, or (max, argmax)
//   accept    one warp per request: lse of each row, p(x_k), the acceptance
//             scan with stream-1 uniforms; decides residual / bonus / done
//   residual  rejecting requests only: w = max(p_j - q_j, 0) over the row,
//             q_j rebuilt from U_j, code_j W2 and lse_j; per-chunk mass
//   sample    one CTA per request that still needs a token: descend the
//             binary sum tree (chunk masses above, exact element weights in
//             double inside the chosen chunk), one stream-2 uniform a level
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace dspark {

bool verify_tc_supported(const VerifyArgs& a);
cudaError_t launch_verify_tc_residual(VerifyArgs& a, cudaStream_t s);

// exp(a) for a double argument without double-precision transcendentals:
// exp(a_hi) in float times the first-order correction for a - a_hi
// (relative error about 1e-7 for |a| < 80).  exp(-inf) = 0: a masked logit
// (-inf) has no mass, and neither has an argument that underflows.
__device__ __forceinline__ double exp_from_double(double a) {
    const float ah = (float)a;
    const float e = expf(ah);
    return e == 0.f ? 0.0 : (double)e * (1.0 + (a - (double)ah));
}

__device__ __forceinline__ int verify_len_of(const VerifyArgs& A, int r) {
    if (!A.verify_len) return A.gamma;
    int L = A.verify_len[r];
    return L < 0 ? 0 : (L > A.gamma ? A.gamma : L);
}

// ------------------------------------------------------------------ waves
// Verification reads the target rows in waves: a request needs row k
// (0-based) only while positions 1..k were all accepted, and row L (the
// bonus row) only when all L were.  Wave w covers rows [lo_w, hi_w) of the
// requests still live (all of them in wave 1); its pass 1 streams those rows,
// its acceptance pass decides every live request on them and lists the ones
// that passed the whole window for the next wave.
// Windows [0, 1), [1, 3), [3, 7), [7, gamma + 1) for P in device memory (of
// the edge sets timed on the 256-request, gamma = 5 workload, the fastest:
// fewer rows read than wider first windows, fewer launches than a window per
// row).  With P in host memory every row read crosses the host link, which
// bounds the call, so there each wave is one row: [w - 1, w), and only the
// rows the decisions need are read.
__host__ __device__ __forceinline__ int wave_lo(int w, bool unit) {
    if (unit) return w - 1;
    return w <= 1 ? 0 : (w == 2 ? 1 : (w == 3 ? 3 : 7));
}
__host__ __device__ __forceinline__ int wave_hi(int w, int G1, bool unit) {
    const int e = unit ? w : (w <= 1 ? 1 : (w == 2 ? 3 : (w == 3 ? 7 : G1)));
    return e < G1 ? e : G1;
}
__host__ __device__ __forceinline__ int wave_count(int G1, bool unit) {
    int n = 0;
    while (n < (unit ? G1 : 4) && wave_lo(n + 1, unit) < G1) ++n;
    return n;
}
__host__ __device__ __forceinline__ int live_count(const VerifyArgs& A, int w) {
    return w == 1 ? A.R : A.wcount_alive[w];
}
__device__ __forceinline__ int live_request(const VerifyArgs& A, int w, int i) {
    return w == 1 ? i : A.alive[(size_t)(w & 1) * A.R + i];
}

// The counter block of the workspace: rej_count (+0), vflags (+16), live
// requests per wave (+32: gamma + 2 ints).  The first pass-1 launch of a
// call clears it (block 0, before it lets the acceptance pass launch).
constexpr size_t kCounterBytes = 512;
static_assert(32 + 4 * (64 + 2) <= kCounterBytes, "wave counters");

// ------------------------------------------------------------------ pass 1
// Warp tasks over (live request, row of the window, 1024-column chunk).
// STAGE: also copy each row read into A.P_stage (P is host memory, and the
// later passes read the rows from there instead of across the link again).
template <int PT, bool GREEDY, bool STAGE>
__global__ void __launch_bounds__(256) verify_pass1(VerifyArgs A, int w) {
    // wave 1 is the call's first kernel, launched after all earlier work:
    // its block 0 clears the counters before any acceptance pass can start
    if (w == 1 && blockIdx.x == 0)
        for (int i = threadIdx.x; i < (int)(kCounterBytes / 4); i += blockDim.x) A.rej_count[i] = 0;
    pdl_launch_dependents();
    pdl_wait();   // the list of live requests (waves after the first)
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * (blockDim.x >> 5);
    const int V = A.V, G1 = A.gamma + 1, NCH = A.nch;
    const int lo = wave_lo(w, A.unit_waves), nrow = wave_hi(w, G1, A.unit_waves) - lo;
    const long long tasks = (long long)live_count(A, w) * nrow * NCH;
    const float invT = GREEDY ? 1.f : 1.f / A.T;
    for (long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < tasks;
         task += warps_total) {
        const int ch = (int)(task % NCH);
        const long long rr = task / NCH;
        const int row = lo + (int)(rr % nrow);
        const int r = live_request(A, w, (int)(rr / nrow));
        if (row > verify_len_of(A, r)) continue;            // warp-uniform
        const size_t base = ((size_t)r * G1 + row) * (size_t)V;
        const int c0 = ch * kChunk;
        float x[32];
        bool ok[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + 4 * lane + 128 * i;
            ok[i] = c < V;
            float4 v = ok[i] ? load4_stream<PT>(A.P, base + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            x[4 * i + 0] = v.x;
            x[4 * i + 1] = v.y;
            x[4 * i + 2] = v.z;
            x[4 * i + 3] = v.w;
        }
        if (STAGE) {
            // stored after all eight loads are issued: the staging buffer
            // might alias P as far as the compiler knows
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (ok[i])
                    store4<PT>(A.P_stage, base + c0 + 4 * lane + 128 * i,
                               make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]));
        }
        float2 out;
        if (GREEDY) {
            float best = -INFINITY;
            int arg = INT_MAX;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + 4 * lane + 128 * i + q;
                    const float y = x[4 * i + q];
                    if (ok[i] && (y > best || (y == best && c < arg))) {
                        best = y;
                        arg = c;
                    }
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
                const int a2 = __shfl_xor_sync(0xffffffffu, arg, o);
                if (b2 > best || (b2 == best && a2 < arg)) {
                    best = b2;
                    arg = a2;
                }
            }
            out = make_float2(best, __int_as_float(arg));
        } else {
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (ok[i]) m = fmaxf(m, x[4 * i + q] * invT);
            const float mw = warp_max(m);
            // a chunk of masked logits only (all -inf) has no mass: (-inf, 0)
            const float mr = mw == -INFINITY ? 0.f : mw;
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (ok[i]) s += ex2_approx((x[4 * i + q] * invT - mr) * kLog2e);
            s = warp_sum(s);
            out = make_float2(mw, s);
        }
        if (lane == 0) A.vparts[((size_t)r * G1 + row) * NCH + ch] = out;
    }
}

// ------------------------------------------------------------------ accept
// One CTA per request; in wave w only the requests still undecided
// (live_mark[r] == w, every request in wave 1) go past the wait.  The
// drafted tokens, their target logits P_k[x_k], q(x_k) and the acceptance
// uniforms are inputs of the call, so they are fetched before the wait,
// under the tail of pass 1.  After it, warp v reduces the window's rows
// lo + v, lo + v + 8, ... of pass 1's partials (the log-sum-exp of each P
// row, or its argmax at T = 0); then every position of the window is tested
// at once and the first rejection decides (everything after it is
// discarded).  A request that passes the whole window goes to the next
// wave's list, unless the window held its bonus row.
template <int PT, bool GREEDY>
__global__ void __launch_bounds__(256) verify_accept(VerifyArgs A, int w) {
    __shared__ double s_lse[65];
    __shared__ int s_arg[65];
    __shared__ int s_x[64];
    __shared__ float s_px[64];
    __shared__ int s_first;
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int r = blockIdx.x;
    const int G1 = A.gamma + 1, NCH = A.nch, V = A.V;
    const int L = verify_len_of(A, r);
    const int lo = wave_lo(w, A.unit_waves), hi = wave_hi(w, G1, A.unit_waves);
    const int rhi = min(hi - 1, L);        // the window's rows this request needs: lo .. rhi
    const int npos = min(hi, L) - lo;      // positions lo + 1 .. lo + npos are tested
    const float invT = GREEDY ? 1.f : 1.f / A.T;
    const bool staged = A.Pv != A.P;       // P_stage is filled by pass 1: read it after the wait
    int x = 0;
    bool bad_x = false;
    float px_raw = 0.f, qx = 1.f;
    double u = 0.0;
    if (tid < npos) {
        const int row = lo + tid, k = row + 1;
        x = A.tokens[(size_t)r * A.gamma + row];
        if (x < 0 || x >= V) {
            bad_x = true;
            x = 0;
        }
        if (!GREEDY) {
            if (!staged) px_raw = ld_elem(A.P, PT, ((size_t)r * G1 + row) * (size_t)V + x);
            qx = A.q_tok[(size_t)r * A.gamma + row];
            const uint32_t req = A.req_ids ? A.req_ids[r] : (uint32_t)r;
            u = rng_uniform_d(philox_key(A.seed), req, (uint32_t)k, 1u, 0u);
        }
    }
    pdl_wait();
    if (w > 1 && A.live_mark[r] != w) return;
    int32_t* out = A.out_tokens + (size_t)r * G1;
    if (w == 1 && tid < G1) {
        // outputs start empty; lse_p rows computed in this wave are written below
        out[tid] = -1;
        if (A.lse_p && (GREEDY || tid > rhi)) A.lse_p[(size_t)r * G1 + tid] = NAN;
        if (A.p_tok && tid < A.gamma) A.p_tok[(size_t)r * A.gamma + tid] = NAN;
    }
    if (tid == 0) s_first = INT_MAX;
    if (tid < npos) {
        const int row = lo + tid;
        if (bad_x) raise_status(A.ws, kStatBadToken);
        s_x[row] = x;
        if (!GREEDY) s_px[row] = staged ? ld_elem(A.Pv, PT, ((size_t)r * G1 + row) * (size_t)V + x) : px_raw;
    }
    const float2* parts = A.vparts + (size_t)r * G1 * NCH;
    for (int row = lo + warp; row <= rhi; row += blockDim.x >> 5) {
        const float2* pr = parts + (size_t)row * NCH;
        if (GREEDY) {
            float best = -INFINITY;
            int arg = INT_MAX;
            for (int c = lane; c < NCH; c += 32) {
                const float2 p = pr[c];
                const int a2 = __float_as_int(p.y);
                if (p.x > best || (p.x == best && a2 < arg)) {
                    best = p.x;
                    arg = a2;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
                const int a2 = __shfl_xor_sync(0xffffffffu, arg, o);
                if (b2 > best || (b2 == best && a2 < arg)) {
                    best = b2;
                    arg = a2;
                }
            }
            if (lane == 0) s_arg[row] = (arg < 0 || arg >= V) ? 0 : arg;
        } else {
            float m = -INFINITY;
            for (int c = lane; c < NCH; c += 32) m = fmaxf(m, pr[c].x);
            m = warp_max(m);
            double sum = 0.0;
            for (int c = lane; c < NCH; c += 32) {
                const float2 p = pr[c];
                sum += (double)p.y * (double)expf(p.x - m);      // exact difference: both are float maxima
            }
            sum = warp_sum_d(sum);
            if (lane == 0) {
                // log(sum) = e ln 2 + log(mant), mant in [1/2, 1): only the
                // mantissa's logarithm is taken, in float (error ~1e-7)
                int e = 0;
                const double mant = frexp(sum, &e);
                const double l = ((double)m + (double)e * 0.69314718055994531) + (double)logf((float)mant);
                s_lse[row] = l;
                A.lsep_ws[(size_t)r * G1 + row] = l;
                if (A.lse_p) A.lse_p[(size_t)r * G1 + row] = l;
            }
        }
    }
    __syncthreads();
    // position k = lo + tid + 1: accept or reject
    double px = 0.0;
    if (tid < npos) {
        const int row = lo + tid, k = row + 1;
        bool rej;
        if (GREEDY) {
            rej = s_x[row] != s_arg[row];
        } else {
            // p(x) = exp(P_x / T - lse_P), the difference formed in double
            px = exp_from_double((double)s_px[row] * (double)invT - s_lse[row]);
            const double ratio = px / (double)qx;
            rej = !(u < ratio);
        }
        if (rej) atomicMin(&s_first, k);
    }
    __syncthreads();
    const int j = s_first == INT_MAX ? 0 : s_first;      // first rejected position, 0 if none
    if (tid < npos) {
        const int row = lo + tid, k = row + 1;
        if (!GREEDY && A.p_tok && (!j || k <= j)) A.p_tok[(size_t)r * A.gamma + row] = (float)px;
        if (!j || k < j) out[row] = s_x[row];
        else if (GREEDY && k == j) out[row] = s_arg[row];   // the target's own token replaces x_j
    }
    if (tid == 0) {
        A.live_mark[r] = 0;
        if (j) {
            A.vstate[r] = GREEDY ? make_int2(kModeDone, 0) : make_int2(kModeResidual, j);
            A.accept_len[r] = j - 1;
            A.n_out[r] = j;
        } else if (L < hi) {
            // all L drafts accepted and the bonus row was in this window
            if (GREEDY) {
                out[L] = s_arg[L];
                A.vstate[r] = make_int2(kModeDone, 0);
            } else {
                A.vstate[r] = make_int2(kModeBonus, L + 1);
            }
            A.accept_len[r] = L;
            A.n_out[r] = L + 1;
        } else {
            A.live_mark[r] = w + 1;
            const int slot = atomicAdd(A.wcount_alive + w + 1, 1);
            A.alive[(size_t)((w + 1) & 1) * A.R + slot] = r;
        }
    }
    if (GREEDY || !j) return;
    // queue the rejecting request for the residual pass with its code e_j as
    // three bf16 terms hi + mid + lo (exact for f32: each term takes the next
    // 8 significand bits; mid = lo = 0 when e_j is bf16-exact)
    __shared__ int s_slot;
    if (tid == 0) {
        const int slot = atomicAdd(A.rej_count, 1);
        A.rej_list[slot] = r;
        s_slot = slot;
    }
    __syncthreads();
    const int slot = s_slot;
    const float* e = A.code + ((size_t)r * A.gamma + (j - 1)) * A.r;
    const size_t plane = (size_t)((A.R + 127) / 128) * 128 * A.r;
    bool inexact = false;
    for (int i = tid; i < A.r; i += blockDim.x) {
        const float v = e[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(h);
        const __nv_bfloat16 m = __float2bfloat16_rn(r1);
        const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
        uint16_t* dst = A.a_res + (size_t)slot * A.r + i;
        dst[0] = __bfloat16_as_ushort(h);
        dst[plane] = __bfloat16_as_ushort(m);
        dst[2 * plane] = __bfloat16_as_ushort(l);
        inexact |= r1 != 0.f;
    }
    if (__syncthreads_or(inexact) && tid == 0) atomicOr(A.vflags, 1u);
}

// ------------------------------------------------------------------ residual (generic)
// Rejecting requests only: w = max(p_j - q_j, 0) over the row, with
// B = e_j W2 on CUDA cores, for the shapes the tensor-core pass does not take.
// One CTA task = (1024 columns, request); the mass of each 256-column chunk
// goes to rpart[r][c][0].
template <int PT, int UT, int WT>
__global__ void __launch_bounds__(256) verify_residual_generic(VerifyArgs A) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ float e_sh[];
    __shared__ double sh[8];
    const int V = A.V, G1 = A.gamma + 1;
    const float invT = 1.f / A.T;
    const long long tasks = (long long)A.nch * A.R;
    for (long long task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int ch = (int)(task % A.nch), r = (int)(task / A.nch);
        const int2 st = A.vstate[r];
        if (st.x != kModeResidual) continue;                     // block-uniform
        const int j = st.y;
        __syncthreads();
        for (int i = threadIdx.x; i < A.r; i += blockDim.x)
            e_sh[i] = A.code[((size_t)r * A.gamma + (j - 1)) * A.r + i];
        __syncthreads();
        const int c = ch * kChunk + 4 * threadIdx.x;
        double wsum = 0.0;
        if (c < V) {
            float b[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = 0; i < A.r; ++i) {
                const float4 w = load4<WT>(A.W2, (size_t)i * V + c);
                const float ei = e_sh[i];
                b[0] = fmaf(ei, w.x, b[0]);
                b[1] = fmaf(ei, w.y, b[1]);
                b[2] = fmaf(ei, w.z, b[2]);
                b[3] = fmaf(ei, w.w, b[3]);
            }
            const double lq = A.lse[(size_t)r * A.gamma + (j - 1)];
            const double lp = A.lsep_ws[(size_t)r * G1 + (j - 1)];
            const float lq_hi = (float)lq, lq_lo = (float)(lq - (double)lq_hi);
            const float lp_hi = (float)lp, lp_lo = (float)(lp - (double)lp_hi);
            const float4 u4 = load4<UT>(A.U, ((size_t)r * A.gamma + (j - 1)) * V + c);
            const float4 p4 = load4<PT>(A.Pv, ((size_t)r * G1 + (j - 1)) * V + c);
            const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
            const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float qv = expf(((uu[q] + b[q]) * invT - lq_hi) - lq_lo);
                const float pv = expf((pp[q] * invT - lp_hi) - lp_lo);
                const float w = pv - qv;
                wsum += w > 0.f ? (double)w : 0.0;
            }
        }
        // 64 threads cover one 256-column chunk: two warps each
        wsum = warp_sum_d(wsum);
        if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = wsum;
        __syncthreads();
        if (threadIdx.x < 4) {
            const int c256 = ch * 4 + threadIdx.x;
            if (c256 < A.nch256) {
                float4* dst = reinterpret_cast<float4*>(A.rpart + ((size_t)r * A.nch256 + c256) * 4);
                *dst = make_float4((float)(sh[2 * threadIdx.x] + sh[2 * threadIdx.x + 1]), 0.f, 0.f, 0.f);
            }
        }
    }
}

// ------------------------------------------------------------------ sample
// Inverse CDF down the binary sum tree over leaves[0 .. 2^levels), levels
// <= 10: node k of the heap (root 1, children 2k and 2k + 1, leaf i = node
// 2^levels + i) at depth d holds the mass under it, and the walk goes right
// at k unless u_level[d] (mL + mR) < mL.  The uniforms do not depend on the
// path, so neither do the decisions: each is taken while its node is built.
// Eight warps build their own subtrees with warp barriers only, thread 0 the
// few nodes above them, then follows the decision bytes down from the root.
// *out receives the chosen leaf and *root the leaves' total.  Every thread
// of the (256-thread) block must call it.
__device__ void tree_descend(const double* leaves, double* tree, uint8_t* go_right, int levels,
                             const double* u_level, int* out, double* root) {
    const int n = 1 << levels;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ls = levels >= 3 ? 3 : 0;          // log2 of the number of subtrees
    const int S = 1 << ls;
    auto mass = [&](int k) { return k >= n ? leaves[k - n] : tree[k]; };
    auto build = [&](int k, int d) {
        const double mL = mass(2 * k), mR = mass(2 * k + 1);
        const double m = mL + mR;
        tree[k] = m;
        go_right[k] = (u_level[d] * m < mL) ? 0 : 1;
    };
    if (warp < S) {
        for (int h = levels - 1; h >= ls; --h) {     // depth h: nodes [2^h, 2^(h+1)), 2^(h-ls) per subtree
            const int per = 1 << (h - ls);
            const int k0 = (1 << h) + warp * per;
            for (int i = lane; i < per; i += 32) build(k0 + i, h);
            __syncwarp();
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int h = ls - 1; h >= 0; --h)
            for (int k = 1 << h; k < (2 << h); ++k) build(k, h);
        int node = 1;
        for (int d = 0; d < levels; ++d) node = 2 * node + go_right[node];
        *out = levels > 0 ? node - n : 0;
        *root = levels > 0 ? tree[1] : leaves[0];
    }
}

// Mass of one 256-column residual chunk: the float sum of its four quarter
// masses (as residual_tc wrote them), in double.
__device__ __forceinline__ double rchunk_mass(float4 q) { return (double)((q.x + q.y) + (q.z + q.w)); }

template <int PT, int UT, int WT>
__global__ void __launch_bounds__(256) verify_sample(VerifyArgs A) {
    __shared__ double cm[1024];          // leaves: top-tree leaf masses first, then leaf weights
    __shared__ double tree[1024];        // inner nodes of the sum tree over cm
    __shared__ uint8_t go_right[1024];   // the walk's decision at every inner node
    __shared__ float e_sh[1024];
    __shared__ double s_u[32];           // the uniform of every tree level
    __shared__ int s_leaf, s_chunk;
    __shared__ double s_root;
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    const int2 st = A.vstate[r];
    if (st.x == kModeDone) return;
    const int mode = st.x, pos = st.y;
    const int V = A.V, G1 = A.gamma + 1;
    const int L = ceil_log2_i(V);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t req = A.req_ids ? A.req_ids[r] : (uint32_t)r;
    if (tid < L) s_u[tid] = rng_uniform_d(philox_key(A.seed), req, (uint32_t)pos, 2u, (uint32_t)tid);
    const double lp = A.lsep_ws[(size_t)r * G1 + (pos - 1)];
    // The tree over the 2^L leaves (columns) is walked in pieces: the top
    // levels over chunk masses, then inside the chosen chunk over exact
    // leaf weights.  `above` counts the levels walked before the chunk.
    bool use_p = mode != kModeResidual;
    int clog = kChunkLog2, above = 0;
    if (!use_p) {
        // residual: masses of the 256-column chunks of max(p_j - q_j, 0); with
        // more than 1024 chunks (V > 2^18) a top-tree leaf is a group of 2^lg
        // neighbouring chunks, its mass their pairwise sum
        for (int i = tid; i < A.r; i += blockDim.x) e_sh[i] = A.code[((size_t)r * A.gamma + (pos - 1)) * A.r + i];
        clog = kRChunkLog2;
        const int Lc = L > kRChunkLog2 ? L - kRChunkLog2 : 0;
        const int Ltop = Lc < 10 ? Lc : 10;
        const int lg = Lc - Ltop;                      // 0, 1 or 2
        const int ntop = 1 << Ltop;
        const float4* rp = reinterpret_cast<const float4*>(A.rpart) + (size_t)r * A.nch256;
        float4 q[4][4];                                // [leaf of this thread][chunk of the leaf]
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int c = ((tid + 256 * t) << lg) + g;
                const bool in = tid + 256 * t < ntop && g < (1 << lg) && c < A.nch256;
                q[t][g] = in ? rp[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int c = tid + 256 * t;
            if (c < ntop) {
                const double m0 = rchunk_mass(q[t][0]), m1 = rchunk_mass(q[t][1]);
                const double m2 = rchunk_mass(q[t][2]), m3 = rchunk_mass(q[t][3]);
                cm[c] = lg == 0 ? m0 : (lg == 1 ? m0 + m1 : (m0 + m1) + (m2 + m3));
            }
        }
        __syncthreads();
        tree_descend(cm, tree, go_right, Ltop, s_u, &s_leaf, &s_root);
        __syncthreads();
        if (s_root > 0.0) {
            if (tid == 0) {
                // the levels inside a group of chunks (none unless V > 2^18)
                const int base = s_leaf << lg;
                int sub = 0;
                if (lg > 0) {
                    double m[4];
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        m[g] = (g < (1 << lg) && base + g < A.nch256) ? rchunk_mass(rp[base + g]) : 0.0;
                    if (lg == 1) {
                        sub = (s_u[Ltop] * (m[0] + m[1]) < m[0]) ? 0 : 1;
                    } else {
                        const double a0 = m[0] + m[1], a1 = m[2] + m[3];
                        const int h = (s_u[Ltop] * (a0 + a1) < a0) ? 0 : 1;
                        sub = 2 * h + ((s_u[Ltop + 1] * (m[2 * h] + m[2 * h + 1]) < m[2 * h]) ? 0 : 1);
                    }
                }
                s_chunk = base + sub;
            }
            above = Lc;
        } else {
            use_p = true;                  // empty residual (rounding only): draw from p_j
        }
    }
    if (use_p) {
        clog = kChunkLog2;
        above = L > kChunkLog2 ? L - kChunkLog2 : 0;
        for (int c = tid; c < (1 << above); c += blockDim.x) {
            double m = 0.0;
            if (c < A.nch) {
                const float2 p2 = A.vparts[((size_t)r * G1 + (pos - 1)) * A.nch + c];
                m = (double)p2.y * exp_from_double((double)p2.x - lp);
            }
            cm[c] = m;
        }
        __syncthreads();
        tree_descend(cm, tree, go_right, above, s_u, &s_chunk, &s_root);
    }
    __syncthreads();
    const int chunk = s_chunk;
    // exact leaf weights of the chosen chunk, in double; the P (and U) values
    // of this thread's columns are fetched first
    const int Lbot = L - above;
    const int nleaf = 1 << Lbot;           // <= 256 (residual) or 1024 (p)
    const double invT = 1.0 / (double)A.T;
    float pvals[4], uval = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int i = tid + t * 256;
        const int v = (chunk << clog) + i;
        pvals[t] = (i < nleaf && v < V) ? ld_elem(A.Pv, PT, ((size_t)r * G1 + (pos - 1)) * V + v) : 0.f;
    }
    if (!use_p && tid < nleaf && (chunk << clog) + tid < V)
        uval = ld_elem(A.U, UT, ((size_t)r * A.gamma + (pos - 1)) * V + (chunk << clog) + tid);
    // residual: B = e W2 on the chunk's (at most 256) columns.  Warp w takes
    // rank rows w, w + 8, ..., lane l columns 8l .. 8l + 7, a batch of rows'
    // loads in flight at once; the warps' sums are added in a fixed order.
    __shared__ float s_b[8][kRChunk];
    if (!use_p) {
        constexpr int kBatch = WT == DSPARK_BF16 ? 16 : 8;
        const int c0 = (chunk << clog) + 8 * lane;
        float b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int i0 = warp; i0 < A.r; i0 += kBatch * 8) {
            Row8<WT> w[kBatch];
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
                const int i = i0 + 8 * t;
                w[t].load(A.W2, (size_t)i * V + c0, i < A.r ? V - c0 : 0);
            }
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
                const int i = i0 + 8 * t;
                const float ei = i < A.r ? e_sh[i] : 0.f;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) b[jj] = fmaf(ei, w[t].get(jj), b[jj]);
            }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) s_b[warp][8 * lane + jj] = b[jj];
        __syncthreads();
    }
    const double lq = (mode == kModeResidual) ? A.lse[(size_t)r * A.gamma + (pos - 1)] : 0.0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int i = tid + t * 256;
        if (i >= nleaf) break;
        const int v = (chunk << clog) + i;
        double w = 0.0;
        if (v < V) {
            const double pv = exp_from_double((double)pvals[t] * invT - lp);
            if (use_p) {
                w = pv;
            } else {
                float b = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) b += s_b[w8][i];
                const double z = ((double)uval + (double)b) * invT;
                const double qv = exp_from_double(z - lq);
                w = pv > qv ? pv - qv : 0.0;
            }
        }
        cm[i] = w;
    }
    __syncthreads();
    tree_descend(cm, tree, go_right, Lbot, s_u + above, &s_leaf, &s_root);
    __syncthreads();
    if (tid == 0) {
        int y = (chunk << clog) + s_leaf;
        if (y >= V) y = V - 1;
        A.out_tokens[(size_t)r * G1 + (pos - 1)] = y;
    }
}

// ------------------------------------------------------------------ host
static int nch_of(int V) { return (V + kChunk - 1) / kChunk; }
static int nch256_of(int V) { return (V + kRChunk - 1) / kRChunk; }

size_t verify_workspace_bytes(int R, int gamma, int V, int r) {
    const int G1 = gamma + 1, NCH = nch_of(V), N2 = nch256_of(V);
    size_t off = sizeof(WsHeader);
    off = align_up(off + (size_t)R * G1 * NCH * sizeof(float2), 256);   // vparts
    off = align_up(off + (size_t)R * G1 * sizeof(double), 256);         // lse of P rows
    off = align_up(off + (size_t)R * sizeof(int2), 256);                // vstate
    off = align_up(off + (size_t)R * N2 * 4 * sizeof(float), 256);      // rpart
    off = align_up(off + kCounterBytes, 256);                            // counters, flags
    off = align_up(off + (size_t)R * sizeof(int), 256);                 // rej_list
    off = align_up(off + 2ull * R * sizeof(int), 256);                  // live requests of the waves
    off = align_up(off + (size_t)R * sizeof(int), 256);                 // live_mark
    const size_t rpad = (size_t)((R + 127) / 128) * 128;
    off = align_up(off + 3 * rpad * r * sizeof(uint16_t), 256);          // a_res: hi, mid, lo planes
    return off;
}

int verify_carve(VerifyArgs& a, size_t ws_bytes) {
    if (ws_bytes < verify_workspace_bytes(a.R, a.gamma, a.V, a.r)) return DSPARK_ERR_WORKSPACE;
    const int G1 = a.gamma + 1, NCH = nch_of(a.V), N2 = nch256_of(a.V);
    a.nch = NCH;
    a.nch256 = N2;
    char* base = static_cast<char*>(a.ws);
    size_t off = sizeof(WsHeader);
    a.vparts = reinterpret_cast<float2*>(base + off);
    off = align_up(off + (size_t)a.R * G1 * NCH * sizeof(float2), 256);
    a.lsep_ws = reinterpret_cast<double*>(base + off);
    off = align_up(off + (size_t)a.R * G1 * sizeof(double), 256);
    a.vstate = reinterpret_cast<int2*>(base + off);
    off = align_up(off + (size_t)a.R * sizeof(int2), 256);
    a.rpart = reinterpret_cast<float*>(base + off);
    off = align_up(off + (size_t)a.R * N2 * 4 * sizeof(float), 256);
    // counters cleared before each verification (one block): rejection
    // count, flags, live requests per wave (up to gamma + 2 <= 66 entries)
    a.rej_count = reinterpret_cast<int*>(base + off);
    a.vflags = reinterpret_cast<uint32_t*>(base + off + 16);
    a.wcount_alive = reinterpret_cast<int*>(base + off + 32);
    off = align_up(off + kCounterBytes, 256);
    a.rej_list = reinterpret_cast<int*>(base + off);
    off = align_up(off + (size_t)a.R * sizeof(int), 256);
    a.alive = reinterpret_cast<int*>(base + off);
    off = align_up(off + 2ull * a.R * sizeof(int), 256);
    a.live_mark = reinterpret_cast<int*>(base + off);
    off = align_up(off + (size_t)a.R * sizeof(int), 256);
    a.a_res = reinterpret_cast<uint16_t*>(base + off);
    return DSPARK_OK;
}

template <int PT, int UT, int WT>
static cudaError_t launch_typed(VerifyArgs& a, cudaStream_t s) {
    const bool greedy = !(a.T > 0.f);
    const int nsm = num_sms();
    const int G1 = a.gamma + 1;
    cudaError_t e = cudaSuccess;
    a.unit_waves = a.P_stage ? 1 : 0;
    const bool unit = a.unit_waves != 0;
    // the waves: the first pass 1 waits for the caller's work (and the
    // cleared counters); every later launch overlaps the previous kernel's tail
    const int nw = wave_count(G1, unit);
    // pass 1 keeps its loads in registers (32 floats a lane), so the number
    // of resident warps bounds the bytes in flight: five 256-thread CTAs per
    // SM at 48 registers (four for the staging variant, at 58)
    const long long per_sm = a.P_stage ? 4 : 5;
    for (int w = 1; w <= nw; ++w) {
        const long long tasks = (long long)a.R * (wave_hi(w, G1, unit) - wave_lo(w, unit)) * a.nch;
        const long long want = (tasks + 7) / 8;
        int grid = (int)(want < (long long)nsm * per_sm ? want : (long long)nsm * per_sm);
        if (grid < 1) grid = 1;
        prof_begin(kPVerifyPass1, s);
        if (a.P_stage)
            e = greedy ? launch_kernel(verify_pass1<PT, true, true>, dim3(grid), dim3(256), 0, s, w > 1, a, w)
                       : launch_kernel(verify_pass1<PT, false, true>, dim3(grid), dim3(256), 0, s, w > 1, a, w);
        else
            e = greedy ? launch_kernel(verify_pass1<PT, true, false>, dim3(grid), dim3(256), 0, s, w > 1, a, w)
                       : launch_kernel(verify_pass1<PT, false, false>, dim3(grid), dim3(256), 0, s, w > 1, a, w);
        prof_end(s);
        if (e != cudaSuccess) return e;
        prof_begin(kPVerifyAccept, s);
        e = greedy ? launch_kernel(verify_accept<PT, true>, dim3(a.R), dim3(256), 0, s, true, a, w)
                   : launch_kernel(verify_accept<PT, false>, dim3(a.R), dim3(256), 0, s, true, a, w);
        prof_end(s);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (greedy) return cudaSuccess;
    a.tc = verify_tc_supported(a) ? 1 : 0;
    if (a.tc) {
        e = launch_verify_tc_residual(a, s);
        if (e != cudaSuccess) return e;
    } else {
        // CUDA-core residual for the shapes the tensor-core pass does not take
        const long long rt = (long long)a.nch * a.R;
        const int g2 = (int)(rt < (long long)nsm * 8 ? rt : (long long)nsm * 8);
        prof_begin(kPVerifyResidualGeneric, s);
        e = launch_kernel(verify_residual_generic<PT, UT, WT>, dim3(g2 > 0 ? g2 : 1), dim3(256), a.r * sizeof(float),
                          s, true, a);
        prof_end(s);
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    // the sampling pass starts after the residual pass has finished: with
    // programmatic overlap the whole cycle measured about 12 us slower on the
    // 256-request, 151936-column workload
    prof_begin(kPVerifySample, s);
    e = launch_kernel(verify_sample<PT, UT, WT>, dim3(a.R), dim3(256), 0, s, false, a);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_verify(VerifyArgs& a, cudaStream_t s) {
    const int key = a.p_dtype * 4 + a.u_dtype * 2 + a.w_dtype;
    switch (key) {
        case 0: return launch_typed<DSPARK_F32, DSPARK_F32, DSPARK_F32>(a, s);
        case 1: return launch_typed<DSPARK_F32, DSPARK_F32, DSPARK_BF16>(a, s);
        case 2: return launch_typed<DSPARK_F32, DSPARK_BF16, DSPARK_F32>(a, s);
        case 3: return launch_typed<DSPARK_F32, DSPARK_BF16, DSPARK_BF16>(a, s);
        case 4: return launch_typed<DSPARK_BF16, DSPARK_F32, DSPARK_F32>(a, s);
        case 5: return launch_typed<DSPARK_BF16, DSPARK_F32, DSPARK_BF16>(a, s);
        case 6: return launch_typed<DSPARK_BF16, DSPARK_BF16, DSPARK_F32>(a, s);
        default: return launch_typed<DSPARK_BF16, DSPARK_BF16, DSPARK_BF16>(a, s);
    }
}

}  // namespace dspark
