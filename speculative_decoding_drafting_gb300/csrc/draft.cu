// draft.cu -- the sequential stage of the semi-autoregressive drafter.
//
// "DSpark: DeepSeek 线上跑的投机解码" blog, section 3.2: for k = 1..gamma a
// light head adds B_k to the parallel backbone's base logits U_k and x_k is
// sampled from softmax(U_k + B_k); the Markov head has B_k = W1[x_{k-1}] W2,
// the RNN head B_k = tanh(out_k) W2 after a GRU-like state update.  DSpark
// explainer, section 03: q_k = softmax(U_k + B_k), B_k = W1[x_{k-1}] W2.
//
// Launch structure per call (one stream):
//   for k = 1..gamma:
//     prep(k)   one CTA per request: reduce the V-slices of step k-1 to
//               x_{k-1} (writes tokens/q_tok/lse of step k-1), then build the
//               rank-r code e_k (Markov gather or RNN step) into `code`
//     sweep(k)  the V sweep: B_k = e_k W2, z = (U_k + B_k) / T, online
//               log-sum-exp and Gumbel race per V-slice -> partials
//   prep(gamma + 1) reduces the last step.
// The tensor-core sweep (draft_tc.cu) replaces the generic sweep when the
// weights are bf16 and r is a multiple of 64.
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"
#include "row_acc.cuh"

namespace dspark {

bool draft_tc_supported(const DraftArgs& a);
int draft_tc_slices(const DraftArgs& a);
cudaError_t launch_draft_tc_sweep(DraftArgs& a, int k, cudaStream_t s);

constexpr int kPrepThreads = 512;   // threads of a prep CTA (one request)

// Leading dimension of the GRU input rows in the workspace: 2r + d rounded
// up to a multiple of 4 floats (16-byte rows; the padding holds zeros).
__host__ __device__ __forceinline__ int gru_ldz(int r, int d) { return (2 * r + d + 3) & ~3; }

// ------------------------------------------------------------------ reduce
// Block-wide reduction of n partials into thread 0's RowAcc.
__device__ RowAcc reduce_partials(const DraftPartial* p, int n) {
    __shared__ RowAcc sh[32];
    RowAcc a;
    acc_init(a);
    for (int i = threadIdx.x; i < n; i += blockDim.x) acc_merge(a, partial_to_acc(p[i]));
    acc_warp_reduce(a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh[warp] = a;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        RowAcc b;
        acc_init(b);
        if (lane < nw) b = sh[lane];
        acc_warp_reduce(b);
        a = b;
    }
    __syncthreads();
    return a;
}

// Greedy step (T = 0): x_{k-1} = argmax over the V-slice partials.
__device__ int finish_greedy(const DraftArgs& A, int r, int kprev, const DraftPartial* parts) {
    __shared__ int s_x;
    RowAcc a = reduce_partials(parts, A.n_slices);
    if (threadIdx.x == 0) {
        int x = a.ib;
        const size_t o = (size_t)r * A.gamma + (kprev - 1);
        if (x < 0 || x >= A.V) {     // cannot happen for finite logits; stay in bounds
            raise_status(A.ws, kStatBadToken);
            x = 0;
        }
        A.tokens[o] = x;
        A.q_tok[o] = 1.f;
        A.lse[o] = 0.0;
        s_x = x;
    }
    __syncthreads();
    return s_x;
}

// Warp-wide merge of (online log-sum-exp pair M, S with S = sum 2^(lm - M);
// race winner key, index); every lane ends with the warp's result.
__device__ __forceinline__ void merge_lse_race(float& M, float& S, float& key, int& idx) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
        const float k2 = __shfl_xor_sync(0xffffffffu, key, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
        if (m2 != -INFINITY) {
            if (M == -INFINITY) {
                M = m2;
                S = s2;
            } else if (m2 > M) {
                S = fmaf(S, ex2_approx(M - m2), s2);
                M = m2;
            } else {
                S = fmaf(s2, ex2_approx(m2 - M), S);
            }
        }
        if (key_better(k2, i2, key, idx)) {
            key = k2;
            idx = i2;
        }
    }
}

// Block-wide argmax of (key, index), ties to the lower index, with a payload
// that travels with the winner; thread 0 ends with the result.
__device__ void block_argmax_with(float& key, int& idx, float& pay) {
    __shared__ float sk[32], sp[32];
    __shared__ int si[32];
    auto warp_step = [&]() {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float k2 = __shfl_xor_sync(0xffffffffu, key, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
            const float p2 = __shfl_xor_sync(0xffffffffu, pay, o);
            if (key_better(k2, i2, key, idx)) {
                key = k2;
                idx = i2;
                pay = p2;
            }
        }
    };
    warp_step();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if (lane == 0) {
        sk[warp] = key;
        si[warp] = idx;
        sp[warp] = pay;
    }
    __syncthreads();
    if (warp == 0) {
        key = lane < nw ? sk[lane] : -INFINITY;
        idx = lane < nw ? si[lane] : INT_MAX;
        pay = lane < nw ? sp[lane] : 0.f;
        warp_step();
    }
}

// Sampling step (T > 0): Gumbel-max in two levels, an exact sampler of
// q = softmax(z).  Level 1 picks a 256-column chunk c with key
// log2(chunk mass) - log2(E_c) (E = -ln u, stream 3, index c); level 2 picks
// the column inside it with key y_v - log2(E_v) (stream 0, index v), the
// chunk's logits rebuilt here from e_k, W2 and U_k.  The chunk masses come
// from the V sweep as (reference, sum of 2^(y - reference)) per quarter.
template <int UT, int WT>
__device__ int finish_sample(const DraftArgs& A, int r, int kprev) {
    constexpr int NW = kPrepThreads / 32;
    __shared__ float e_sh[1024];
    __shared__ float s_M[NW], s_S[NW], s_k[NW];
    __shared__ int s_ci[NW];
    __shared__ int s_c, s_x;
    __shared__ float s_lseM, s_lseL;
    __shared__ int s_lseE;
    const int V = A.V, NC = A.nchunk;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t req = A.req_ids ? A.req_ids[r] : (uint32_t)r;
    const PhiloxKey key = philox_key(A.seed);
    // the code e of step k-1: loads issued now, stored to shared memory after level 1
    const float* crow = A.code + ((size_t)r * A.gamma + (kprev - 1)) * A.r;
    float ev[1024 / kPrepThreads];
#pragma unroll
    for (int t = 0; t < 1024 / kPrepThreads; ++t) {
        const int i = threadIdx.x + t * kPrepThreads;
        ev[t] = i < A.r ? crow[i] : 0.f;
    }
    // level 1: chunk log-masses (bits), their log-sum-exp and the chunk race
    float M = -INFINITY, S = 0.f;          // online: S = sum 2^(lm - M)
    float kbest = -INFINITY;
    int cbest = INT_MAX;
    const float4* cm = reinterpret_cast<const float4*>(A.cmass + (size_t)r * NC * 4);
    for (int cb = threadIdx.x; cb < NC; cb += 2 * kPrepThreads) {
        // up to two chunks per pass, their (reference, sum) quads loaded first
        float4 e8[2][2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int c = cb + t * kPrepThreads;
            e8[t][0] = c < NC ? cm[(size_t)c * 2] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
            e8[t][1] = c < NC ? cm[(size_t)c * 2 + 1] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int c = cb + t * kPrepThreads;
            const float2 e4[4] = {make_float2(e8[t][0].x, e8[t][0].y), make_float2(e8[t][0].z, e8[t][0].w),
                                  make_float2(e8[t][1].x, e8[t][1].y), make_float2(e8[t][1].z, e8[t][1].w)};
            float mq = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (e4[q].y > 0.f) mq = fmaxf(mq, e4[q].x);
            if (c >= NC || mq == -INFINITY) continue;
            float sq = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (e4[q].y > 0.f) sq += e4[q].y * ex2_approx(e4[q].x - mq);
            const float lm = mq + log2f(sq);                 // log2 of the chunk mass
            if (lm > M) {
                S = S * ex2_approx(M - lm) + 1.f;
                M = lm;
            } else {
                S += ex2_approx(lm - M);
            }
            const uint4 w = philox4x32_10(make_uint4((uint32_t)c >> 2, req, (uint32_t)kprev, 3u), key);
            const float kc = race_key2(lm, pick_word(w, (uint32_t)c & 3u));
            if (key_better(kc, c, kbest, cbest)) {
                kbest = kc;
                cbest = c;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 1024 / kPrepThreads; ++t) {
        const int i = threadIdx.x + t * kPrepThreads;
        if (i < A.r) e_sh[i] = ev[t];
    }
    // one block reduction for the chunks' log-sum-exp (online pair M, S) and
    // the chunk race; the log-sum-exp stays as M + e + log2(mant) with
    // S = mant 2^e, so that nothing is rounded at the magnitude of M
    {
        merge_lse_race(M, S, kbest, cbest);
        if (lane == 0) {
            s_M[warp] = M;
            s_S[warp] = S;
            s_k[warp] = kbest;
            s_ci[warp] = cbest;
        }
        __syncthreads();
        if (warp == 0) {
            M = lane < NW ? s_M[lane] : -INFINITY;
            S = lane < NW ? s_S[lane] : 0.f;
            kbest = lane < NW ? s_k[lane] : -INFINITY;
            cbest = lane < NW ? s_ci[lane] : INT_MAX;
            merge_lse_race(M, S, kbest, cbest);
            if (lane == 0) {
                int e = 0;
                const float mant = frexpf(S, &e);           // S = mant 2^e, mant in [1/2, 1)
                s_lseM = M;
                s_lseE = e;
                s_lseL = log2f(mant);
                s_c = (cbest >= 0 && cbest < NC) ? cbest : 0;
            }
        }
        __syncthreads();
    }
    const int c = s_c;
    // level 2: rebuild the chosen chunk's logits, B = e W2 on its 256 columns.
    // Thread j < 256 owns column c 256 + j; its U value is fetched first so
    // that its latency hides behind the W2 rows.  Warp w takes rank rows
    // w, w + NW, ..., lane l columns 8l .. 8l + 7, a batch of rows' loads in
    // flight at once; the warps' sums are added in a fixed order.
    const int j = threadIdx.x;
    const int v = c * kRChunk + j;
    const bool own = j < kRChunk && v < V;
    float u = 0.f;
    if (own) u = Elem<UT>::get(static_cast<const typename Elem<UT>::T*>(A.U), ((size_t)r * A.gamma + (kprev - 1)) * V + v);
    __shared__ __align__(16) float s_b[NW][kRChunk];
    {
        constexpr int kBatch = WT == DSPARK_BF16 ? 16 : 8;
        const int c0 = c * kRChunk + 8 * lane;
        float b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int i0 = warp; i0 < A.r; i0 += kBatch * NW) {
            Row8<WT> w[kBatch];
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
                const int i = i0 + NW * t;
                w[t].load(A.W2, (size_t)i * V + c0, i < A.r ? V - c0 : 0);
            }
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
                const int i = i0 + NW * t;
                const float ei = i < A.r ? e_sh[i] : 0.f;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) b[jj] = fmaf(ei, w[t].get(jj), b[jj]);
            }
        }
        {
            // two 16-byte stores per lane: eight scalar stores at a stride of
            // eight floats would put eight lanes on each of four banks
            float4* dst = reinterpret_cast<float4*>(&s_b[warp][8 * lane]);
            dst[0] = make_float4(b[0], b[1], b[2], b[3]);
            dst[1] = make_float4(b[4], b[5], b[6], b[7]);
        }
    }
    __syncthreads();
    const float invT = 1.f / A.T;
    float kx = -INFINITY;
    int ix = INT_MAX;
    float yx = 0.f;
    if (own) {
        float bs = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < NW; ++w8) bs += s_b[w8][j];
        const float y = (u + bs) * invT * kLog2e;
        const uint4 wd = philox4x32_10(make_uint4((uint32_t)v >> 2, req, (uint32_t)kprev, 0u), key);
        kx = race_key2(y, pick_word(wd, (uint32_t)v & 3u));
        ix = v;
        yx = y;
    }
    // the winner, its logit travelling with it
    block_argmax_with(kx, ix, yx);
    if (threadIdx.x == 0) {
        int x = ix;
        const size_t o = (size_t)r * A.gamma + (kprev - 1);
        if (x < 0 || x >= V) {
            raise_status(A.ws, kStatBadToken);
            x = 0;
        }
        s_x = x;
        A.tokens[o] = x;
        // q(x) = 2^(y_x - lse2), lse2 = M + e + l: the exponent formed in
        // double, then 2^hi (1 + lo ln 2) with hi + lo = the exponent
        const double lse2 = ((double)s_lseM + (double)s_lseE) + (double)s_lseL;
        const double d = (double)yx - lse2;
        const float dh = (float)d;
        A.q_tok[o] = exp2f(dh) * (1.f + (float)(d - (double)dh) * kLn2);
        A.lse[o] = 0.69314718055994531 * lse2;
    }
    __syncthreads();
    return s_x;
}

template <int UT, int WT>
__device__ int finish_step(const DraftArgs& A, int r, int kprev) {
    if (A.T > 0.f) return finish_sample<UT, WT>(A, r, kprev);
    const DraftPartial* p = A.parts + (size_t)(kprev & 1) * A.parts_stride + (size_t)r * A.n_slices;
    return finish_greedy(A, r, kprev, p);
}

__device__ __forceinline__ int read_anchor(const DraftArgs& A, int r) {
    __shared__ int s_x;
    if (threadIdx.x == 0) {
        int x = A.anchor[r];
        if (x < 0 || x >= A.V) {
            raise_status(A.ws, kStatBadToken);
            x = 0;
        }
        s_x = x;
    }
    __syncthreads();
    return s_x;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits_rn(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Write e (float) for request r at step k into code and its three-way bf16
// split e = hi + mid + lo (each term rounds the remainder of the previous
// ones; 3 x 8 significand bits cover a float's 24, so the sum is e exactly
// for the codes drafting produces).
__device__ __forceinline__ void store_code(const DraftArgs& A, int r, int k, int i, float e) {
    A.code[((size_t)r * A.gamma + (k - 1)) * A.r + i] = e;
    const uint16_t hi = f32_to_bf16_bits_rn(e);
    const float rest = e - bf16_bits_to_float(hi);
    const uint16_t mid = f32_to_bf16_bits_rn(rest);
    const float rest2 = rest - bf16_bits_to_float(mid);
    const size_t plane = (size_t)A.R * A.r;
    A.ebf[(size_t)r * A.r + i] = hi;
    A.ebf[plane + (size_t)r * A.r + i] = mid;
    A.ebf[2 * plane + (size_t)r * A.r + i] = f32_to_bf16_bits_rn(rest2);
}

// Confidence head (blog section 4.1, ConfidenceHead) for request r at step k:
// c_k = sigmoid(wc . [h_k, W1[x_{k-1}]] / t_k), no bias, t_k = 1 unless
// per-position temperatures (blog section 4.2) are given.  The block's threads take
// strided shares of the d + r products (f32 FMAs; the h_k terms first, from
// confidence_h_part), then the warps and the block add them in a fixed order.
__device__ __forceinline__ float confidence_h_part(const DraftArgs& A, int r, int k) {
    const int d = A.dc;
    const unsigned short* h = static_cast<const unsigned short*>(A.Hc) + ((size_t)r * A.gamma + (k - 1)) * d;
    float t = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) t = fmaf(A.wc[i], bf16_bits_to_float(h[i]), t);
    return t;
}

__device__ void confidence_head(const DraftArgs& A, int r, int k, int x, float t) {
    __shared__ float s_part[kPrepThreads / 32];
    const int d = A.dc, rr = A.r;
    for (int i = threadIdx.x; i < rr; i += blockDim.x)
        t = fmaf(A.wc[d + i], ld_elem(A.W1, A.w_dtype, (size_t)x * rr + i), t);
    t = warp_sum(t);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        float u = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) u += s_part[w];
        if (A.tc) u *= (float)(1.0 / A.tc[k - 1]);   // sequential temperature scaling of position k
        A.conf[(size_t)r * A.gamma + (k - 1)] = 1.f / (1.f + expf(-u));
    }
}

// prep(k) for the Markov head: x_{k-1} then e_k = W1[x_{k-1}] (and c_k).
template <int UT, int WT>
__global__ void __launch_bounds__(kPrepThreads) draft_prep_markov(DraftArgs A, int k) {
    pdl_launch_dependents();
    // the head's h_k half reads only the caller's inputs, so it runs before
    // the wait, under the previous kernel's tail
    const float th = (A.conf && k <= A.gamma) ? confidence_h_part(A, blockIdx.x, k) : 0.f;
    pdl_wait();
    const int r = blockIdx.x;
    int x;
    if (k == 1) {
        x = read_anchor(A, r);
    } else {
        x = finish_step<UT, WT>(A, r, k - 1);
    }
    if (k > A.gamma) return;
    if (threadIdx.x == 0) A.best[r] = kOrderNegInf;
    for (int i = threadIdx.x; i < A.r; i += blockDim.x)
        store_code(A, r, k, i, ld_elem(A.W1, A.w_dtype, (size_t)x * A.r + i));
    if (A.conf) confidence_head(A, r, k, x, th);
}

// prep(k) for the RNN head (blog section 3.2 RNNHead.step), first half:
// x_{k-1}, then the GRU input z = [s_{k-1}, W1[x_{k-1}], h_k] of the request
// goes to the workspace (and c_k); rnn_gru (below) forms G = z Wgco for all
// requests.
template <int UT, int WT>
__global__ void __launch_bounds__(kPrepThreads) draft_prep_rnn(DraftArgs A, int k) {
    pdl_launch_dependents();
    const float th = (A.conf && k <= A.gamma) ? confidence_h_part(A, blockIdx.x, k) : 0.f;
    pdl_wait();
    const int r = blockIdx.x;
    int x;
    if (k == 1) {
        x = read_anchor(A, r);
    } else {
        x = finish_step<UT, WT>(A, r, k - 1);
    }
    const int rr = A.r;
    float* srow = A.rnn_state + (size_t)r * rr;
    if (k > A.gamma) {
        if (A.state_out)
            for (int i = threadIdx.x; i < rr; i += blockDim.x) A.state_out[(size_t)r * rr + i] = srow[i];
        return;
    }
    if (threadIdx.x == 0) A.best[r] = kOrderNegInf;
    const unsigned short* Hb = static_cast<const unsigned short*>(A.H) + ((size_t)r * A.gamma + (k - 1)) * A.d;
    if (A.gru_tc) {
        // bf16 row [s_hi | s_mid | s_lo | W1[x] | h | 0] for the tensor-core GRU
        // (the three terms of s add up to s exactly; W1 and h are bf16 already)
        const int ldzb = gru_ldzb(rr, A.d);
        uint16_t* zr = A.zb + (size_t)r * ldzb;
        const uint16_t* w1 = static_cast<const uint16_t*>(A.W1) + (size_t)x * rr;
        for (int i = threadIdx.x; i < rr; i += blockDim.x) {
            const float sv = (k == 1) ? 0.f : srow[i];
            const uint16_t hi = f32_to_bf16_bits_rn(sv);
            const float rest = sv - bf16_bits_to_float(hi);
            const uint16_t mid = f32_to_bf16_bits_rn(rest);
            zr[i] = hi;
            zr[rr + i] = mid;
            zr[2 * rr + i] = f32_to_bf16_bits_rn(rest - bf16_bits_to_float(mid));
            zr[3 * rr + i] = w1[i];
        }
        for (int i = threadIdx.x; i < A.d; i += blockDim.x) zr[4 * rr + i] = Hb[i];
        for (int i = 4 * rr + A.d + threadIdx.x; i < ldzb; i += blockDim.x) zr[i] = 0;
    } else {
        const int Kin = 2 * rr + A.d, ldz = gru_ldz(rr, A.d);
        float* z = A.zbuf + (size_t)r * ldz;
        for (int i = threadIdx.x; i < rr; i += blockDim.x) {
            z[i] = (k == 1) ? 0.f : srow[i];
            z[rr + i] = ld_elem(A.W1, A.w_dtype, (size_t)x * rr + i);
        }
        for (int i = threadIdx.x; i < A.d; i += blockDim.x) z[2 * rr + i] = bf16_bits_to_float(Hb[i]);
        for (int i = Kin + threadIdx.x; i < ldz; i += blockDim.x) z[i] = 0.f;
    }
    if (A.conf) confidence_head(A, r, k, x, th);
}

// The GRU step for all requests (blog section 3.2 RNNHead.step):
//   G = z Wgco = (gate | cand | out);
//   s_k = sigmoid(gate) s_{k-1} + (1 - sigmoid(gate)) tanh(cand);  e_k = tanh(out).
// One CTA = 16 requests x 32 state columns j, with the gate, candidate and
// output columns of those j (96 columns of Wgco), so the update has all three
// at hand.  Thread (m, n): request m of the tile, columns n, n + 1.  K runs in
// tiles of 64 with the next tile's loads in flight during the current one;
// the sum over z still runs in index order (f32 FMAs).  VEC: bf16 Wgco with
// r % 8 == 0, loaded 8 values at a time; otherwise element by element.
constexpr int kGruTM = 16, kGruTN = 32, kGruTK = 64;
template <int WT, bool VEC>
__global__ void __launch_bounds__(256) rnn_gru(DraftArgs A, int k) {
    __shared__ __align__(16) float zs[kGruTK][kGruTM];
    __shared__ __align__(16) float ws[kGruTK][3 * kGruTN];
    pdl_launch_dependents();
    pdl_wait();
    const int rr = A.r, Kin = 2 * rr + A.d, ldz = gru_ldz(rr, A.d);
    const int j0 = blockIdx.x * kGruTN, m0 = blockIdx.y * kGruTM;
    const int t = threadIdx.x;
    const int m = t >> 4, n = (t & 15) * 2;
    // this thread's loads of a K tile: z as one float4 (row t / 16, columns
    // 4 (t % 16) ..), Wgco as three 8-value pieces (see below)
    float4 zr[1];
    uint4 wr[3];
    float wsc[24];
    auto load = [&](int k0) {
#pragma unroll
        for (int i = 0; i < 1; ++i) {
            const int f = t + 256 * i, mm = f >> 4, c4 = f & 15, row = m0 + mm;
            zr[i] = (row < A.R && k0 + 4 * c4 < ldz)
                        ? *reinterpret_cast<const float4*>(A.zbuf + (size_t)row * ldz + k0 + 4 * c4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (VEC) {
            // piece p = t + 256 i (i < 3): tile row p / 12, gate (p % 12) / 4, columns 8 (p % 4) ..
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int pc = t + 256 * i, kk = pc / 12, g = (pc % 12) >> 2, c8 = pc & 3;
                const int col = j0 + 8 * c8;
                wr[i] = (k0 + kk < Kin && col < rr)
                            ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(A.Wgco) +
                                                                   (size_t)(k0 + kk) * 3 * rr + (size_t)g * rr + col))
                            : make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 24; ++i) {
                const int e = t + 256 * i, kk = e / 96, c = e % 96, g = c / kGruTN, jj = c % kGruTN;
                wsc[i] = (k0 + kk < Kin && j0 + jj < rr)
                             ? ld_elem(A.Wgco, WT, (size_t)(k0 + kk) * 3 * rr + (size_t)g * rr + j0 + jj)
                             : 0.f;
            }
        }
    };
    auto store = [&]() {
#pragma unroll
        for (int i = 0; i < 1; ++i) {
            const int f = t + 256 * i, mm = f >> 4, c4 = f & 15;
            zs[4 * c4 + 0][mm] = zr[i].x;
            zs[4 * c4 + 1][mm] = zr[i].y;
            zs[4 * c4 + 2][mm] = zr[i].z;
            zs[4 * c4 + 3][mm] = zr[i].w;
        }
        if (VEC) {
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int pc = t + 256 * i, kk = pc / 12, g = (pc % 12) >> 2, c8 = pc & 3;
                const uint32_t w4[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
                float* dst = &ws[kk][g * kGruTN + 8 * c8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dst[2 * e] = bf16_bits_to_float(w4[e] & 0xFFFFu);
                    dst[2 * e + 1] = bf16_bits_to_float(w4[e] >> 16);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 24; ++i) {
                const int e = t + 256 * i;
                ws[e / 96][e % 96] = wsc[i];
            }
        }
    };
    float acc[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    load(0);
    for (int k0 = 0; k0 < Kin; k0 += kGruTK) {
        __syncthreads();                  // the previous tile has been read
        store();
        __syncthreads();
        if (k0 + kGruTK < Kin) load(k0 + kGruTK);
#pragma unroll 8
        for (int kk = 0; kk < kGruTK; ++kk) {
            const float zv = zs[kk][m];
#pragma unroll
            for (int g = 0; g < 3; ++g) {
                acc[g][0] = fmaf(zv, ws[kk][g * kGruTN + n], acc[g][0]);
                acc[g][1] = fmaf(zv, ws[kk][g * kGruTN + n + 1], acc[g][1]);
            }
        }
    }
    const int row = m0 + m;
    if (row >= A.R) return;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int j = j0 + n + q;
        if (j >= rr) continue;
        const float sg = 1.f / (1.f + expf(-acc[0][q]));
        const float sprev = A.zbuf[(size_t)row * ldz + j];      // s_{k-1}, the first block of z
        A.rnn_state[(size_t)row * rr + j] = sg * sprev + (1.f - sg) * tanhf(acc[1][q]);
        store_code(A, row, k, j, tanhf(acc[2][q]));
    }
}

// The end of the tensor-core GRU step (gru_tc.cu computes G in K parts):
// one thread per (request, j) adds the parts in order and applies the update
//   s_k = sigmoid(gate) s_{k-1} + (1 - sigmoid(gate)) tanh(cand),  e_k = tanh(out).
__global__ void __launch_bounds__(256) gru_finish(DraftArgs A, int k) {
    pdl_launch_dependents();
    pdl_wait();
    const int rr = A.r;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)A.R * rr) return;
    const int row = (int)(idx / rr), j = (int)(idx % rr);
    float gate = 0.f, cand = 0.f, out = 0.f;
    for (int s = 0; s < A.gru_parts; ++s) {
        const float* gp = A.gpart + ((size_t)s * A.R + row) * 3 * rr;
        gate += gp[j];
        cand += gp[rr + j];
        out += gp[2 * rr + j];
    }
    const float sg = 1.f / (1.f + expf(-gate));
    float* srow = A.rnn_state + (size_t)row * rr;
    const float sprev = k == 1 ? 0.f : srow[j];
    srow[j] = sg * sprev + (1.f - sg) * tanhf(cand);
    store_code(A, row, k, j, tanhf(out));
}

// ------------------------------------------------------------------ generic sweep
// One CTA per (V-slice of 4096, request); thread t owns columns
// v0 + 4t + 1024 g, g = 0..3.  B = e W2 on CUDA cores.
template <int UT, int WT, bool GREEDY>
__global__ void __launch_bounds__(256) draft_sweep_generic(DraftArgs A, int k) {
    extern __shared__ float e_sh[];
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.y;
    const int slice = blockIdx.x;
    const int V = A.V;
    for (int i = threadIdx.x; i < A.r; i += blockDim.x)
        e_sh[i] = A.code[((size_t)r * A.gamma + (k - 1)) * A.r + i];
    __syncthreads();
    constexpr int G = 4;
    float acc[G][4];
    int col[G];
    bool ok[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        col[g] = slice * kGenericSlice + 4 * threadIdx.x + 1024 * g;
        ok[g] = col[g] < V;
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[g][q] = 0.f;
    }
    for (int i = 0; i < A.r; ++i) {
        const float ei = e_sh[i];
#pragma unroll
        for (int g = 0; g < G; ++g)
            if (ok[g]) {
                const float4 w = load4<WT>(A.W2, (size_t)i * V + col[g]);
                acc[g][0] = fmaf(ei, w.x, acc[g][0]);
                acc[g][1] = fmaf(ei, w.y, acc[g][1]);
                acc[g][2] = fmaf(ei, w.z, acc[g][2]);
                acc[g][3] = fmaf(ei, w.w, acc[g][3]);
            }
    }
    const float c2 = GREEDY ? 1.f : kLog2e / A.T;     // tempered logits in bits
    const size_t urow = ((size_t)r * A.gamma + (k - 1)) * (size_t)V;
    float y[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float4 u = ok[g] ? load4<UT>(A.U, urow + col[g]) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) y[g][q] = ok[g] ? (uu[q] + acc[g][q]) * c2 : -INFINITY;
    }
    __shared__ RowAcc sh[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (GREEDY) {
        RowAcc a;
        acc_init(a);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            int c4[4];
            bool v4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                c4[q] = col[g] + q;
                v4[q] = ok[g];
            }
            acc_update_greedy<4>(a, y[g], c4, v4);
        }
        acc_warp_reduce(a);
        if (lane == 0) sh[warp] = a;
        __syncthreads();
        if (warp == 0) {
            RowAcc b;
            acc_init(b);
            if (lane < 8) b = sh[lane];
            acc_warp_reduce(b);
            if (lane == 0)
                A.parts[(size_t)(k & 1) * A.parts_stride + (size_t)r * A.n_slices + slice] = acc_to_partial(b);
        }
        return;
    }
    // sampling: mass of each 256-column chunk of the slice against the slice max.
    // Thread t's group g lies in chunk 4 g + t / 64 of the slice, which the 64
    // threads of warps 2 (t / 64) and 2 (t / 64) + 1 cover together.
    float mloc = -INFINITY;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int q = 0; q < 4; ++q) mloc = fmaxf(mloc, y[g][q]);
    __shared__ float s_m[8];
    __shared__ float s_sum[G][8];
    mloc = warp_max(mloc);
    if (lane == 0) s_m[warp] = mloc;
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) M = fmaxf(M, s_m[i]);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float sg = 0.f;
        if (M != -INFINITY)
#pragma unroll
            for (int q = 0; q < 4; ++q) sg += ex2_approx(y[g][q] - M);
        sg = warp_sum(sg);
        if (lane == 0) s_sum[g][warp] = sg;
    }
    __syncthreads();
    if (threadIdx.x < 16) {
        const int g = threadIdx.x >> 2, h = threadIdx.x & 3;     // chunk 4 g + h of the slice
        const int chunk = slice * (kGenericSlice / kRChunk) + 4 * g + h;
        if (chunk < A.nchunk) {
            const float sc = s_sum[g][2 * h] + s_sum[g][2 * h + 1];
            float2* e = A.cmass + ((size_t)r * A.nchunk + chunk) * 4;
            e[0] = make_float2(M, sc);
            e[1] = make_float2(-INFINITY, 0.f);
            e[2] = make_float2(-INFINITY, 0.f);
            e[3] = make_float2(-INFINITY, 0.f);
        }
    }
}

// ------------------------------------------------------------------ host
size_t draft_workspace_bytes(int R, int gamma, int V, int r, int d) {
    (void)gamma;
    const int ns = (V + kGenericSlice - 1) / kGenericSlice;
    const int ns_max = ns > 1024 ? ns : 1024;
    size_t off = sizeof(WsHeader);
    off = align_up(off + 2ull * R * ns_max * sizeof(DraftPartial), 256);
    off = align_up(off + (size_t)R * gru_ldz(r, d) * sizeof(float), 256);   // GRU input z (RNN head)
    if (d > 0) {
        off = align_up(off + (size_t)R * gru_ldzb(r, d) * sizeof(uint16_t), 256);               // bf16 z
        off = align_up(off + (size_t)gru_tc_parts(R, r, d) * R * 3 * r * sizeof(float), 256);  // partial G
    }
    off = align_up(off + 3ull * R * r * sizeof(uint16_t), 256);
    off = align_up(off + (size_t)R * r * sizeof(float), 256);
    off = align_up(off + (size_t)R * sizeof(uint32_t), 256);
    off = align_up(off + (size_t)R * ((V + kRChunk - 1) / kRChunk) * 4 * sizeof(float2), 256);
    return off;
}

int draft_carve(DraftArgs& a, size_t ws_bytes) {
    const size_t need = draft_workspace_bytes(a.R, a.gamma, a.V, a.r, a.d);
    if (ws_bytes < need) return DSPARK_ERR_WORKSPACE;
    const int ns = (a.V + kGenericSlice - 1) / kGenericSlice;
    const int ns_max = ns > 1024 ? ns : 1024;
    char* base = static_cast<char*>(a.ws);
    size_t off = sizeof(WsHeader);
    a.parts = reinterpret_cast<DraftPartial*>(base + off);
    a.parts_stride = a.R * ns_max;
    off = align_up(off + 2ull * a.R * ns_max * sizeof(DraftPartial), 256);
    a.zbuf = reinterpret_cast<float*>(base + off);
    off = align_up(off + (size_t)a.R * gru_ldz(a.r, a.d) * sizeof(float), 256);
    a.zb = nullptr;
    a.gpart = nullptr;
    a.gru_parts = 0;
    if (a.d > 0) {
        a.zb = reinterpret_cast<uint16_t*>(base + off);
        off = align_up(off + (size_t)a.R * gru_ldzb(a.r, a.d) * sizeof(uint16_t), 256);
        a.gpart = reinterpret_cast<float*>(base + off);
        a.gru_parts = gru_tc_parts(a.R, a.r, a.d);
        off = align_up(off + (size_t)a.gru_parts * a.R * 3 * a.r * sizeof(float), 256);
    }
    a.ebf = reinterpret_cast<uint16_t*>(base + off);
    off = align_up(off + 3ull * a.R * a.r * sizeof(uint16_t), 256);
    a.rnn_state = reinterpret_cast<float*>(base + off);
    off = align_up(off + (size_t)a.R * a.r * sizeof(float), 256);
    a.best = reinterpret_cast<uint32_t*>(base + off);
    off = align_up(off + (size_t)a.R * sizeof(uint32_t), 256);
    a.cmass = reinterpret_cast<float2*>(base + off);
    a.nchunk = (a.V + kRChunk - 1) / kRChunk;
    return DSPARK_OK;
}

template <int UT, int WT, bool GREEDY>
static cudaError_t sweep_generic(DraftArgs& a, int k, cudaStream_t s) {
    dim3 grid((a.V + kGenericSlice - 1) / kGenericSlice, a.R);
    prof_begin(kPDraftSweepGeneric, s);
    cudaError_t e = launch_kernel(draft_sweep_generic<UT, WT, GREEDY>, grid, dim3(256), a.r * sizeof(float), s, true,
                                  a, k);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

static cudaError_t launch_sweep(DraftArgs& a, int k, bool use_tc, cudaStream_t s) {
    if (use_tc) return launch_draft_tc_sweep(a, k, s);
    const bool greedy = !(a.T > 0.f);
    const int key = a.u_dtype * 4 + a.w_dtype * 2 + (greedy ? 1 : 0);
    switch (key) {
        case 0: return sweep_generic<DSPARK_F32, DSPARK_F32, false>(a, k, s);
        case 1: return sweep_generic<DSPARK_F32, DSPARK_F32, true>(a, k, s);
        case 2: return sweep_generic<DSPARK_F32, DSPARK_BF16, false>(a, k, s);
        case 3: return sweep_generic<DSPARK_F32, DSPARK_BF16, true>(a, k, s);
        case 4: return sweep_generic<DSPARK_BF16, DSPARK_F32, false>(a, k, s);
        case 5: return sweep_generic<DSPARK_BF16, DSPARK_F32, true>(a, k, s);
        case 6: return sweep_generic<DSPARK_BF16, DSPARK_BF16, false>(a, k, s);
        default: return sweep_generic<DSPARK_BF16, DSPARK_BF16, true>(a, k, s);
    }
}

cudaError_t launch_draft(DraftArgs& a, bool rnn, cudaStream_t s) {
    a.rnn = rnn ? 1 : 0;
    a.gru_tc = (rnn && gru_tc_supported(a)) ? 1 : 0;
    const bool use_tc = draft_tc_supported(a);
    a.n_slices = use_tc ? draft_tc_slices(a) : (a.V + kGenericSlice - 1) / kGenericSlice;
    void (*prep_m)(DraftArgs, int);
    void (*prep_r)(DraftArgs, int);
    switch (a.u_dtype * 2 + a.w_dtype) {
        case 0: prep_m = draft_prep_markov<DSPARK_F32, DSPARK_F32>; prep_r = draft_prep_rnn<DSPARK_F32, DSPARK_F32>; break;
        case 1: prep_m = draft_prep_markov<DSPARK_F32, DSPARK_BF16>; prep_r = draft_prep_rnn<DSPARK_F32, DSPARK_BF16>; break;
        case 2: prep_m = draft_prep_markov<DSPARK_BF16, DSPARK_F32>; prep_r = draft_prep_rnn<DSPARK_BF16, DSPARK_F32>; break;
        default: prep_m = draft_prep_markov<DSPARK_BF16, DSPARK_BF16>; prep_r = draft_prep_rnn<DSPARK_BF16, DSPARK_BF16>; break;
    }
    void (*gru)(DraftArgs, int) = a.w_dtype == DSPARK_F32 ? rnn_gru<DSPARK_F32, false>
                                  : (a.r % 8 == 0 ? rnn_gru<DSPARK_BF16, true> : rnn_gru<DSPARK_BF16, false>);
    const dim3 gru_grid((a.r + kGruTN - 1) / kGruTN, (a.R + kGruTM - 1) / kGruTM);
    for (int k = 1; k <= a.gamma + 1; ++k) {
        // prep(1) waits for the caller's work; every later launch overlaps
        // the previous kernel's tail
        cudaError_t e;
        if (rnn) {
            prof_begin(kPDraftPrepRnn, s);
            e = launch_kernel(prep_r, dim3(a.R), dim3(kPrepThreads), 0, s, k > 1, a, k);
            prof_end(s);
            if (e == cudaSuccess && k <= a.gamma) {
                if (a.gru_tc) {
                    e = launch_gru_tc(a, k, s);
                    if (e == cudaSuccess) {
                        const size_t n = (size_t)a.R * a.r;
                        prof_begin(kPDraftRnnGruFinish, s);
                        e = launch_kernel(gru_finish, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, true, a, k);
                    }
                } else {
                    prof_begin(kPDraftRnnGru, s);
                    e = launch_kernel(gru, gru_grid, dim3(256), 0, s, true, a, k);
                }
            }
        } else {
            prof_begin(kPDraftPrep, s);
            e = launch_kernel(prep_m, dim3(a.R), dim3(kPrepThreads), 0, s, k > 1, a, k);
        }
        prof_end(s);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (k > a.gamma) break;
        e = launch_sweep(a, k, use_tc, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dspark
