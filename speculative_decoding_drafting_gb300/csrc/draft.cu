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

// Finish step k-1 for request r from its partials; returns x_{k-1} (valid id)
// to every thread of the block.
__device__ int finish_step(const DraftArgs& A, int r, int kprev, const DraftPartial* parts) {
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
        if (A.T > 0.f) {
            // base-2 state: q(x) = 2^(y_x - m) / s;  lse = ln2 (m + log2 s)
            A.q_tok[o] = (float)((double)exp2f(a.zb - a.m) / a.s);
            A.lse[o] = 0.69314718055994531 * ((double)a.m + log2(a.s));
        } else {
            A.q_tok[o] = 1.f;
            A.lse[o] = 0.0;
        }
        s_x = x;
    }
    __syncthreads();
    return s_x;
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

// Write e (float) for request r at step k into code and the bf16 hi/lo split.
__device__ __forceinline__ void store_code(const DraftArgs& A, int r, int k, int i, float e) {
    A.code[((size_t)r * A.gamma + (k - 1)) * A.r + i] = e;
    const uint16_t hi = f32_to_bf16_bits_rn(e);
    const float rest = e - bf16_bits_to_float(hi);
    A.ebf[(size_t)r * A.r + i] = hi;
    A.ebf[(size_t)A.R * A.r + (size_t)r * A.r + i] = f32_to_bf16_bits_rn(rest);
}

// prep(k) for the Markov head: x_{k-1} then e_k = W1[x_{k-1}].
__global__ void __launch_bounds__(256) draft_prep_markov(DraftArgs A, int k) {
    const int r = blockIdx.x;
    int x;
    if (k == 1) {
        x = read_anchor(A, r);
    } else {
        const DraftPartial* p = A.parts + (size_t)((k - 1) & 1) * A.parts_stride + (size_t)r * A.n_slices;
        x = finish_step(A, r, k - 1, p);
    }
    if (k > A.gamma) return;
    if (threadIdx.x == 0) A.best[r] = kOrderNegInf;
    for (int i = threadIdx.x; i < A.r; i += blockDim.x)
        store_code(A, r, k, i, ld_elem(A.W1, A.w_dtype, (size_t)x * A.r + i));
}

// prep(k) for the RNN head (blog section 3.2 RNNHead.step):
//   z = [s_{k-1}, W1[x_{k-1}], h_k];  G = z Wgco = (gate | cand | out)
//   s_k = sigmoid(gate) s_{k-1} + (1 - sigmoid(gate)) tanh(cand);  e_k = tanh(out)
__global__ void __launch_bounds__(256) draft_prep_rnn(DraftArgs A, int k) {
    extern __shared__ float zin[];   // 2r + d
    const int r = blockIdx.x;
    int x;
    if (k == 1) {
        x = read_anchor(A, r);
    } else {
        const DraftPartial* p = A.parts + (size_t)((k - 1) & 1) * A.parts_stride + (size_t)r * A.n_slices;
        x = finish_step(A, r, k - 1, p);
    }
    const int rr = A.r;
    float* srow = A.rnn_state + (size_t)r * rr;
    if (k > A.gamma) {
        if (A.state_out)
            for (int i = threadIdx.x; i < rr; i += blockDim.x) A.state_out[(size_t)r * rr + i] = srow[i];
        return;
    }
    if (threadIdx.x == 0) A.best[r] = kOrderNegInf;
    const int Kin = 2 * rr + A.d;
    for (int i = threadIdx.x; i < rr; i += blockDim.x) {
        zin[i] = (k == 1) ? 0.f : srow[i];
        zin[rr + i] = ld_elem(A.W1, A.w_dtype, (size_t)x * rr + i);
    }
    const unsigned short* Hb = static_cast<const unsigned short*>(A.H);
    for (int i = threadIdx.x; i < A.d; i += blockDim.x)
        zin[2 * rr + i] = bf16_bits_to_float(Hb[((size_t)r * A.gamma + (k - 1)) * A.d + i]);
    __syncthreads();
    for (int j = threadIdx.x; j < rr; j += blockDim.x) {
        float g = 0.f, c = 0.f, o = 0.f;
        for (int i = 0; i < Kin; ++i) {
            const float zi = zin[i];
            const size_t row = (size_t)i * 3 * rr;
            g = fmaf(zi, ld_elem(A.Wgco, A.w_dtype, row + j), g);
            c = fmaf(zi, ld_elem(A.Wgco, A.w_dtype, row + rr + j), c);
            o = fmaf(zi, ld_elem(A.Wgco, A.w_dtype, row + 2 * rr + j), o);
        }
        const float sg = 1.f / (1.f + expf(-g));
        const float sprev = zin[j];
        const float snew = sg * sprev + (1.f - sg) * tanhf(c);
        srow[j] = snew;
        store_code(A, r, k, j, tanhf(o));
    }
}

// ------------------------------------------------------------------ generic sweep
// One CTA per (V-slice of 4096, request); thread t owns columns
// v0 + 4t + 1024 g, g = 0..3.  B = e W2 on CUDA cores.
template <int UT, int WT, bool GREEDY>
__global__ void __launch_bounds__(256) draft_sweep_generic(DraftArgs A, int k) {
    extern __shared__ float e_sh[];
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
    const uint32_t req = A.req_ids ? A.req_ids[r] : (uint32_t)r;
    const PhiloxKey key = philox_key(A.seed);
    const float c2 = GREEDY ? 1.f : kLog2e / A.T;     // tempered logits in bits
    const size_t urow = ((size_t)r * A.gamma + (k - 1)) * (size_t)V;
    RowAcc a;
    acc_init(a);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float y[4];
        int c4[4];
        bool v4[4];
        float4 u = ok[g] ? load4<UT>(A.U, urow + col[g]) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            y[q] = GREEDY ? (uu[q] + acc[g][q]) : (uu[q] + acc[g][q]) * c2;
            c4[q] = col[g] + q;
            v4[q] = ok[g];
        }
        if (GREEDY) {
            acc_update_greedy<4>(a, y, c4, v4);
        } else {
            uint4 w = ok[g] ? philox4x32_10(make_uint4((uint32_t)col[g] >> 2, req, (uint32_t)k, 0u), key)
                            : make_uint4(0, 0, 0, 0);
            const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
            acc_update_exact<4>(a, y, wd, c4, v4);
        }
    }
    // block reduce -> partial of this slice
    __shared__ RowAcc sh[8];
    acc_warp_reduce(a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
}

// ------------------------------------------------------------------ host
size_t draft_workspace_bytes(int R, int gamma, int V, int r, int d) {
    (void)gamma;
    (void)d;
    const int ns = (V + kGenericSlice - 1) / kGenericSlice;
    const int ns_max = ns > 1024 ? ns : 1024;
    size_t off = sizeof(WsHeader);
    off = align_up(off + 2ull * R * ns_max * sizeof(DraftPartial), 256);
    off = align_up(off + 2ull * R * r * sizeof(uint16_t), 256);
    off = align_up(off + (size_t)R * r * sizeof(float), 256);
    off = align_up(off + (size_t)R * sizeof(uint32_t), 256);
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
    a.ebf = reinterpret_cast<uint16_t*>(base + off);
    off = align_up(off + 2ull * a.R * a.r * sizeof(uint16_t), 256);
    a.rnn_state = reinterpret_cast<float*>(base + off);
    off = align_up(off + (size_t)a.R * a.r * sizeof(float), 256);
    a.best = reinterpret_cast<uint32_t*>(base + off);
    return DSPARK_OK;
}

template <int UT, int WT, bool GREEDY>
static cudaError_t sweep_generic(DraftArgs& a, int k, cudaStream_t s) {
    dim3 grid((a.V + kGenericSlice - 1) / kGenericSlice, a.R);
    prof_begin(kPDraftSweepGeneric, s);
    draft_sweep_generic<UT, WT, GREEDY><<<grid, 256, a.r * sizeof(float), s>>>(a, k);
    prof_end(s);
    return cudaGetLastError();
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
    const bool use_tc = draft_tc_supported(a);
    a.n_slices = use_tc ? draft_tc_slices(a) : (a.V + kGenericSlice - 1) / kGenericSlice;
    const size_t rnn_smem = (size_t)(2 * a.r + a.d) * sizeof(float);
    if (rnn && rnn_smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(draft_prep_rnn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)rnn_smem);
        if (e != cudaSuccess) return e;
    }
    for (int k = 1; k <= a.gamma + 1; ++k) {
        if (rnn) {
            prof_begin(kPDraftPrepRnn, s);
            draft_prep_rnn<<<a.R, 256, rnn_smem, s>>>(a, k);
        } else {
            prof_begin(kPDraftPrep, s);
            draft_prep_markov<<<a.R, 256, 0, s>>>(a, k);
        }
        prof_end(s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (k > a.gamma) break;
        e = launch_sweep(a, k, use_tc, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dspark
