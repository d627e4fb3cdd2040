// sts.cu -- Sequential Temperature Scaling (blog section 4.2) on the GPU.
//
// Raw confidences c[n, k] of a calibration set (blocks n, positions k) are
// tempered per position, c' = sigmoid(logit(c) / t_k), with t_k chosen left
// to right from a grid: position k takes the temperature whose calibrated
// prefix survival a'_k = c'_1 ... c'_k has the smallest expected calibration
// error (Guo et al., ICML 2017, section 2: M equal-width bins,
// ECE = sum_b |B_b|/N |acc_b - conf_b| = sum_b |sum_{B_b} y - sum_{B_b} p| / N)
// against the outcome y = (accept_len >= k), with t_1 .. t_{k-1} fixed.
//
// Per position, three launches:
//   sts_hist    one CTA per (2048 samples, 8 grid points), one warp per grid
//               point; every lane keeps private per-bin sums in shared memory
//               (sum p as integers of 2^-32, exact and order-free; sum y as a
//               count), then lane b adds bin b over the 32 lanes.  p is formed
//               in float32 (no double arithmetic on this path: GB300's FP64
//               rate is a small fraction of its FP32 rate).  A value within
//               twice its float error bound (tracked per sample and position
//               from the ulp limits of logf, log1pf and expf) of an interior
//               bin edge is left out and
//               queued (sample, grid point): first in the CTA's shared memory,
//               then copied to the workspace with one reservation per CTA.
//   sts_fix     the queued values, one warp each: lane i forms position i's
//               tempered confidence in double, lane 0 multiplies them in
//               position order (the oracle's arithmetic), which decides the bin; the
//               value is added to that bin's sums with integer atomics (exact,
//               so the order does not matter).  Bin membership therefore never
//               depends on float rounding.
//   sts_ece     one CTA per (32 grid points, bin): the chunks' sums in a fixed
//               order, |sum y - sum p| in double; the last CTA to finish adds
//               the bins of every grid point in order (the ECE) and takes the
//               smallest (lowest grid index on ties) and the gap to the second.
//   sts_advance the float32 prefix survival of every sample with the chosen
//               temperature (the same expression sts_hist evaluated).
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace dspark {

namespace {

constexpr int kStsChunk = 1024;          // samples per CTA of sts_hist
constexpr int kStsWarps = 8;             // grid points per CTA (one per warp)
constexpr float kUlp = 1.1920929e-7f;    // 2^-23
constexpr double kStsScale = 4294967296.0;
constexpr int kStsLocalQ = 256;          // near-edge entries a CTA of sts_hist holds before flushing

struct StsArgs {
    const float* c;
    const int32_t* accept_len;
    int N, gamma;
    const double* grid;
    int G, M;
    double* t_out;
    int32_t* g_out;
    double* ece_out;
    double* gap_out;
    float* a_prev;                 // [N] calibrated prefix survival of the positions before k (float32)
    float* e_prev;                 // [N] bound on the relative error of a_prev against the double value
    unsigned long long* psum;      // [nchunk][M][G] sum of p, integers of 2^-32
    uint32_t* ysum;                // [nchunk][M][G] number of outcomes y = 1
    double* ece;                   // [M][G] |sum y - sum p| of each bin and grid point at the current position
    unsigned int* done;            // CTAs of sts_ece finished (the last one resets it and qcount)
    unsigned int* qcount;          // entries appended to the near-edge queue at this position
    uint2* queue;                  // [qcap] (sample, grid point) of values near a bin edge
    unsigned int qcap;
    int nchunk;
};

__device__ __forceinline__ float logit_f(float c) { return logf(c) - log1pf(-c); }

// logit in float32 and a bound on its absolute error: logf and log1pf are
// within 1 ulp and the difference rounds once, so the error is below
// 2.5 ulp of the largest of |ln c|, |ln(1 - c)| and |z|.
__device__ __forceinline__ float logit_f_err(float c, float* dz) {
    const float l0 = logf(c), l1 = log1pf(-c);
    const float z = l0 - l1;
    *dz = 2.5f * kUlp * fmaxf(fmaxf(fabsf(l0), fabsf(l1)), fabsf(z));
    return z;
}

// Bound on the relative error of the float32 tempered confidence
// 1 / (1 + expf(x)), x = -z inv_t, against the double value: the error of x
// (from z and the two roundings of the product) moves the result by (1 - s)
// times it, expf adds 2 ulp and the sum and the division one rounding each.
__device__ __forceinline__ float tempered_rel_err(float x, float s, float dz, float inv_t) {
    return (1.f - s) * (dz * inv_t + fabsf(x) * kUlp + 2.f * kUlp) + kUlp;
}
__device__ __forceinline__ double logit_d(float c) {
    const double cd = (double)c;
    return log(cd) - log1p(-cd);
}
__device__ __forceinline__ double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

// p in [0, 1] as an integer number of 2^-32 (the bits below 2^-32 dropped):
// s = p 2^16 is exact, its integer and fraction parts are exact floats.
__device__ __forceinline__ unsigned long long fixed32(float p) {
    const float s = p * 65536.f;
    const uint32_t hi = (uint32_t)s;
    const uint32_t lo = (uint32_t)((s - (float)hi) * 65536.f);
    return ((unsigned long long)hi << 16) + lo;
}

// The calibrated prefix survival of sample n through position k in double,
// as the oracle forms it: a = 1, then a *= sigmoid(logit(c_i) / t_i) for
// i = 1 .. k with t_i the chosen temperatures and t_k = tk.
__device__ __noinline__ double survival_exact(const StsArgs& A, int n, int k, double tk) {
    double a = 1.0;
    for (int i = 1; i <= k; ++i) {
        const double t = i < k ? A.t_out[i - 1] : tk;
        a *= sigmoid_d(logit_d(A.c[(size_t)n * A.gamma + (i - 1)]) / t);
    }
    return a;
}

// One warp of sts_hist: grid point g over the chunk's samples.
__device__ __forceinline__ void hist_warp(const StsArgs& A, int k, int g, int n0, int nn, unsigned long long* lp,
                                          uint32_t* ly, const float* sa, const float* sz, const float* sdz,
                                          const float* se, const unsigned char* sy, uint2* s_q, unsigned int* s_nq) {
    const int M = A.M;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const double tg = A.grid[g];
    const float inv_t = (float)(1.0 / tg);
    const float fM = (float)M;
    unsigned long long* mp = lp + (size_t)warp * M * 32 + lane;
    uint32_t* my = ly + (size_t)warp * M * 32 + lane;
    for (int i = lane; i < nn; i += 32) {
        const float x = -sz[i] * inv_t;
        const float sg = 1.f / (1.f + expf(x));
        const float p = sa[i] * sg;
        const float q = p * fM;
        // only the interior edges 1 .. M-1 separate bins (0 and M are clamped);
        // a value whose error bound (doubled) reaches an edge is decided in double
        const float edge = rintf(q);
        int b;
        unsigned long long pi;
        if (edge >= 1.f && edge <= fM - 1.f &&
            fabsf(q - edge) < 2.f * q * (se[i] + tempered_rel_err(x, sg, sdz[i], inv_t) + kUlp)) {
            // near a bin edge: the oracle's double arithmetic decides, in
            // sts_fix; here only when the CTA's queue is full
            const unsigned int slot = atomicAdd(s_nq, 1u);
            if (slot < (unsigned int)kStsLocalQ) {
                s_q[slot] = make_uint2((unsigned)(n0 + i), (unsigned)g);
                continue;
            }
            const double pd = survival_exact(A, n0 + i, k, tg);
            b = (int)floor(pd * (double)M);
            pi = (unsigned long long)(pd * kStsScale);
        } else {
            b = (int)q;
            pi = fixed32(p);
        }
        b = min(max(b, 0), M - 1);
        mp[b * 32] += pi;
        my[b * 32] += sy[i];
    }
    __syncwarp();
    if (lane < M) {
        const unsigned long long* rp = lp + ((size_t)warp * M + lane) * 32;
        const uint32_t* ry = ly + ((size_t)warp * M + lane) * 32;
        unsigned long long sp = 0ull;
        uint32_t sy_ = 0u;
        for (int j = 0; j < 32; ++j) {
            sp += rp[j];
            sy_ += ry[j];
        }
        const size_t o = ((size_t)blockIdx.x * M + lane) * A.G + g;
        A.psum[o] = sp;
        A.ysum[o] = sy_;
    }
}

__global__ void __launch_bounds__(256) sts_hist(StsArgs A, int k) {
    pdl_launch_dependents();
    pdl_wait();   // a_prev comes from the previous position's sts_advance
    extern __shared__ unsigned long long sts_smem[];
    const int M = A.M;
    unsigned long long* lp = sts_smem;                                     // [warp][M][32]
    uint32_t* ly = reinterpret_cast<uint32_t*>(lp + kStsWarps * M * 32);  // [warp][M][32]
    float* sa = reinterpret_cast<float*>(ly + kStsWarps * M * 32);        // [chunk] a_prev
    float* sz = sa + kStsChunk;                                            // [chunk] logit of c_k
    float* sdz = sz + kStsChunk;                                           // [chunk] its error bound
    float* se = sdz + kStsChunk;                                           // [chunk] a_prev's relative error bound
    unsigned char* sy = reinterpret_cast<unsigned char*>(se + kStsChunk); // [chunk] outcome
    __shared__ uint2 s_q[kStsLocalQ];
    __shared__ unsigned int s_nq, s_base;
    if (threadIdx.x == 0) s_nq = 0u;
    const int n0 = blockIdx.x * kStsChunk;
    const int nn = min(kStsChunk, A.N - n0);
    for (int i = threadIdx.x; i < nn; i += blockDim.x) {
        const int n = n0 + i;
        float dz;
        sz[i] = logit_f_err(A.c[(size_t)n * A.gamma + (k - 1)], &dz);
        sdz[i] = dz;
        sa[i] = k > 1 ? A.a_prev[n] : 1.f;
        se[i] = k > 1 ? A.e_prev[n] : 0.f;
        sy[i] = A.accept_len[n] >= k ? 1 : 0;
    }
    for (int i = threadIdx.x; i < kStsWarps * M * 32; i += blockDim.x) {
        lp[i] = 0ull;
        ly[i] = 0u;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y * kStsWarps + warp;
    if (g < A.G) hist_warp(A, k, g, n0, nn, lp, ly, sa, sz, sdz, se, sy, s_q, &s_nq);
    // the CTA's queued entries go to the workspace queue (one reservation)
    __syncthreads();
    const unsigned int nq = min(s_nq, (unsigned int)kStsLocalQ);
    if (nq == 0u) return;
    if (threadIdx.x == 0) s_base = atomicAdd(A.qcount, nq);
    __syncthreads();
    for (unsigned int e = threadIdx.x; e < nq; e += blockDim.x) {
        const unsigned int slot = s_base + e;
        if (slot < A.qcap) {
            A.queue[slot] = s_q[e];
        } else {
            // workspace queue full: decide here
            const uint2 qe = s_q[e];
            const double pd = survival_exact(A, (int)qe.x, k, A.grid[qe.y]);
            const int b = min(max((int)floor(pd * (double)A.M), 0), A.M - 1);
            const size_t o = ((size_t)blockIdx.x * A.M + b) * A.G + qe.y;
            atomicAdd(&A.psum[o], (unsigned long long)(pd * kStsScale));
            if (A.accept_len[qe.x] >= k) atomicAdd(&A.ysum[o], 1u);
        }
    }
}

// The queued near-edge values of position k, one warp each: lane i forms the
// tempered confidence of position i + 1 (and i + 33) in double, every lane
// multiplies them in position order (the oracle's order), lane 0 adds the value
// to its bin's sums in the sample's chunk.
__global__ void __launch_bounds__(256) sts_fix(StsArgs A, int k) {
    pdl_launch_dependents();
    pdl_wait();
    const unsigned int nq = min(*A.qcount, A.qcap);
    const int M = A.M;
    const int lane = threadIdx.x & 31;
    const unsigned int nw = (gridDim.x * blockDim.x) >> 5;
    for (unsigned int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; e < nq; e += nw) {
        const uint2 qe = A.queue[e];
        const int n = (int)qe.x, g = (int)qe.y;
        const float* cn = A.c + (size_t)n * A.gamma;
        double f0 = 1.0, f1 = 1.0;
        if (lane < k) f0 = sigmoid_d(logit_d(cn[lane]) / (lane + 1 < k ? A.t_out[lane] : A.grid[g]));
        if (lane + 32 < k) f1 = sigmoid_d(logit_d(cn[lane + 32]) / (lane + 33 < k ? A.t_out[lane + 32] : A.grid[g]));
        double pd = 1.0;
        for (int i = 0; i < k; ++i) pd *= __shfl_sync(0xffffffffu, i < 32 ? f0 : f1, i & 31);
        if (lane == 0) {
            const int b = min(max((int)floor(pd * (double)M), 0), M - 1);
            const size_t o = ((size_t)(n / kStsChunk) * M + b) * A.G + g;
            atomicAdd(&A.psum[o], (unsigned long long)(pd * kStsScale));
            if (A.accept_len[n] >= k) atomicAdd(&A.ysum[o], 1u);
        }
    }
}

// (best, its index, second best) of a set of ECE values; ties keep the lower index.
struct Best {
    double b;
    int i;
    double s;
};

__device__ __forceinline__ Best merge(Best x, Best y) {
    const bool xf = x.b < y.b || (x.b == y.b && x.i < y.i);
    Best r;
    r.b = xf ? x.b : y.b;
    r.i = xf ? x.i : y.i;
    r.s = xf ? fmin(x.s, y.b) : fmin(y.s, x.b);
    return r;
}

// One CTA per (32 grid points, bin b = blockIdx.y): thread (l, j) adds the
// chunks l, l + 32, ... of grid point 32 blockIdx.x + j, then the 32 partial
// sums of each grid point are added in order and |sum y - sum p| is stored.
// The last CTA to finish forms every grid point's ECE (bins in order) and
// picks the temperature.
__global__ void __launch_bounds__(1024) sts_ece(StsArgs A, int k) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ unsigned long long s_p[32][33];
    __shared__ unsigned int s_y[32][33];
    __shared__ Best s_w[32];
    __shared__ bool s_last;
    const int M = A.M, b = blockIdx.y;
    const int j = threadIdx.x & 31, l = threadIdx.x >> 5;
    const int g = blockIdx.x * 32 + j;
    unsigned long long sp = 0ull;
    unsigned int sy = 0u;
    if (g < A.G) {
#pragma unroll 4
        for (int ch = l; ch < A.nchunk; ch += 32) {
            const size_t o = ((size_t)ch * M + b) * A.G + g;
            sp += A.psum[o];
            sy += A.ysum[o];
        }
    }
    s_p[l][j] = sp;
    s_y[l][j] = sy;
    __syncthreads();
    if (l == 0 && g < A.G) {
        unsigned long long tp = 0ull;
        unsigned int ty = 0u;
        for (int ll = 0; ll < 32; ++ll) {
            tp += s_p[ll][j];
            ty += s_y[ll][j];
        }
        A.ece[(size_t)b * A.G + g] = fabs((double)ty - (double)tp / kStsScale);
    }
    // the last CTA to finish picks the temperature
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(A.done, 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    Best mine{INFINITY, INT_MAX, INFINITY};
    const volatile double* eb = A.ece;
    for (int gg = threadIdx.x; gg < A.G; gg += blockDim.x) {
        double e = 0.0;
        for (int bb = 0; bb < M; ++bb) e += eb[(size_t)bb * A.G + gg];
        mine = merge(mine, Best{e / (double)A.N, gg, INFINITY});
    }
    for (int o = 16; o > 0; o >>= 1) {
        Best other;
        other.b = __shfl_xor_sync(0xffffffffu, mine.b, o);
        other.i = __shfl_xor_sync(0xffffffffu, mine.i, o);
        other.s = __shfl_xor_sync(0xffffffffu, mine.s, o);
        mine = merge(mine, other);
    }
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = mine;
    __syncthreads();
    if (threadIdx.x == 0) {
        Best r = s_w[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = merge(r, s_w[w]);
        A.t_out[k - 1] = A.grid[r.i];
        A.g_out[k - 1] = r.i;
        A.ece_out[k - 1] = r.b;
        A.gap_out[k - 1] = r.s - r.b;
        *A.done = 0u;
        *A.qcount = 0u;
    }
}

__global__ void __launch_bounds__(256) sts_advance(StsArgs A, int k) {
    pdl_launch_dependents();
    pdl_wait();
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= A.N) return;
    const float inv_t = (float)(1.0 / A.t_out[k - 1]);
    const float a = k > 1 ? A.a_prev[n] : 1.f;
    const float e = k > 1 ? A.e_prev[n] : 0.f;
    float dz;
    const float x = -logit_f_err(A.c[(size_t)n * A.gamma + (k - 1)], &dz) * inv_t;
    const float sg = 1.f / (1.f + expf(x));
    A.a_prev[n] = a * sg;
    A.e_prev[n] = e + tempered_rel_err(x, sg, dz, inv_t) + kUlp;
}

// c_out = sigmoid(logit(c) / t_k), float32.
__global__ void __launch_bounds__(256) sts_apply_kernel(const float* c, int N, int gamma, const double* t,
                                                        float* out) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)N * gamma) return;
    const float inv_t = (float)(1.0 / t[i % gamma]);
    out[i] = 1.f / (1.f + expf(-logit_f(c[i]) * inv_t));
}

// Near-edge queue capacity: the expected load is a few 1e-4 of the N G values
// of a position; degenerate inputs (every value on an edge) overflow it and are
// then decided inline.
unsigned int sts_queue_cap(int N, int G) {
    const unsigned long long want = (unsigned long long)N * (unsigned long long)G / 64ull + 4096ull;
    return (unsigned int)(want < (1ull << 22) ? want : (1ull << 22));
}

size_t hist_smem(int M) {
    return (size_t)kStsWarps * M * 32 * (8 + 4) + (size_t)kStsChunk * (4 + 4 + 4 + 4 + 1);
}

}  // namespace

size_t sts_workspace_bytes(int N, int gamma, int G, int M) {
    (void)gamma;
    const size_t nchunk = (size_t)(N + kStsChunk - 1) / kStsChunk;
    size_t off = sizeof(WsHeader);
    off = align_up(off + 256, 256);                                          // done, qcount
    off = align_up(off + (size_t)sts_queue_cap(N, G) * sizeof(uint2), 256);  // near-edge queue
    off = align_up(off + (size_t)N * sizeof(float), 256);                    // a_prev
    off = align_up(off + (size_t)N * sizeof(float), 256);                    // e_prev
    off = align_up(off + (size_t)M * G * sizeof(double), 256);               // ece per bin
    off = align_up(off + nchunk * M * G * sizeof(unsigned long long), 256);  // psum
    off = align_up(off + nchunk * M * G * sizeof(uint32_t), 256);            // ysum
    return off;
}

cudaError_t launch_sts_fit(const float* c, const int32_t* accept_len, int N, int gamma, const double* grid, int G,
                           int M, double* t_out, int32_t* g_out, double* ece_out, double* gap_out, void* ws,
                           cudaStream_t s) {
    StsArgs A;
    A.c = c;
    A.accept_len = accept_len;
    A.N = N;
    A.gamma = gamma;
    A.grid = grid;
    A.G = G;
    A.M = M;
    A.t_out = t_out;
    A.g_out = g_out;
    A.ece_out = ece_out;
    A.gap_out = gap_out;
    A.nchunk = (N + kStsChunk - 1) / kStsChunk;
    char* base = static_cast<char*>(ws);
    size_t off = sizeof(WsHeader);
    A.done = reinterpret_cast<unsigned int*>(base + off);
    A.qcount = A.done + 1;
    off = align_up(off + 256, 256);
    A.qcap = sts_queue_cap(N, G);
    A.queue = reinterpret_cast<uint2*>(base + off);
    off = align_up(off + (size_t)A.qcap * sizeof(uint2), 256);
    A.a_prev = reinterpret_cast<float*>(base + off);
    off = align_up(off + (size_t)N * sizeof(float), 256);
    A.e_prev = reinterpret_cast<float*>(base + off);
    off = align_up(off + (size_t)N * sizeof(float), 256);
    A.ece = reinterpret_cast<double*>(base + off);
    off = align_up(off + (size_t)M * G * sizeof(double), 256);
    A.psum = reinterpret_cast<unsigned long long*>(base + off);
    off = align_up(off + (size_t)A.nchunk * M * G * sizeof(unsigned long long), 256);
    A.ysum = reinterpret_cast<uint32_t*>(base + off);
    const size_t smem = hist_smem(M);
    cudaError_t e = cudaFuncSetAttribute(sts_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(A.done, 0, 2 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const dim3 hgrid(A.nchunk, (G + kStsWarps - 1) / kStsWarps);
    for (int k = 1; k <= gamma; ++k) {
        prof_begin(kPStsHist, s);
        e = launch_kernel(sts_hist, hgrid, dim3(256), smem, s, k > 1, A, k);
        prof_end(s);
        if (e != cudaSuccess) return e;
        prof_begin(kPStsFix, s);
        e = launch_kernel(sts_fix, dim3(num_sms()), dim3(256), 0, s, true, A, k);
        prof_end(s);
        if (e != cudaSuccess) return e;
        prof_begin(kPStsEce, s);
        e = launch_kernel(sts_ece, dim3((G + 31) / 32, M), dim3(1024), 0, s, true, A, k);
        prof_end(s);
        if (e != cudaSuccess) return e;
        if (k < gamma) {
            prof_begin(kPStsAdvance, s);
            e = launch_kernel(sts_advance, dim3((N + 255) / 256), dim3(256), 0, s, true, A, k);
            prof_end(s);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaGetLastError();
}

cudaError_t launch_sts_apply(const float* c, int N, int gamma, const double* t, float* out, cudaStream_t s) {
    const size_t n = (size_t)N * gamma;
    prof_begin(kPStsApply, s);
    cudaError_t e = launch_kernel(sts_apply_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, false, c, N,
                                  gamma, t, out);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
