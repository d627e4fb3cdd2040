// schedule.cu -- the confidence-driven greedy early-stop verify-length scheduler.
//
// Blog section 4.3 and DSpark explainer section 04: with calibrated
// confidences c, the prefix survival of request r at depth j is
// a_{r,j} = c_{r,1} ... c_{r,j}; sending l_r drafts of request r to the target
// costs B = sum_r (1 + l_r) tokens and is expected to yield
// tau = sum_r (1 + sum_{j <= l_r} a_{r,j}) tokens, so the batch objective is
// Theta = tau * SPS(B).  Extending prefixes in decreasing order of a and
// stopping at the first non-improving Theta is the page's synchronous
// algorithm.  Its inputs are c and SPS only: it never sees the target's
// logits nor any random number (the explainer's causal no-peek condition).
//
// One CTA of 1024 threads does the whole batch in shared memory:
//   1. a = running float32 product of c along each request
//   2. 64-bit keys (~bits(a) << 32 | r * gamma + j) bitonic-sorted ascending,
//      i.e. a descending, then r, then j ascending; a <= 0 sorts last.  Up to
//      2048 keys sit eight per thread in registers (warp shuffles below
//      stride 256); larger batches sort in shared memory, where a pass with
//      stride <= 32 only touches the 64 keys of its warp, so block barriers
//      are needed only around passes of stride >= 64.
//   3. tau_n = R + inclusive scan of the sorted a (double)
//   4. Theta(n) = tau_n * SPS[R + n]; n* = first n with Theta(n+1) <= Theta(n)
//   5. l_r = number of the first n* candidates that belong to r
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace dspark {

constexpr int kSchedThreads = 1024;

// Key p lives at p + p / 8 in shared memory: one spare slot per eight keys,
// so the eight consecutive keys of a sorting thread start 72 bytes after its
// neighbour's and a warp's register <-> shared transfers do not pile onto two
// banks.
__host__ __device__ __forceinline__ int kslot(int p) { return p + (p >> 3); }
constexpr int kSchedMaxPer = 8;    // candidates per thread at the largest batch (R gamma <= 8192)

__device__ __forceinline__ double sps_at(const double* sps, int n_sps, long long B) {
    return (B >= 0 && B < n_sps) ? sps[B] : 0.0;
}

// One compare-exchange of a bitonic pass: `mine` and `theirs` sit at
// positions p and p ^ stride; the lower position keeps the smaller key when
// the block of `size` containing p sorts ascending.
__device__ __forceinline__ unsigned long long cmpx(unsigned long long mine, unsigned long long theirs, bool lower,
                                                  bool up) {
    const bool keep_min = lower == up;
    return keep_min ? (mine < theirs ? mine : theirs) : (mine < theirs ? theirs : mine);
}

// One intra-thread pass of stride S (1, 2 or 4) over a thread's eight keys
// at positions p0 .. p0 + 7 of a bitonic merge of blocks of `size`.
template <int S>
__device__ __forceinline__ void intra_pass(unsigned long long (&k)[8], int p0, int size) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (e & S) continue;
        const int f = e | S;
        const bool up = ((p0 + e) & size) == 0;
        const unsigned long long a = k[e], b = k[f];
        if ((a > b) == up) {
            k[e] = b;
            k[f] = a;
        }
    }
}

// Ascending bitonic sort of keys[0 .. Np), Np <= 2048 a power of two.
// Threads 0 .. 255 hold eight keys each (positions 8t .. 8t + 7) in
// registers: strides 1, 2, 4 stay inside a thread, strides 8 .. 128 are
// warp shuffles with thread t ^ (stride / 8), strides >= 256 go through
// shared memory (all threads).  Every thread of the block must call it.
constexpr int kSortThreads = 256;
__device__ void bitonic_sort_regs(unsigned long long* keys, int Np) {
    const int t = threadIdx.x;
    const bool active = t < kSortThreads;           // whole warps
    const bool live = active && 8 * t < Np;
    unsigned long long k[8];
    // positions past Np (Np < 8) are padding: they only ever meet each other
#pragma unroll
    for (int e = 0; e < 8; ++e) k[e] = (live && 8 * t + e < Np) ? keys[kslot(8 * t + e)] : ~0ull;
    for (int size = 2; size <= Np; size <<= 1) {
        int stride = size >> 1;
        if (stride >= 256) {
            if (live)
#pragma unroll
                for (int e = 0; e < 8; ++e) keys[kslot(8 * t + e)] = k[e];
            __syncthreads();
            for (; stride >= 256; stride >>= 1) {
                const int ls = __ffs(stride) - 1;
                for (int i = t; i < Np / 2; i += blockDim.x) {
                    const int lo = ((i >> ls) << (ls + 1)) | (i & (stride - 1));
                    const int hi = lo + stride;
                    const bool upp = (lo & size) == 0;
                    const unsigned long long a = keys[kslot(lo)], b = keys[kslot(hi)];
                    if ((a > b) == upp) {
                        keys[kslot(lo)] = b;
                        keys[kslot(hi)] = a;
                    }
                }
                __syncthreads();
            }
            if (live)
#pragma unroll
                for (int e = 0; e < 8; ++e) k[e] = keys[kslot(8 * t + e)];
        }
        if (active) {
            for (; stride >= 8; stride >>= 1) {
                const int pt = stride >> 3;                  // partner thread t ^ pt, same warp
                const bool lower = (t & pt) == 0;
                const bool up = ((8 * t) & size) == 0;       // size >= 16 here: one direction per thread
#pragma unroll
                for (int e = 0; e < 8; ++e) k[e] = cmpx(k[e], __shfl_xor_sync(0xffffffffu, k[e], pt), lower, up);
            }
            if (stride >= 4) intra_pass<4>(k, 8 * t, size);
            if (stride >= 2) intra_pass<2>(k, 8 * t, size);
            intra_pass<1>(k, 8 * t, size);
        }
    }
    __syncthreads();
    if (live)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (8 * t + e < Np) keys[kslot(8 * t + e)] = k[e];
}

// budget (may be null): the capacity decided two steps back (the
// production-style scheduler of explainer section 04); the candidates fill
// min(budget, count) places instead of n*, and nstar still receives this
// step's own n* (the capacity for two steps later).  A negative budget means
// none yet.
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float* c, const double* sps, int n_sps,
                                                                 int R, int gamma, int Np, const int32_t* budget,
                                                                 int32_t* len, double* theta, int32_t* nstar) {
    pdl_launch_dependents();
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
    const int Nk = kslot(Np);                       // key slots
    double* val = reinterpret_cast<double*>(smem + (size_t)Nk * 8);
    int* cnt = reinterpret_cast<int*>(smem + (size_t)Nk * 8 + (size_t)Np * 8);
    __shared__ double wsum[kSchedThreads / 32];
    __shared__ int s_wfirst[kSchedThreads / 32];
    __shared__ int s_nvalid, s_nstar;
    const int tid = threadIdx.x;
    const int N = R * gamma;

    // the SPS values step 4 reads for this thread's first two candidates
    // (n = tid + k blockDim needs SPS[R + n] and SPS[R + n + 1]), fetched now
    // so their latency hides behind the sort; larger batches fetch the rest
    // when they get there
    constexpr int kEarly = 2;
    double sp0[kEarly], sp1[kEarly];
#pragma unroll
    for (int k = 0; k < kEarly; ++k) {
        const int n = tid + k * kSchedThreads;
        sp0[k] = n < N ? sps_at(sps, n_sps, (long long)R + n) : 0.0;
        sp1[k] = n < N ? sps_at(sps, n_sps, (long long)R + n + 1) : 0.0;
    }
    // 1-2: products and keys; c goes through shared memory (val is free until step 3)
    float* c_sh = reinterpret_cast<float*>(val);
    for (int i = tid; i < N; i += blockDim.x) c_sh[i] = c[i];
    if (tid == 0) s_nvalid = 0;
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) {
        float prod = 1.0f;
        for (int j = 0; j < gamma; ++j) {
            const int idx = r * gamma + j;
            prod = __fmul_rn(prod, c_sh[idx]);
            keys[kslot(idx)] = (prod > 0.0f) ? (((unsigned long long)(~__float_as_uint(prod)) << 32) | (unsigned)idx)
                                             : ~0ull;
        }
        cnt[r] = 0;
    }
    for (int i = N + tid; i < Np; i += blockDim.x) keys[kslot(i)] = ~0ull;
    __syncthreads();
    if (Np <= 8 * kSortThreads) {
        bitonic_sort_regs(keys, Np);
    } else {
    for (int ls = 1; (1 << ls) <= Np; ++ls) {
        const int size = 1 << ls;
        for (int lst = ls - 1; lst >= 0; --lst) {
            const int stride = 1 << lst;
            for (int i = tid; i < Np / 2; i += blockDim.x) {
                const int lo = ((i >> lst) << (lst + 1)) | (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = ((lo & size) == 0);
                const unsigned long long a = keys[kslot(lo)], b = keys[kslot(hi)];
                if ((a > b) == up) {
                    keys[kslot(lo)] = b;
                    keys[kslot(hi)] = a;
                }
            }
            // the next pass: stride / 2 within this size, else the next size's first
            const int next_stride = lst > 0 ? stride >> 1 : size;
            if (stride >= 64 || next_stride >= 64)
                __syncthreads();
            else
                __syncwarp();
        }
    }
    }
    __syncthreads();
    // 3: scan of the sorted a (double), sequential within a thread's run
    const int per = (Np + blockDim.x - 1) / blockDim.x;
    const int b0 = tid * per;
    double run = 0.0;
    for (int i = b0; i < b0 + per && i < Np; ++i) {
        const unsigned long long k = keys[kslot(i)];
        double a = 0.0;
        if (k != ~0ull) {
            a = (double)__uint_as_float(~(unsigned)(k >> 32));
            // the valid candidates sort first: the last valid one gives their count
            if (i + 1 == Np || keys[kslot(i + 1)] == ~0ull) s_nvalid = i + 1;
        }
        run += a;
        val[i] = run;
    }
    // block exclusive scan of the per-thread totals
    const int lane = tid & 31, warp = tid >> 5;
    double x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        double w = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;     // inclusive over warps
    }
    __syncthreads();
    const double offset = (x - run) + (warp > 0 ? wsum[warp - 1] : 0.0);
    for (int i = b0; i < b0 + per && i < Np; ++i) val[i] += offset;
    if (tid == 0) s_nstar = INT_MAX;
    __syncthreads();
    const int nvalid = s_nvalid;
    // 4: first non-improvement.  Theta(n) = (R + S_{n-1}) * SPS[R + n]
    int first = INT_MAX;
#pragma unroll
    for (int k = 0; k < kSchedMaxPer; ++k) {
        const int n = tid + k * kSchedThreads;
        if (n < nvalid && first == INT_MAX) {
            const double tn = (double)R + (n > 0 ? val[n - 1] : 0.0);
            const double tn1 = (double)R + val[n];
            const double s0 = k < kEarly ? sp0[k < kEarly ? k : 0] : sps_at(sps, n_sps, (long long)R + n);
            const double s1 = k < kEarly ? sp1[k < kEarly ? k : 0] : sps_at(sps, n_sps, (long long)R + n + 1);
            const double th_n = tn * s0;
            const double th_n1 = tn1 * s1;
            if (!(th_n1 > th_n)) first = n;
        }
    }
    first = (int)__reduce_min_sync(0xffffffffu, (unsigned)first);
    if ((tid & 31) == 0) s_wfirst[tid >> 5] = first;
    __syncthreads();
    if (tid < 32) {
        int f = tid < (int)(blockDim.x >> 5) ? s_wfirst[tid] : INT_MAX;
        f = (int)__reduce_min_sync(0xffffffffu, (unsigned)f);
        if (tid == 0) s_nstar = f;
    }
    __syncthreads();
    const int ns = s_nstar == INT_MAX ? nvalid : s_nstar;
    int nb = ns;
    if (budget) {
        const int b = *budget;
        nb = b < 0 ? ns : (b < nvalid ? b : nvalid);
    }
    // 5: lengths
    for (int i = tid; i < nb; i += blockDim.x) {
        const int idx = (int)(unsigned)(keys[kslot(i)] & 0xFFFFFFFFull);
        atomicAdd(&cnt[idx / gamma], 1);
    }
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) len[r] = cnt[r];
    if (tid == 0) {
        *nstar = ns;
        const double tn = (double)R + (nb > 0 ? val[nb - 1] : 0.0);
        *theta = tn * sps_at(sps, n_sps, (long long)R + nb);
    }
}

static int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

size_t schedule_smem_bytes(int R, int gamma) {
    const int Np = next_pow2(R * gamma < 2 ? 2 : R * gamma);
    return (size_t)kslot(Np) * 8 + (size_t)Np * 8 + (size_t)R * sizeof(int);
}

cudaError_t launch_schedule(const float* c, const double* sps, int n_sps, int R, int gamma, const int32_t* budget,
                            int32_t* len, double* theta, int32_t* nstar, void* ws, cudaStream_t s) {
    (void)ws;
    const int Np = next_pow2(R * gamma < 2 ? 2 : R * gamma);
    const size_t smem = schedule_smem_bytes(R, gamma);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(kPSchedule, s);
    e = launch_kernel(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, s, false, c, sps, n_sps, R, gamma, Np,
                      budget, len, theta, nstar);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Threshold filter (blog section 4.3, the confidence-threshold sweep): one
// thread per request walks its positions in order, forming the same float32
// prefix product a_{r,j} as the scheduler, and stops at the first position
// whose score (a in mode 0, c in mode 1) falls below theta (or is NaN).
__global__ void __launch_bounds__(256) schedule_threshold_kernel(const float* c, int R, int gamma, float theta,
                                                                 int mode, int32_t* len) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    const float* cr = c + (size_t)r * gamma;
    float a = 1.f;
    int n = 0;
    for (int j = 0; j < gamma; ++j) {
        const float cj = cr[j];
        a = __fmul_rn(a, cj);
        if (!((mode == 0 ? a : cj) >= theta)) break;
        ++n;
    }
    len[r] = n;
}

cudaError_t launch_schedule_threshold(const float* c, int R, int gamma, float theta, int mode, int32_t* len,
                                      cudaStream_t s) {
    prof_begin(kPScheduleThreshold, s);
    cudaError_t e = launch_kernel(schedule_threshold_kernel, dim3((R + 255) / 256), dim3(256), 0, s, false, c, R,
                                  gamma, theta, mode, len);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
