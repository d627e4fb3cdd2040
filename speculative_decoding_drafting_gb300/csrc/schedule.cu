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
//      i.e. a descending, then r, then j ascending; a <= 0 sorts last.  A
//      pass with stride <= 32 only touches the 64 keys of its warp, so block
//      barriers are needed only around passes of stride >= 64.
//   3. tau_n = R + inclusive scan of the sorted a (double)
//   4. Theta(n) = tau_n * SPS[R + n]; n* = first n with Theta(n+1) <= Theta(n)
//   5. l_r = number of the first n* candidates that belong to r
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace dspark {

constexpr int kSchedThreads = 1024;
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

// Ascending bitonic sort of keys[0 .. Np), Np <= 2 kSchedThreads a power of
// two: thread t holds positions 2t and 2t + 1 in registers, so passes of
// stride 1 stay in the thread and strides 2 .. 32 are warp shuffles with
// thread t ^ (stride / 2); strides >= 64 go through shared memory.
__device__ void bitonic_sort_regs(unsigned long long* keys, int Np) {
    const int t = threadIdx.x;
    const bool live = 2 * t < Np;
    unsigned long long k0 = live ? keys[2 * t] : ~0ull, k1 = live ? keys[2 * t + 1] : ~0ull;
    for (int size = 2; size <= Np; size <<= 1) {
        const bool up = ((2 * t) & size) == 0;
        int stride = size >> 1;
        if (stride >= 64) {
            // cross-warp strides in shared memory, one pair per thread
            if (live) {
                keys[2 * t] = k0;
                keys[2 * t + 1] = k1;
            }
            __syncthreads();
            for (; stride >= 64; stride >>= 1) {
                const int ls = __ffs(stride) - 1;
                if (t < Np / 2) {
                    const int lo = ((t >> ls) << (ls + 1)) | (t & (stride - 1));
                    const int hi = lo + stride;
                    const bool upp = (lo & size) == 0;
                    const unsigned long long a = keys[lo], b = keys[hi];
                    if ((a > b) == upp) {
                        keys[lo] = b;
                        keys[hi] = a;
                    }
                }
                __syncthreads();
            }
            if (live) {
                k0 = keys[2 * t];
                k1 = keys[2 * t + 1];
            }
        }
        for (; stride >= 2; stride >>= 1) {
            const int pt = stride >> 1;                      // partner thread t ^ pt
            const bool lower = (t & pt) == 0;
            const unsigned long long o0 = __shfl_xor_sync(0xffffffffu, k0, pt);
            const unsigned long long o1 = __shfl_xor_sync(0xffffffffu, k1, pt);
            k0 = cmpx(k0, o0, lower, up);
            k1 = cmpx(k1, o1, lower, up);
        }
        // stride 1: the thread's own pair
        const unsigned long long lo = k0 < k1 ? k0 : k1, hi = k0 < k1 ? k1 : k0;
        k0 = up ? lo : hi;
        k1 = up ? hi : lo;
    }
    __syncthreads();
    if (live) {
        keys[2 * t] = k0;
        keys[2 * t + 1] = k1;
    }
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float* c, const double* sps, int n_sps,
                                                                 int R, int gamma, int Np, int32_t* len,
                                                                 double* theta, int32_t* nstar) {
    pdl_launch_dependents();
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
    double* val = reinterpret_cast<double*>(smem + (size_t)Np * 8);
    int* cnt = reinterpret_cast<int*>(smem + (size_t)Np * 16);
    __shared__ double wsum[kSchedThreads / 32];
    __shared__ int s_nvalid, s_nstar;
    const int tid = threadIdx.x;
    const int N = R * gamma;

    // the SPS values step 4 reads (candidate n = tid + k blockDim needs
    // SPS[R + n] and SPS[R + n + 1]), fetched now so their latency hides
    // behind the sort
    double sp0[kSchedMaxPer], sp1[kSchedMaxPer];
#pragma unroll
    for (int k = 0; k < kSchedMaxPer; ++k) {
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
            keys[idx] = (prod > 0.0f) ? (((unsigned long long)(~__float_as_uint(prod)) << 32) | (unsigned)idx)
                                      : ~0ull;
        }
        cnt[r] = 0;
    }
    for (int i = N + tid; i < Np; i += blockDim.x) keys[i] = ~0ull;
    __syncthreads();
    if (Np <= 2 * kSchedThreads) {
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
                const unsigned long long a = keys[lo], b = keys[hi];
                if ((a > b) == up) {
                    keys[lo] = b;
                    keys[hi] = a;
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
    int nv = 0;
    for (int i = b0; i < b0 + per && i < Np; ++i) {
        const unsigned long long k = keys[i];
        double a = 0.0;
        if (k != ~0ull) {
            a = (double)__uint_as_float(~(unsigned)(k >> 32));
            ++nv;
        }
        run += a;
        val[i] = run;
    }
    nv = __reduce_add_sync(0xffffffffu, (unsigned)nv);
    if ((tid & 31) == 0) atomicAdd(&s_nvalid, nv);
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
            const double th_n = tn * sp0[k];
            const double th_n1 = tn1 * sp1[k];
            if (!(th_n1 > th_n)) first = n;
        }
    }
    first = (int)__reduce_min_sync(0xffffffffu, (unsigned)first);
    if ((tid & 31) == 0 && first != INT_MAX) atomicMin(&s_nstar, first);
    __syncthreads();
    const int ns = s_nstar == INT_MAX ? nvalid : s_nstar;
    // 5: lengths
    for (int i = tid; i < ns; i += blockDim.x) {
        const int idx = (int)(unsigned)(keys[i] & 0xFFFFFFFFull);
        atomicAdd(&cnt[idx / gamma], 1);
    }
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) len[r] = cnt[r];
    if (tid == 0) {
        *nstar = ns;
        const double tn = (double)R + (ns > 0 ? val[ns - 1] : 0.0);
        *theta = tn * sps_at(sps, n_sps, (long long)R + ns);
    }
}

static int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

size_t schedule_smem_bytes(int R, int gamma) {
    const int Np = next_pow2(R * gamma < 2 ? 2 : R * gamma);
    return (size_t)Np * 16 + (size_t)R * sizeof(int);
}

cudaError_t launch_schedule(const float* c, const double* sps, int n_sps, int R, int gamma, int32_t* len,
                            double* theta, int32_t* nstar, void* ws, cudaStream_t s) {
    (void)ws;
    const int Np = next_pow2(R * gamma < 2 ? 2 : R * gamma);
    const size_t smem = schedule_smem_bytes(R, gamma);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(kPSchedule, s);
    e = launch_kernel(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, s, false, c, sps, n_sps, R, gamma, Np, len,
                      theta, nstar);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
