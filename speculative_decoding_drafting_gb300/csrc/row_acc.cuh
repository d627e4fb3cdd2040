// row_acc.cuh -- per-row running state of the draft's sweep over the vocabulary.
//
// Everything is kept in base-2 units: y = z log2(e) with z = (U_k + B_k) / T.
// For one (request, position) row the sweep keeps
//   m, s    the log-sum-exp in online form: s = sum_v 2^(y_v - m)
//   kb, ib  the Gumbel-max winner so far: key2_v = y_v - log2(E_v), with
//           E_v = -ln u_v an Exp(1) variate (Gumbel-max as an exponential race)
// so that log-sum-exp = ln2 (m + log2 s) and q(x) = 2^(y_x - m) / s.
// At T = 0 the key is the raw logit U + B and only (kb, ib) are used.
#pragma once

#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

// Order-preserving map of float keys to unsigned (atomicMax on keys).
__device__ __forceinline__ uint32_t key_order(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_from_order(uint32_t e) {
    return __uint_as_float((e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e);
}
constexpr uint32_t kOrderNegInf = 0x007FFFFFu;   // key_order(-inf)

struct RowAcc {
    float m;
    float kb;
    float zb;
    int ib;
    double s;
};

__device__ __forceinline__ void acc_init(RowAcc& a) {
    a.m = -INFINITY;
    a.kb = -INFINITY;
    a.zb = 0.f;
    a.ib = INT_MAX;
    a.s = 0.0;
}

__device__ __forceinline__ bool key_better(float k1, int i1, float k2, int i2) {
    return k1 > k2 || (k1 == k2 && i1 < i2);
}

// Fold a chunk's (max mt, sum st of 2^(y - mt)) into the running (m, s).
__device__ __forceinline__ void acc_add_mass(RowAcc& a, float mt, float st) {
    if (mt > a.m) {
        a.s = a.s * (double)ex2_approx(a.m - mt) + (double)st;
        a.m = mt;
    } else {
        a.s += (double)st * (double)ex2_approx(mt - a.m);
    }
}

__device__ __forceinline__ void acc_take(RowAcc& a, float key, float y, int col) {
    if (key_better(key, col, a.kb, a.ib)) {
        a.kb = key;
        a.zb = y;
        a.ib = col;
    }
}

// Merge b into a.
__device__ __forceinline__ void acc_merge(RowAcc& a, const RowAcc& b) {
    if (b.m != -INFINITY) {
        if (b.m > a.m) {
            a.s = a.s * (double)ex2_approx(a.m - b.m) + b.s;
            a.m = b.m;
        } else {
            a.s += b.s * (double)ex2_approx(b.m - a.m);
        }
    }
    acc_take(a, b.kb, b.zb, b.ib);
}

__device__ __forceinline__ RowAcc acc_shfl_xor(const RowAcc& a, int o) {
    RowAcc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.kb = __shfl_xor_sync(0xffffffffu, a.kb, o);
    b.zb = __shfl_xor_sync(0xffffffffu, a.zb, o);
    b.ib = __shfl_xor_sync(0xffffffffu, a.ib, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    return b;
}

__device__ __forceinline__ void acc_warp_reduce(RowAcc& a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        RowAcc b = acc_shfl_xor(a, o);
        acc_merge(a, b);
    }
}

__device__ __forceinline__ DraftPartial acc_to_partial(const RowAcc& a) {
    DraftPartial p;
    p.m = a.m;
    p.kb = a.kb;
    p.zb = a.zb;
    p.ib = a.ib;
    p.s = a.s;
    return p;
}
__device__ __forceinline__ RowAcc partial_to_acc(const DraftPartial& p) {
    RowAcc a;
    a.m = p.m;
    a.kb = p.kb;
    a.zb = p.zb;
    a.ib = p.ib;
    a.s = p.s;
    return a;
}

// Straightforward sampling update: log-sum-exp mass and the exact race key of
// every element (the generic path; the tensor-core sweep has its own filtered
// version of the same arithmetic).
template <int N>
__device__ __forceinline__ void acc_update_exact(RowAcc& a, const float (&y)[N], const uint32_t (&word)[N],
                                                 const int (&col)[N], const bool (&valid)[N]) {
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (valid[i]) mt = fmaxf(mt, y[i]);
    if (mt == -INFINITY) return;
    float st = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (valid[i]) st += ex2_approx(y[i] - mt);
    acc_add_mass(a, mt, st);
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (valid[i]) acc_take(a, race_key2(y[i], word[i]), y[i], col[i]);
}

// Greedy update (T = 0): the key is the logit itself.
template <int N>
__device__ __forceinline__ void acc_update_greedy(RowAcc& a, const float (&y)[N], const int (&col)[N],
                                                  const bool (&valid)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (valid[i]) acc_take(a, y[i], y[i], col[i]);
}

}  // namespace dspark
