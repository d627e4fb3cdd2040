// row_acc.cuh -- per-row running state of the draft's sweep over the vocabulary.
//
// For one (request, position) row the sweep keeps
//   m, s   the log-sum-exp of z = (U_k + B_k) / T in online form, and
//   kb, ib the Gumbel-max winner so far.
// Gumbel-max (x = argmax z_v + G_v, G_v = -ln(-ln u_v)) is evaluated as an
// exponential race: the key of v is z_v - ln E_v with E_v = -ln u_v.  Since
// E_v >= t_v = 1 - u_v, the key is at most z_v - ln t_v, so an element can
// only beat the current best kb if t_v < exp(z_v - kb).  That test costs one
// multiply per element (exp(z_v - kb) = w_v exp(m_t - kb) reuses the
// log-sum-exp term w_v = exp(z_v - m_t)); only the few elements that pass it
// pay for the two logarithms of the exact key.
#pragma once

#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

// Margin on the cheap test; the exact key decides, this only has to be
// conservative against the rounding of w_v and exp(m_t - kb).
constexpr float kRaceSafety = 1.0009765625f;   // 1 + 2^-10

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

// Merge b into a (log-sum-exp part and race part).
__device__ __forceinline__ void acc_merge(RowAcc& a, const RowAcc& b) {
    if (b.m != -INFINITY) {
        if (b.m > a.m) {
            a.s = a.s * (double)ex2_approx((a.m - b.m) * kLog2e) + b.s;
            a.m = b.m;
        } else {
            a.s += b.s * (double)ex2_approx((b.m - a.m) * kLog2e);
        }
    }
    if (key_better(b.kb, b.ib, a.kb, a.ib)) {
        a.kb = b.kb;
        a.zb = b.zb;
        a.ib = b.ib;
    }
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

// Sampling update with N consecutive-in-register values of one row.
// z[i]: tempered logits, t[i] = 1 - u_i (exact), col[i]: vocabulary index,
// valid[i]: column inside [0, V).
template <int N>
__device__ __forceinline__ void acc_update_sample(RowAcc& a, const float (&z)[N], const float (&t)[N],
                                                  const int (&col)[N], const bool (&valid)[N]) {
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (valid[i]) mt = fmaxf(mt, z[i]);
    if (mt == -INFINITY) return;
    float w[N];
    float st = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        w[i] = valid[i] ? ex2_approx((z[i] - mt) * kLog2e) : 0.f;
        st += w[i];
    }
    if (mt > a.m) {
        a.s = a.s * (double)ex2_approx((a.m - mt) * kLog2e) + (double)st;
        a.m = mt;
    } else {
        a.s += (double)st * (double)ex2_approx((mt - a.m) * kLog2e);
    }
    float c = (a.kb == -INFINITY) ? INFINITY : ex2_approx((mt - a.kb) * kLog2e) * kRaceSafety;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (valid[i] && (a.kb == -INFINITY || t[i] < w[i] * c)) {
            const float key = race_key(z[i], t[i]);
            if (key_better(key, col[i], a.kb, a.ib)) {
                a.kb = key;
                a.zb = z[i];
                a.ib = col[i];
                c = ex2_approx((mt - a.kb) * kLog2e) * kRaceSafety;
            }
        }
    }
}

// Greedy update (T = 0): the key is the logit itself.
template <int N>
__device__ __forceinline__ void acc_update_greedy(RowAcc& a, const float (&y)[N], const int (&col)[N],
                                                  const bool (&valid)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (valid[i] && key_better(y[i], col[i], a.kb, a.ib)) {
            a.kb = y[i];
            a.zb = y[i];
            a.ib = col[i];
        }
}

}  // namespace dspark
