// common.cuh -- device helpers shared by the DSpark kernels.
//
// Counter-based RNG: Philox4x32-10 as published by Salmon, Moraes, Dror and
// Shaw ("Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): two 32x32->64
// multiplies per round, the high halves xored into the other two lanes with
// the round key, the key bumped by the Weyl constants between rounds.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status bits kept in the first word of every workspace.
enum : uint32_t { kStatBadToken = 1u, kStatTimeout = 2u };

struct WsHeader {
    uint32_t status;
    uint32_t test_withhold;   // test hook: 1 = the draft sweep's U producer withholds its first stage
    uint64_t wait_limit;      // SM cycles a bounded wait may take (0: the default, 2^32)
    uint32_t wait_marker;     // kWaitMarker when dspark_workspace_set_wait wrote the two fields above
    uint32_t pad[59];         // keep what follows 256-byte aligned
};
static_assert(sizeof(WsHeader) == 256, "the workspace header is 256 bytes");
// The two fields count only with the marker, so that the arbitrary contents
// of a workspace nobody set (only its status word must start at zero) leave
// the defaults in force.
constexpr uint32_t kWaitMarker = 0x57414954u;

// The bounded-wait limit and the test hook a workspace carries.
__device__ __forceinline__ uint64_t ws_wait_limit(const void* ws) {
    const WsHeader* h = static_cast<const WsHeader*>(ws);
    const uint64_t v = h->wait_marker == kWaitMarker ? h->wait_limit : 0;
    return v ? v : (1ull << 32);
}
__device__ __forceinline__ uint32_t ws_test_withhold(const void* ws) {
    const WsHeader* h = static_cast<const WsHeader*>(ws);
    return h->wait_marker == kWaitMarker ? h->test_withhold : 0u;
}

__device__ __forceinline__ void raise_status(void* ws, uint32_t bits) {
    atomicOr(reinterpret_cast<uint32_t*>(ws), bits);
}

// Programmatic dependent launch: let the next kernel of the stream be
// scheduled, and wait until the previous kernel has finished and its memory
// operations are visible (returns at once for a kernel launched without it).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- Philox
struct PhiloxKey {
    uint32_t k0, k1;
};

__host__ __device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
    return PhiloxKey{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
}

// 32 x 32 -> 64-bit product as one wide multiply.
__device__ __forceinline__ uint64_t mul_wide_u32(uint32_t a, uint32_t b) {
    uint64_t r;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
    uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint64_t p0 = mul_wide_u32(0xD2511F53u, c.x);
        const uint64_t p1 = mul_wide_u32(0xCD9E8D57u, c.z);
        const uint32_t lo0 = (uint32_t)p0, hi0 = (uint32_t)(p0 >> 32);
        const uint32_t lo1 = (uint32_t)p1, hi1 = (uint32_t)(p1 >> 32);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Philox4x32-10 with the ten round keys precomputed (kernel parameters live in
// the constant bank, so the rounds need no key arithmetic).
struct PhiloxSchedule {
    uint32_t k[20];   // (k0, k1) of rounds 0..9
};

__host__ __device__ __forceinline__ PhiloxSchedule philox_schedule(uint64_t seed) {
    PhiloxSchedule s;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int i = 0; i < 10; ++i) {
        s.k[2 * i] = k0;
        s.k[2 * i + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return s;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxSchedule& ks) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint64_t p0 = mul_wide_u32(0xD2511F53u, c.x);
        const uint64_t p1 = mul_wide_u32(0xCD9E8D57u, c.z);
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ ks.k[2 * i], (uint32_t)p1,
                       (uint32_t)(p0 >> 32) ^ c.w ^ ks.k[2 * i + 1], (uint32_t)p0);
    }
    return c;
}

// u = (w + 1/2) 2^-32 in (0, 1), exact in double.
__device__ __forceinline__ double word_to_uniform_d(uint32_t w) {
    return ((double)w + 0.5) * (1.0 / 4294967296.0);
}
// t = 1 - u = (~w + 1/2) 2^-32 in float (relative error below 2^-24).
__device__ __forceinline__ float word_to_t(uint32_t w) {
    return fmaf(__uint2float_rn(~w), 2.3283064365386963e-10f, 1.1641532182693481e-10f);
}
// A lower bound on t from the top 23 bits of ~w: floor(~w / 2^9) 2^-23 <= t.
__device__ __forceinline__ float word_to_t_lower(uint32_t w) {
    return __uint_as_float(0x3F800000u | ((~w) >> 9)) - 1.0f;
}

__device__ __forceinline__ uint32_t pick_word(uint4 w, uint32_t i) {
    return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
}

// One uniform (double) for index v of (req, pos, stream).
__device__ __forceinline__ double rng_uniform_d(PhiloxKey key, uint32_t req, uint32_t pos, uint32_t stream,
                                                uint32_t v) {
    uint4 w = philox4x32_10(make_uint4(v >> 2, req, pos, stream), key);
    return word_to_uniform_d(pick_word(w, v & 3u));
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// E = -ln(1 - t) for t in (0, 1) with small relative error everywhere: the
// Maclaurin series t + t^2/2 + ... + t^9/9 below t = 1/4 (truncation below
// t^9/10 < 4e-7 relative), the hardware base-2 logarithm of 1 - t above it
// (|log2(1 - t)| >= 0.41 there, so its absolute error stays relative-small).
__device__ __forceinline__ float neg_log1m(float t) {
    if (t < 0.25f) {
        float p = 1.f / 9.f;
        p = fmaf(p, t, 1.f / 8.f);
        p = fmaf(p, t, 1.f / 7.f);
        p = fmaf(p, t, 1.f / 6.f);
        p = fmaf(p, t, 1.f / 5.f);
        p = fmaf(p, t, 1.f / 4.f);
        p = fmaf(p, t, 1.f / 3.f);
        p = fmaf(p, t, 1.f / 2.f);
        p = fmaf(p, t, 1.f);
        return p * t;
    }
    return -kLn2 * lg2_approx(1.f - t);
}

// Gumbel-max key in base-2 units.  With y = z log2(e) the tempered logit in
// bits and t = 1 - u, E = -ln u = -ln(1 - t) is an Exp(1) variate and
// z + G = z - ln E (G = -ln(-ln u)); in bits the key is y - log2(E).
__device__ __forceinline__ float race_key2(float y, uint32_t word) {
    return y - lg2_approx(neg_log1m(word_to_t(word)));
}

// ---------------------------------------------------------------- loads
template <int DT>
struct Elem;
template <>
struct Elem<DSPARK_F32> {
    using T = float;
    static __device__ __forceinline__ float get(const float* p, size_t i) { return p[i]; }
};
template <>
struct Elem<DSPARK_BF16> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float get(const __nv_bfloat16* p, size_t i) {
        return __bfloat162float(p[i]);
    }
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// 4 consecutive elements starting at a multiple of 4 (16 B f32 / 8 B bf16).
template <int DT>
__device__ __forceinline__ float4 load4(const void* base, size_t i);
template <>
__device__ __forceinline__ float4 load4<DSPARK_F32>(const void* base, size_t i) {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
}
template <>
__device__ __forceinline__ float4 load4<DSPARK_BF16>(const void* base, size_t i) {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + i));
    return make_float4(bf16_bits_to_float(v.x & 0xFFFFu), bf16_bits_to_float(v.x >> 16),
                       bf16_bits_to_float(v.y & 0xFFFFu), bf16_bits_to_float(v.y >> 16));
}
// Streaming variant (read once): evict-first in L2, no L1 allocation.
template <int DT>
__device__ __forceinline__ float4 load4_stream(const void* base, size_t i);
template <>
__device__ __forceinline__ float4 load4_stream<DSPARK_F32>(const void* base, size_t i) {
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
}
template <>
__device__ __forceinline__ float4 load4_stream<DSPARK_BF16>(const void* base, size_t i) {
    uint2 v = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + i));
    return make_float4(bf16_bits_to_float(v.x & 0xFFFFu), bf16_bits_to_float(v.x >> 16),
                       bf16_bits_to_float(v.y & 0xFFFFu), bf16_bits_to_float(v.y >> 16));
}

// Store 4 values at element i of an array of type DT (bf16 values that came
// from bf16 storage are stored back exactly).
template <int DT>
__device__ __forceinline__ void store4(void* base, size_t i, float4 v);
template <>
__device__ __forceinline__ void store4<DSPARK_F32>(void* base, size_t i, float4 v) {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + i) = v;
}
template <>
__device__ __forceinline__ void store4<DSPARK_BF16>(void* base, size_t i, float4 v) {
    const uint32_t a = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
                       ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
    const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
                       ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + i) = make_uint2(a, b);
}

// 8 consecutive elements starting at i (a multiple of 8 for bf16, of 4 for
// f32); `avail` = how many of them exist (elements past it read as 0).
template <int DT>
__device__ __forceinline__ void load8(const void* base, size_t i, int avail, float (&w)[8]);
template <>
__device__ __forceinline__ void load8<DSPARK_BF16>(const void* base, size_t i, int avail, float (&w)[8]) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (avail >= 8) v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + i));
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        w[2 * e] = bf16_bits_to_float(x[e] & 0xFFFFu);
        w[2 * e + 1] = bf16_bits_to_float(x[e] >> 16);
    }
}
template <>
__device__ __forceinline__ void load8<DSPARK_F32>(const void* base, size_t i, int avail, float (&w)[8]) {
    const float* p = static_cast<const float*>(base) + i;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (avail >= 4) a = __ldg(reinterpret_cast<const float4*>(p));
    if (avail >= 8) b = __ldg(reinterpret_cast<const float4*>(p + 4));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// 8 consecutive values of one W2 row (bf16: kept packed until used).
template <int WT>
struct Row8;
template <>
struct Row8<DSPARK_BF16> {
    uint4 v;
    __device__ __forceinline__ void load(const void* base, size_t i, int avail) {
        v = avail >= 8 ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i))
                       : make_uint4(0u, 0u, 0u, 0u);
    }
    __device__ __forceinline__ float get(int jj) const {
        const uint32_t x = jj < 2 ? v.x : (jj < 4 ? v.y : (jj < 6 ? v.z : v.w));
        return bf16_bits_to_float((jj & 1) ? (x >> 16) : (x & 0xFFFFu));
    }
};
template <>
struct Row8<DSPARK_F32> {
    float w[8];
    __device__ __forceinline__ void load(const void* base, size_t i, int avail) { load8<DSPARK_F32>(base, i, avail, w); }
    __device__ __forceinline__ float get(int jj) const { return w[jj]; }
};

__device__ __forceinline__ float ld_elem(const void* p, int dt, size_t i) {
    if (dt == DSPARK_F32) return __ldg(static_cast<const float*>(p) + i);
    return bf16_bits_to_float(__ldg(static_cast<const unsigned short*>(p) + i));
}

// ---------------------------------------------------------------- warp ops
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__host__ __device__ __forceinline__ int ceil_log2_i(int V) {
    int L = 0;
    while ((1 << L) < V) ++L;
    return L;
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace dspark
