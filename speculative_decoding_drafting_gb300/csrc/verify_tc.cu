// verify_tc.cu -- tensor-core residual pass of the verifier (sm_103a, tcgen05 + cp.async).
//
// DSpark explainer, section 05: after the first rejection at position j the
// new token comes from r(v) = max(p_j(v) - q_j(v), 0) / Z.  q_j is never
// stored, so it is rebuilt here: q_j(v) = exp((U_j + e_j W2)[v] / T - lse_j)
// with e_j the rank-r code of the draft step (blog section 3.2 MarkovHead,
// B_j = W1[x_{j-1}] W2).  This pass produces the mass of every 256-column
// chunk of max(p_j - q_j, 0); the sampling kernel descends from there.
//
// One CTA = 128 rejecting requests (compact order, set by the accept pass) x a
// run of 256-column chunks.  The rows of U and P differ per request (each has
// its own j), so no tensor map describes them: every epilogue warp fetches the
// 16 columns of its own 32 rows with cp.async, two tiles ahead, into padded
// shared rows (conflict-free for the row-per-thread reads), while the rank-r
// product runs as tcgen05.mma (M = 128 requests, N = 64 columns, K = r): the
// codes (A) sit in tensor memory next to the accumulators, W2 tiles come by
// TMA through a six-stage ring.  As in the draft sweep, pairs of M-groups of
// a column slice form a cluster that shares every W2 stage by multicast; a
// cluster member whose M-group has no rejecting requests still runs the W2
// pipeline so that its peer is served.
#include <atomic>
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"
#include "sm100.cuh"

namespace dspark {

bool draft_tc_encode_available();
bool draft_tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const cuuint64_t* dims,
                       const cuuint64_t* strides_bytes, const cuuint32_t* box);

namespace {

constexpr int kBM = 128;
constexpr int kBN = 64;
constexpr int kNB = 6;             // W2 stages (64 columns x 64 rows of r, 8 KB)
constexpr int kNS = 2;             // U/P row stages
constexpr int kNACC = 2;
constexpr int kEpiWG = 4;
constexpr int kEpiWarps = 4 * kEpiWG;
constexpr int kEpiWarp0 = 3;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr uint32_t kACol = kNACC * kBN;   // A: columns [128, 128 + nsplit r/2) of tensor memory
// tensor-memory columns: two 64-column accumulators and nsplit blocks of r/2
// A columns (r <= 256: 256 columns for one bf16 term, 512 for three)
__host__ __device__ constexpr uint32_t tmem_cols_for(int nsplit) { return nsplit > 1 ? 512u : 256u; }

__host__ __device__ constexpr int pitch_of(int es) { return kBN * es + 16; }   // padded row, bytes
__host__ __device__ constexpr size_t stage_bytes(int esu, int esp) {
    return (size_t)kBM * (pitch_of(esu) + pitch_of(esp));
}
__host__ __device__ constexpr size_t smem_bytes(int /*r*/, int esu, int esp) {
    return 1024 + (size_t)kNB * 8192 + (size_t)kNS * stage_bytes(esu, esp) + 256;
}

struct ResParams {
    const uint16_t* a_res;   // codes of the rejecting requests, compact order: [3][rpad][r] bf16 terms
    int a_plane;             // elements between the hi, mid and lo planes of a_res (rpad r)
    const void* U;
    const void* P;
    const int* rej_count;
    const int* rej_list;
    const int2* vstate;
    const uint32_t* vflags;
    const double* lse;       // draft lse [R, gamma]
    const double* lsep;      // target lse [R, gamma+1]
    float* rpart;            // [R][nch256][4]
    void* ws;
    int R, gamma, V, r, ntiles, nch256, nslices;
    float c2;                // log2(e) / T
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
struct MmaBars {
    uint64_t* a_full;
    uint64_t* b_full;
    uint64_t* b_empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
};

// MMA issuer of one CTA (one thread): for every 64-column tile, r/64 W2
// stages of four K=16 steps, each step one MMA per bf16 term of the code
// (NS = 1 or 3) into the tile's accumulator.  Every stage is released to all
// CTAs of the cluster.
template <int NS, int CS>
__device__ __forceinline__ void issue_mma(const MmaBars& mb, const uint8_t* sB, uint32_t tmem, int r, int nt,
                                          int kblocks, volatile WaitState* abort_flag) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, true);
    bool ok = mbar_wait(mb.a_full, 0, abort_flag);
    tc_fence_after();
    for (int t = 0; ok && t < nt; ++t) {
        const int buf = t % kNACC;
        const uint32_t aph = (uint32_t)(t / kNACC) & 1u;
        if (!mbar_wait(&mb.acc_empty[buf], aph ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kBN);
        for (int kb = 0; ok && kb < kblocks; ++kb) {
            const int g = t * kblocks + kb;
            const int bs = g % kNB;
            if (!mbar_wait(&mb.b_full[bs], (uint32_t)(g / kNB) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint8_t* bstage = sB + (size_t)bs * 8192;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = smem_desc_sw128(bstage + kk * 2048, 1024, 1024);
                // A: 16 K values = 8 tensor-memory columns per step, one
                // block of r/2 columns per bf16 term of the code
#pragma unroll
                for (int sp = 0; sp < NS; ++sp) {
                    const uint32_t at = tmem + kACol + (uint32_t)(sp * (r / 2) + kb * 32 + kk * 8);
                    umma_bf16_ts(d, at, bd, idesc, (kb | kk | sp) ? 1u : 0u);
                }
            }
            if (CS > 1)
                umma_commit_mc(&mb.b_empty[bs], (1u << CS) - 1u);
            else
                umma_commit(&mb.b_empty[bs]);
        }
        if (!ok) break;
        umma_commit(&mb.acc_full[buf]);
    }
}

// CS: CTAs per cluster (1, 2 or 4), a template parameter so that the
// multicast masks below are compile-time constants
template <int UT, int PT, int CS>
__global__ void __launch_bounds__(kThreads, 1)
    residual_tc(const __grid_constant__ CUtensorMap tmB, ResParams p) {
    pdl_launch_dependents();
    pdl_wait();   // the rejecting requests come from the acceptance pass
    constexpr int esu = UT == DSPARK_F32 ? 4 : 2;
    constexpr int esp = PT == DSPARK_F32 ? 4 : 2;
    constexpr int pu = pitch_of(esu), pp = pitch_of(esp);
    const int n_rej = *p.rej_count;
    const int mg = blockIdx.y, slice = blockIdx.x;
    const int mg_first = mg - mg % CS;                         // first M-group of this cluster
    if (mg_first * kBM >= n_rej) return;   // nothing to do (cluster-uniform)
    // codes that are not bf16-exact (the RNN head's f32 tanh outputs) enter as
    // three bf16 terms hi + mid + lo, each multiplied into the same accumulator
    const int nsplit = (*p.vflags & 1u) ? 3 : 1;
    const uint32_t tcols = tmem_cols_for(nsplit);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sB = base;
    uint8_t* sS = sB + (size_t)kNB * 8192;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sS + (size_t)kNS * stage_bytes(esu, esp));
    uint64_t* a_full = bars;
    uint64_t* b_full = a_full + 1;
    uint64_t* b_empty = b_full + kNB;
    uint64_t* s_full = b_empty + kNB;
    uint64_t* s_empty = s_full + kNS;
    uint64_t* acc_full = s_empty + kNS;
    uint64_t* acc_empty = acc_full + kNACC;
    WaitState* wst = reinterpret_cast<WaitState*>(acc_empty + kNACC);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(wst + 1);
    volatile WaitState* abort_flag = wst;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c_begin = (int)((long long)slice * p.nch256 / p.nslices);
    const int c_end = (int)((long long)(slice + 1) * p.nch256 / p.nslices);
    const int t_begin = c_begin * 4;
    const int t_end = min(c_end * 4, p.ntiles);
    const int nt = t_end > t_begin ? t_end - t_begin : 0;
    const int kblocks = p.r / 64;
    const int rows_here = max(0, min(kBM, n_rej - mg * kBM));   // 0 for an empty M-group

    if (threadIdx.x == 0) {
        mbar_init(a_full, kEpiWarps);
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], (uint32_t)CS);   // one release per CTA of the cluster
        }
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&s_full[i], 32 * kEpiWarps);   // every epilogue thread, once its copies land
            mbar_init(&s_empty[i], kEpiWarps);       // every epilogue warp, once it has read the stage
        }
        for (int i = 0; i < kNACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        wst->abort = 0;
        wst->limit = ws_wait_limit(p.ws);
        fence_mbar_init();
        prefetch_tmap(&tmB);
    }
    if (warp == 1) tmem_alloc(tmem_holder, tcols);
    tc_fence_before();
    cluster_sync();   // the peers' barriers are initialised before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // (rows of U_j and P_j are fetched by the epilogue warps themselves)
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- W2 producer: in a cluster of cs CTAs, CTA i loads
            // K rows [i 64/cs, (i + 1) 64/cs) of every stage and multicasts them
            const uint64_t pol_last = policy_evict_last();
            constexpr int prow = 64 / CS;
            const int ro = (int)cluster_ctarank() * prow;
            constexpr uint32_t mask = (1u << CS) - 1u;
            int issued = 0;
            for (int g = 0; g < nt * kblocks; ++g) {
                const int t = g / kblocks, kb = g - t * kblocks;
                const int bs = g % kNB;
                const uint32_t bph = (uint32_t)(g / kNB) & 1u;
                if (!mbar_wait(&b_empty[bs], bph ^ 1u, abort_flag)) break;
                mbar_expect_tx(&b_full[bs], 8192u);
                if (CS == 1)
                    tma_load_2d(sB + (size_t)bs * 8192, &tmB, &b_full[bs], (t_begin + t) * kBN, kb * 64, pol_last);
                else
                    tma_load_2d_mc(sB + (size_t)bs * 8192 + ro * 128, &tmB, &b_full[bs], (t_begin + t) * kBN,
                                   kb * 64 + ro, mask, pol_last);
                issued = g + 1;
            }
            // the last release of every stage (the peers' included) lands
            // here before the CTA may exit
            for (int g = (issued > kNB ? issued - kNB : 0); g < issued && !abort_flag->abort; ++g)
                mbar_wait(&b_empty[g % kNB], (uint32_t)(g / kNB) & 1u, abort_flag);
            if (abort_flag->abort) {
                for (int g = (issued > kNB ? issued - kNB : 0); g < issued; ++g)
                    mbar_wait_for(&b_full[g % kNB], (uint32_t)(g / kNB) & 1u, abort_flag->limit);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the split count picks a straight-line body)
        if (lane == 0) {
            const MmaBars mb{a_full, b_full, b_empty, acc_full, acc_empty};
            if (nsplit == 1)
                issue_mma<1, CS>(mb, sB, tmem, p.r, nt, kblocks, abort_flag);
            else
                issue_mma<3, CS>(mb, sB, tmem, p.r, nt, kblocks, abort_flag);
        }
    } else {
        // ---------------- epilogue: thread = (rejecting request, 16-column quarter)
        const int wg = (warp - kEpiWarp0) >> 2;
        const int q = warp & 3;
        const int rit = q * 32 + lane;
        const bool row_ok = rit < rows_here;
        {
            // A operand: this thread's share (r/8 columns, r/4 values) of its
            // row's code goes to tensor memory, one block of r/2 columns per
            // bf16 term; column j of a block holds the values 2j (low half)
            // and 2j + 1 (high half)
            const int ncol = p.r / 8;
            const int c0 = wg * ncol;
            for (int sp = 0; sp < nsplit; ++sp)
                for (int c = 0; c < ncol; c += 8) {
                    uint32_t v[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    if (row_ok) {
                        const uint4* src = reinterpret_cast<const uint4*>(
                            p.a_res + (size_t)sp * p.a_plane + (size_t)(mg * kBM + rit) * p.r + 2 * (c0 + c));
                        const uint4 a0 = src[0], a1 = src[1];
                        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
                        v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
                    }
                    tmem_st8(tmem + ((uint32_t)(q * 32) << 16) + kACol + (uint32_t)(sp * (p.r / 2) + c0 + c), v);
                }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full);
        }
        const int r = row_ok ? p.rej_list[mg * kBM + rit] : 0;
        const int j = row_ok ? p.vstate[r].y : 1;
        // log2-domain normalisers, split hi + lo so the exponent is formed to
        // float precision relative to the element, not to the 17-bit lse
        const double lq2 = row_ok ? p.lse[(size_t)r * p.gamma + (j - 1)] * 1.4426950408889634 : 0.0;
        const double lp2 = row_ok ? p.lsep[(size_t)r * (p.gamma + 1) + (j - 1)] * 1.4426950408889634 : 0.0;
        const float lq_hi = (float)lq2, lq_lo = (float)(lq2 - (double)lq_hi);
        const float lp_hi = (float)lp2, lp_lo = (float)(lp2 - (double)lp_hi);
        float csum = 0.f;
        // The 16 epilogue warps fetch a tile's U_j and P_j rows together with
        // cp.async: warp e takes rows 8e .. 8e + 7 of the M-group and whole
        // 64-column segments of them (256 B per f32 row, 16 lanes a row), kNS
        // tiles ahead, into padded rows of the stage.  A stage is full when all
        // 512 threads' copies have landed (s_full) and free again when all 16
        // warps have read it (s_empty).
        constexpr int pcs_u = 4 * esu, pcs_p = 4 * esp;        // 16-byte pieces per row segment
        constexpr int rpi_u = 32 / pcs_u, rpi_p = 32 / pcs_p;  // rows per instruction
        const int e = warp - kEpiWarp0;
        const char* fsrcU[4];
        const char* fsrcP[4];
        int frU[4], frP[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            frU[i] = 8 * e + i * rpi_u + lane / pcs_u;
            frP[i] = 8 * e + i * rpi_p + lane / pcs_p;
            fsrcU[i] = nullptr;
            fsrcP[i] = nullptr;
            if (i * rpi_u < 8 && frU[i] < rows_here) {
                const int r2 = p.rej_list[mg * kBM + frU[i]];
                fsrcU[i] = static_cast<const char*>(p.U) + ((size_t)r2 * p.gamma + (p.vstate[r2].y - 1)) * (size_t)p.V * esu;
            }
            if (i * rpi_p < 8 && frP[i] < rows_here) {
                const int r2 = p.rej_list[mg * kBM + frP[i]];
                fsrcP[i] = static_cast<const char*>(p.P) + ((size_t)r2 * (p.gamma + 1) + (p.vstate[r2].y - 1)) * (size_t)p.V * esp;
            }
        }
        const int pu_lane = lane % pcs_u, pp_lane = lane % pcs_p;
        // fill number tt into stage tt % kNS; false if a wait gave up
        auto fetch = [&](int tt) -> bool {
            const int stf = tt % kNS;
            if (!mbar_wait(&s_empty[stf], ((uint32_t)(tt / kNS) & 1u) ^ 1u, abort_flag)) return false;
            if (tt < nt) {
                const int vt = (t_begin + tt) * kBN;              // first column of the tile
                uint8_t* stage = sS + (size_t)stf * stage_bytes(esu, esp);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int vu = vt + pu_lane * (16 / esu), vp = vt + pp_lane * (16 / esp);
                    if (fsrcU[i] && vu < p.V)
                        cp_async16(stage + (size_t)frU[i] * pu + pu_lane * 16, fsrcU[i] + (size_t)vu * esu);
                    if (fsrcP[i] && vp < p.V)
                        cp_async16(stage + (size_t)kBM * pu + (size_t)frP[i] * pp + pp_lane * 16,
                                   fsrcP[i] + (size_t)vp * esp);
                }
            }
            cp_async_arrive(&s_full[stf]);
            return true;
        };
        bool fok = true;
#pragma unroll
        for (int tt = 0; tt < kNS; ++tt) fok = fok && fetch(tt);
        for (int t = 0; t < nt; ++t) {
            const int tile = t_begin + t;
            const int v0 = tile * kBN + wg * 16;
            const int buf = t % kNACC;
            const uint32_t aph = (uint32_t)(t / kNACC) & 1u;
            const int st = t % kNS;
            bool ready = fok && mbar_wait(&acc_full[buf], aph, abort_flag);
            ready = ready && mbar_wait(&s_full[st], (uint32_t)(t / kNS) & 1u, abort_flag);   // every warp's copies
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            float y[16];
            tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kBN + wg * 16), y);
            const uint8_t* stage = sS + (size_t)st * stage_bytes(esu, esp);
            float pv[16];
            const uint8_t* urow = stage + (size_t)rit * pu + wg * 16 * esu;
            const uint8_t* prow = stage + (size_t)kBM * pu + (size_t)rit * pp + wg * 16 * esp;
            if (esu == 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 f = *reinterpret_cast<const float4*>(urow + 16 * c);
                    y[4 * c + 0] += f.x;
                    y[4 * c + 1] += f.y;
                    y[4 * c + 2] += f.z;
                    y[4 * c + 3] += f.w;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint4 f = *reinterpret_cast<const uint4*>(urow + 16 * c);
                    const uint32_t w4[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        y[8 * c + 2 * e] += bf16_bits_to_float(w4[e] & 0xFFFFu);
                        y[8 * c + 2 * e + 1] += bf16_bits_to_float(w4[e] >> 16);
                    }
                }
            }
            if (esp == 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 f = *reinterpret_cast<const float4*>(prow + 16 * c);
                    pv[4 * c + 0] = f.x;
                    pv[4 * c + 1] = f.y;
                    pv[4 * c + 2] = f.z;
                    pv[4 * c + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint4 f = *reinterpret_cast<const uint4*>(prow + 16 * c);
                    const uint32_t w4[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pv[8 * c + 2 * e] = bf16_bits_to_float(w4[e] & 0xFFFFu);
                        pv[8 * c + 2 * e + 1] = bf16_bits_to_float(w4[e] >> 16);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();                   // every lane has read stage st and the accumulator
            if (lane == 0) {
                mbar_arrive(&acc_empty[buf]);
                mbar_arrive(&s_empty[st]);
            }
            fok = fetch(t + kNS);           // refill this stage slot with tile t + kNS
            if (row_ok) {
                const int ncols = min(16, p.V - v0);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float qv = ex2_approx(fmaf(y[i], p.c2, -lq_hi) - lq_lo);
                    const float pw = ex2_approx(fmaf(pv[i], p.c2, -lp_hi) - lp_lo);
                    const float w = pw - qv;
                    csum += (i < ncols && w > 0.f) ? w : 0.f;
                }
            }
            if (((tile & 3) == 3 || t == nt - 1) && row_ok && !abort_flag->abort) {
                p.rpart[((size_t)r * p.nch256 + (tile >> 2)) * 4 + wg] = csum;
                csum = 0.f;
            }
        }
        // the arrivals of the last fills (past the final tile) land before the CTA leaves
        if (fok && !abort_flag->abort)
            for (int tt = nt; tt < nt + kNS; ++tt)
                mbar_wait(&s_full[tt % kNS], (uint32_t)(tt / kNS) & 1u, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag->abort) {
        // a peer's multicast copies or releases may still be on their way to
        // this CTA's shared memory: give them a millisecond before leaving
        if (threadIdx.x == 0) raise_status(p.ws, kStatTimeout);
        spin_about_1ms();
    }
    cluster_sync();   // no CTA leaves while a peer may still write into it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tcols);
    }
}

// Clusters of two residual CTAs with `smem` bytes of shared memory each that
// fit on the device at once (0 if unknown), per device.
template <int UT, int PT>
int active_clusters(int cs, size_t smem) {
    constexpr int kMaxDev = 64;
    static std::atomic<long long> cache[kMaxDev];   // (smem << 20) | count, 0 = not yet known
    int dev = 0;
    if (cs != 2 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    const long long c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0 && (size_t)(c >> 20) == smem) return (int)(c & 0xFFFFF);
    auto kern = residual_tc<UT, PT, 2>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, cs, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cs;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (n > 0 && n < (1 << 20)) cache[dev].store(((long long)smem << 20) | n, std::memory_order_relaxed);
    return n;
}

template <int UT, int PT>
cudaError_t launch_typed(VerifyArgs& a, cudaStream_t s) {
    constexpr int esu = UT == DSPARK_F32 ? 4 : 2, esp = PT == DSPARK_F32 ? 4 : 2;
    const size_t smem = smem_bytes(a.r, esu, esp);
    // M-groups per cluster: pairs when the number of groups is even (clusters
    // of four place fewer CTAs at once, as in the draft sweep)
    const int ng = (a.R + kBM - 1) / kBM;
    int cs = ng % 2 == 0 ? 2 : 1;
    int ctas = num_sms();
    if (cs > 1) {
        const int nc = active_clusters<UT, PT>(cs, smem);
        if (nc > 0)
            ctas = nc * cs;
        else
            cs = 1;
    }
    CUtensorMap tmB;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.V, (cuuint64_t)a.r};
        cuuint64_t str[1] = {(cuuint64_t)a.V * 2};
        cuuint32_t box[2] = {kBN, (cuuint32_t)(64 / cs)};
        if (!draft_tc_make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W2), dims, str, box))
            return cudaErrorInvalidValue;
    }
    ResParams p;
    p.a_res = a.a_res;
    p.a_plane = ((a.R + kBM - 1) / kBM) * kBM * a.r;
    p.U = a.U;
    p.P = a.Pv;
    p.rej_count = a.rej_count;
    p.rej_list = a.rej_list;
    p.vstate = a.vstate;
    p.vflags = a.vflags;
    p.lse = a.lse;
    p.lsep = a.lsep_ws;
    p.rpart = a.rpart;
    p.ws = a.ws;
    p.R = a.R;
    p.gamma = a.gamma;
    p.V = a.V;
    p.r = a.r;
    p.ntiles = (a.V + kBN - 1) / kBN;
    p.nch256 = a.nch256;
    int ns = ctas / ng;
    if (ns < 1) ns = 1;
    if (ns > a.nch256) ns = a.nch256;
    p.nslices = ns;
    p.c2 = 1.4426950408889634f / a.T;
    auto kern = cs == 2 ? residual_tc<UT, PT, 2> : residual_tc<UT, PT, 1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ns, ng, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cs;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    prof_begin(kPVerifyResidualTc, s);
    e = cudaLaunchKernelEx(&cfg, kern, tmB, p);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool verify_tc_supported(const VerifyArgs& a) {
    if (!(a.T > 0.f)) return false;
    if (a.w_dtype != DSPARK_BF16 || a.r % 64 != 0 || a.r > 256 || a.V % 8 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(a.U) & 15) || (reinterpret_cast<uintptr_t>(a.P) & 15) ||
        (reinterpret_cast<uintptr_t>(a.W2) & 15))
        return false;
    const int esu = a.u_dtype == DSPARK_F32 ? 4 : 2, esp = a.p_dtype == DSPARK_F32 ? 4 : 2;
    if (smem_bytes(a.r, esu, esp) > 232448) return false;
    return draft_tc_encode_available();
}

cudaError_t launch_verify_tc_residual(VerifyArgs& a, cudaStream_t s) {
    const int key = a.u_dtype * 2 + a.p_dtype;
    switch (key) {
        case 0: return launch_typed<DSPARK_F32, DSPARK_F32>(a, s);
        case 1: return launch_typed<DSPARK_F32, DSPARK_BF16>(a, s);
        case 2: return launch_typed<DSPARK_BF16, DSPARK_F32>(a, s);
        default: return launch_typed<DSPARK_BF16, DSPARK_BF16>(a, s);
    }
}

}  // namespace dspark
