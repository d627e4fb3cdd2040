// draft_tc.cu -- tensor-core V sweep of one draft step (sm_103a, tcgen05, TMA for W2, cp.async for U).
//
// For step k the Markov head's bias is B_k = e_k W2 with e_k = W1[x_{k-1}]
// ("DSpark: DeepSeek 线上跑的投机解码" blog, section 3.2 MarkovHead; DSpark
// explainer, section 03, q_k = softmax(U_k + B_k)).  One CTA owns 128
// requests (an M-group) and a slice of whole 256-column chunks (every
// nslices-th chunk, upwards at odd steps and downwards at even ones), walked
// as 128-column tiles:
//
//   warp 0  U producer: the U_k tile (128 rows x 128 columns) into a ring of
//           stages, by cp.async: one warp instruction moves a row's 512
//           contiguous bytes (f32; two rows of 256 at bf16) into a padded
//           shared row, so DRAM sees 512-byte runs of each row and the
//           epilogue's row-per-thread reads are free of bank conflicts
//   warp 1  MMA issuer: r/16 tcgen05.mma (M=128, N=128, K=16, bf16 -> f32)
//           per tile into one of two TMEM accumulators
//   warp 2  W2 producer: per tile and 64-row K block the W2 stage
//           (64 x 128 bf16, evict-last) into a ring of five stages
//   warps 3-18  first the A operand: the codes e_k of the M-group go to
//           tensor memory (lane = request row), next to the accumulators,
//           which leaves shared memory to the U and W2 rings;
//           then the epilogue: thread = (request row, 32 columns of the tile);
//           tcgen05.ld the accumulator, add U_k from shared memory; sampling
//           keeps each chunk's (reference, sum of 2^(y - reference)) pair,
//           greedy the running argmax of the logits
//
// Pairs of M-groups that share a column slice form a thread-block cluster:
// every W2 stage is cut into one piece per CTA, each CTA loads its piece and
// the copy is multicast to both, so a cluster reads each W2 tile once.  A
// stage is reused only after every CTA's MMAs have released it (the release
// is multicast as well).
//
// B_k and q_k never leave the SM.  Every wait is bounded (mbar_wait); a CTA
// that gives up records DSPARK_ERR_TIMEOUT in the workspace status word,
// lets the other roles wind down, and still frees its tensor memory.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"
#include "row_acc.cuh"
#include "sm100.cuh"

namespace dspark {

namespace {

constexpr int kBM = 128;           // requests per CTA (one M-group)
constexpr int kBN = 128;           // vocabulary columns per tile
constexpr int kNB = 5;             // W2 stages, each 128 columns x 64 rows of r (16 KB)
constexpr int kNUMax = 4;          // U stages (at most; see UStage)
constexpr int kNACC = 2;           // TMEM accumulators (at most; one when A needs the room)
constexpr int kEpiWG = 4;          // epilogue warpgroups; each owns 32 of a tile's 128 columns
constexpr int kEpiWarps = 4 * kEpiWG;
constexpr int kEpiWarp0 = 3;       // warps 0..2: U producer, MMA issuer, W2 producer
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr int kBStageBytes = 16384;

// U stage of one tile: 128 rows of 128 columns, each row padded by 16 bytes
// (row r starts 16 r bytes later within the 128-byte bank window than an
// unpadded row would, so 8 consecutive rows hit 8 different 16-byte slots).
template <int UT>
struct UStage {
    static constexpr int kRowBytes = UT == DSPARK_F32 ? 512 : 256;
    static constexpr int kPitch = kRowBytes + 16;
    static constexpr int kBytes = kBM * kPitch;          // 67,584 (f32) or 34,816 (bf16)
    static constexpr int kN = UT == DSPARK_F32 ? 2 : 4;  // stages: 132 or 136 KB
};

struct TcParams {
    const void* U;           // base logits [R, gamma, V] (u_dtype)
    int gamma;
    const uint16_t* ebf;     // codes e_k, [R][r] bf16 bits
    DraftPartial* parts;     // greedy: this step's partial buffer [R][n_slices]
    float2* cmass;           // sampling: [R][nchunk][4] chunk masses
    int nchunk;
    const uint32_t* req_ids;
    void* ws;
    int R, V, r, k;          // k = 1-based step
    int ntiles, nslices;
    float c2;                // log2(e) / T
    int nsplit;              // bf16 terms of the code: 1 (bf16-exact codes), 2 or 3 (f32 codes: hi + mid (+ lo))
    int nacc;                // TMEM accumulators: 2, or 1 when the split A needs the room
};

struct Smem {
    uint8_t* B;
    uint8_t* U;
    uint64_t* a_full;
    uint64_t* b_full;
    uint64_t* b_empty;
    uint64_t* u_full;
    uint64_t* u_empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint32_t* tmem_holder;
    WaitState* wst;
};

template <int UT>
__host__ __device__ constexpr size_t smem_bytes_for() {
    return 1024 + (size_t)kNB * kBStageBytes + (size_t)UStage<UT>::kN * UStage<UT>::kBytes + 256;
}

template <int UT>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.B = base;
    s.U = s.B + (size_t)kNB * kBStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.U + (size_t)UStage<UT>::kN * UStage<UT>::kBytes);
    s.a_full = bars;
    s.b_full = bars + 1;
    s.b_empty = s.b_full + kNB;
    s.u_full = s.b_empty + kNB;
    s.u_empty = s.u_full + kNUMax;
    s.acc_full = s.u_empty + kNUMax;
    s.acc_empty = s.acc_full + kNACC;
    s.wst = reinterpret_cast<WaitState*>(s.acc_empty + kNACC);
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.wst + 1);
    return s;
}

// MMA issuer of one CTA (one thread): for every tile, r/64 W2 stages of four
// K=16 steps, each step one MMA per bf16 term of the code (NS = 1 or 3) into
// the tile's accumulator.  Every stage is released to all CTAs of the cluster.
template <int NS, int CS>
__device__ __forceinline__ void issue_mma(const Smem& S, const TcParams& p, uint32_t tmem, uint32_t acol, int nt,
                                          int kblocks) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, true);
    volatile WaitState* abort_flag = S.wst;
    // two accumulators, or one when three A blocks take the room (NS = 3, r > 128)
    const bool two = NS == 1 || p.nacc == 2;
    bool ok = mbar_wait(S.a_full, 0, abort_flag);
    tc_fence_after();
    for (int t = 0; ok && t < nt; ++t) {
        const int buf = two ? (t & 1) : 0;
        const uint32_t aph = (uint32_t)(two ? (t >> 1) : t) & 1u;
        if (!mbar_wait(&S.acc_empty[buf], aph ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kBN);
        for (int kb = 0; ok && kb < kblocks; ++kb) {
            const int g = t * kblocks + kb;
            const int bs = g % kNB;
            const uint32_t bph = (uint32_t)(g / kNB) & 1u;
            if (!mbar_wait(&S.b_full[bs], bph, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint8_t* bstage = S.B + (size_t)bs * kBStageBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // B is MN-major: 8-row K groups 1 KB apart, 64-column atoms 8 KB apart
                const uint64_t bd = smem_desc_sw128(bstage + kk * 2048, 8192, 1024);
                // A: 16 K values = 8 tensor-memory columns per step; each
                // bf16 term of the code adds its product into the same accumulator
#pragma unroll
                for (int sp = 0; sp < NS; ++sp) {
                    const uint32_t at = tmem + acol + (uint32_t)(sp * (p.r / 2) + kb * 32 + kk * 8);
                    umma_bf16_ts(d, at, bd, idesc, (kb | kk | sp) ? 1u : 0u);
                }
            }
            if (CS > 1)
                umma_commit_mc(&S.b_empty[bs], (1u << CS) - 1u);
            else
                umma_commit(&S.b_empty[bs]);
        }
        if (!ok) break;
        umma_commit(&S.acc_full[buf]);
    }
}

// CS: CTAs per cluster (1, 2 or 4), a template parameter so that the
// multicast masks below are compile-time constants
template <int UT, bool GREEDY, int CS>
__global__ void __launch_bounds__(kThreads, 1)
    draft_sweep_tc(const __grid_constant__ CUtensorMap tmB, TcParams p) {
    using US = UStage<UT>;
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve<UT>(smem_raw);
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.x, mg = blockIdx.y;
    // a slice holds the 256-column chunks slice, slice + nslices, ... (two
    // tiles each; the last chunk of the vocabulary may have one), so that at
    // any moment the slices of an M-group read neighbouring chunks of each
    // row.  Odd steps walk them upwards, even steps downwards: the W2 columns
    // a step touched last, the likeliest to be still in L2, come first in the
    // next step.  Inside a chunk the tiles go upwards.
    const int nch_mine = p.nchunk > slice ? (p.nchunk - slice + p.nslices - 1) / p.nslices : 0;
    const bool part = nch_mine > 0 && slice + (nch_mine - 1) * p.nslices == p.nchunk - 1 && (p.ntiles & 1);
    const int nt = 2 * nch_mine - (part ? 1 : 0);
    const bool down = (p.k & 1) == 0;
    auto tile_of = [&](int t) {
        const int u = down && part ? t + 1 : t;     // downwards, the one-tile chunk comes first
        const int j = down ? nch_mine - 1 - (u >> 1) : (u >> 1);
        const int half = (down && part && t == 0) ? 0 : (u & 1);
        return 2 * (slice + j * p.nslices) + half;
    };
    const int kblocks = p.r / 64;
    volatile WaitState* abort_flag = S.wst;

    if (threadIdx.x == 0) {
        mbar_init(S.a_full, kEpiWarps);
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&S.b_full[i], 1);
            mbar_init(&S.b_empty[i], (uint32_t)CS);   // one release per CTA of the cluster
        }
        for (int i = 0; i < US::kN; ++i) {
            mbar_init(&S.u_full[i], 32);                // one cp.async arrival per producer lane
            mbar_init(&S.u_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kNACC; ++i) {
            mbar_init(&S.acc_full[i], 1);
            mbar_init(&S.acc_empty[i], kEpiWarps);
        }
        S.wst->abort = 0;
        S.wst->limit = ws_wait_limit(p.ws);
        fence_mbar_init();
        prefetch_tmap(&tmB);
    }
    if (warp == 1) tmem_alloc(S.tmem_holder, kTmemCols);
    tc_fence_before();
    cluster_sync();   // the peers' barriers are initialised before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem = *S.tmem_holder;
    const uint32_t acol = (uint32_t)(p.nacc * kBN);   // A: columns [acol, acol + nsplit r/2)

    if (warp == 0) {
        // ---------------- U producer (all 32 lanes): runs up to US::kN tiles ahead.
        // f32: lane l copies bytes [16 l, 16 l + 16) of one row's 512-byte
        // segment per instruction; bf16: lanes 0-15 an even row, 16-31 the
        // next one.  Rows past R and columns past V are zero-filled (never read).
        constexpr int es = UT == DSPARK_F32 ? 4 : 2;
        constexpr int rows_per_ins = UT == DSPARK_F32 ? 1 : 2;
        const int sub = UT == DSPARK_F32 ? 0 : (lane >> 4);
        const int piece = UT == DSPARK_F32 ? lane : (lane & 15);
        const char* ubase = static_cast<const char*>(p.U);
        const size_t row_bytes = (size_t)p.gamma * p.V * es;           // from one request's rows to the next
        const int nrows = min(kBM, p.R - mg * kBM);                    // rows of this M-group
        // this lane's first row (row k - 1 of request mg 128 + sub) at column 0
        const char* lane_row0 = ubase + (size_t)(mg * kBM + sub) * row_bytes + (size_t)(p.k - 1) * p.V * es;
        const uint64_t pol_first = policy_evict_first();   // U is read once: keep L2 for W2
        // test hook (workspace header): at the first step, issue nothing for
        // the first tile, so that the epilogue's bounded wait on that stage
        // runs out with no copy in flight on it
        const bool withhold = p.k == 1 && ws_test_withhold(p.ws) == 1u;
        for (int t = 0; t < nt; ++t) {
            const int us = t % US::kN;
            const uint32_t uph = (uint32_t)(t / US::kN) & 1u;
            const bool ok = mbar_wait(&S.u_empty[us], uph ^ 1u, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (withhold && t == 0) continue;
            const int v = tile_of(t) * kBN + piece * (16 / es);     // first column of this lane's piece
            const bool col_ok = v < p.V;                               // V % (16 / es) == 0: whole pieces
            uint8_t* dst = S.U + (size_t)us * US::kBytes + sub * US::kPitch + piece * 16;
            const char* src = lane_row0 + (size_t)v * es;
#pragma unroll 8
            for (int i = 0; i < kBM / rows_per_ins; ++i) {
                const bool in = col_ok && i * rows_per_ins + sub < nrows;
                cp_async16_zf(dst + i * (rows_per_ins * US::kPitch), in ? src : ubase, in ? 16u : 0u, pol_first);
                src += rows_per_ins * row_bytes;
            }
            cp_async_arrive(&S.u_full[us]);
        }
        cp_async_wait_all();   // no copy of this warp is in flight when the CTA winds down
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- W2 producer
            const uint64_t pol_last = policy_evict_last();
            // a stage is two 64-column swizzle atoms side by side (8 KB apart);
            // in a cluster of cs CTAs, CTA i loads piece i (atom i / (cs/2),
            // K rows (i % (cs/2)) * 128/cs ..) and multicasts it to all
            const uint32_t rank = cluster_ctarank();
            constexpr int per = CS > 1 ? CS / 2 : 1;
            const int prow = 64 / per;
            const int atom = (int)rank / per, ro = ((int)rank % per) * prow;
            constexpr uint32_t mask = (1u << CS) - 1u;
            const int ng = nt * kblocks;
            int issued = 0;
            for (int g = 0; g < ng; ++g) {
                const int t = g / kblocks, kb = g - t * kblocks;
                const int bs = g % kNB;
                const uint32_t bph = (uint32_t)(g / kNB) & 1u;
                if (!mbar_wait(&S.b_empty[bs], bph ^ 1u, abort_flag)) break;
                mbar_expect_tx(&S.b_full[bs], (uint32_t)kBStageBytes);
                uint8_t* st = S.B + (size_t)bs * kBStageBytes;
                const int v0 = tile_of(t) * kBN;
                if (CS == 1) {
                    tma_load_2d(st, &tmB, &S.b_full[bs], v0, kb * 64, pol_last);
                    tma_load_2d(st + 8192, &tmB, &S.b_full[bs], v0 + 64, kb * 64, pol_last);
                } else {
                    tma_load_2d_mc(st + atom * 8192 + ro * 128, &tmB, &S.b_full[bs], v0 + atom * 64, kb * 64 + ro,
                                   mask, pol_last);
                }
                issued = g + 1;
            }
            // the last release of every stage (the peers' included) lands
            // here before the CTA may exit
            for (int g = (issued > kNB ? issued - kNB : 0); g < issued && !abort_flag->abort; ++g)
                mbar_wait(&S.b_empty[g % kNB], (uint32_t)(g / kNB) & 1u, abort_flag);
            if (abort_flag->abort) {
                for (int g = (issued > kNB ? issued - kNB : 0); g < issued; ++g)
                    mbar_wait_for(&S.b_full[g % kNB], (uint32_t)(g / kNB) & 1u, abort_flag->limit);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the split count picks a straight-line body)
        if (lane == 0) {
            if (p.nsplit == 1)
                issue_mma<1, CS>(S, p, tmem, acol, nt, kblocks);
            else if (p.nsplit == 2)
                issue_mma<2, CS>(S, p, tmem, acol, nt, kblocks);
            else
                issue_mma<3, CS>(S, p, tmem, acol, nt, kblocks);
        }
    } else {
        // ---------------- epilogue: thread = (request row, 32 columns of each tile)
        const int wg = (warp - kEpiWarp0) >> 2;      // which 32-column quarter of a tile
        const int q = warp & 3;                      // TMEM lane quarter of this warp
        const int rit = q * 32 + lane;               // row inside the tile
        const int row = mg * kBM + rit;
        const bool row_ok = row < p.R;
        // the codes and the chunk-mass buffer belong to the previous kernel
        // until it has finished (U and W2 are the caller's inputs)
        pdl_wait();
        {
            // A operand: this thread's share (r/8 columns, r/4 values) of its
            // row's code goes to tensor memory, one block of r/2 columns per
            // bf16 term; column j of a block holds the values 2j (low half)
            // and 2j + 1 (high half)
            const int ncol = p.r / 8;
            const int c0 = wg * ncol;
            for (int sp = 0; sp < p.nsplit; ++sp)
                for (int c = 0; c < ncol; c += 8) {
                    uint32_t v[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    if (row_ok) {
                        const uint4* src = reinterpret_cast<const uint4*>(p.ebf + (size_t)sp * p.R * p.r +
                                                                          (size_t)row * p.r + 2 * (c0 + c));
                        const uint4 a0 = __ldg(src), a1 = __ldg(src + 1);
                        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
                        v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
                    }
                    tmem_st8(tmem + ((uint32_t)(q * 32) << 16) + acol + (uint32_t)(sp * (p.r / 2) + c0 + c), v);
                }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.a_full);
        }
        // sampling: mass of every 256-column chunk against a per-thread reference
        // mref (bits), folded in place if a later column lies far above it;
        // greedy: the running argmax of the logits
        float mref = -INFINITY, csum = 0.f;
        float kb = -INFINITY;
        int ib = INT_MAX;
        for (int t = 0; t < nt; ++t) {
            const int tile = tile_of(t);
            const int buf = p.nacc == 2 ? (t & 1) : 0;
            const uint32_t aph = (uint32_t)(p.nacc == 2 ? (t >> 1) : t) & 1u;
            const int us = t % US::kN;
            const uint32_t uph = (uint32_t)(t / US::kN) & 1u;
            bool ready = mbar_wait(&S.acc_full[buf], aph, abort_flag);
            ready = ready && mbar_wait(&S.u_full[us], uph, abort_flag);
            if (!__all_sync(0xffffffffu, ready)) break;     // the warp stays converged
            tc_fence_after();
            const uint8_t* ust = S.U + (size_t)us * US::kBytes;
            // the thread's 32 columns of the tile: one tensor-memory load and
            // all of its U values before anything waits on them
            float y32[32];
            __syncwarp();
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kBN + wg * 32), y32);
            if (UT == DSPARK_F32) {
                const uint8_t* rowp = ust + (size_t)rit * US::kPitch + wg * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 f = *reinterpret_cast<const float4*>(rowp + c * 16);
                    y32[4 * c + 0] += f.x;
                    y32[4 * c + 1] += f.y;
                    y32[4 * c + 2] += f.z;
                    y32[4 * c + 3] += f.w;
                }
            } else {
                const uint8_t* rowp = ust + (size_t)rit * US::kPitch + wg * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 f = *reinterpret_cast<const uint4*>(rowp + c * 16);
                    const uint32_t w4[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        y32[8 * c + 2 * e + 0] += bf16_bits_to_float(w4[e] & 0xFFFFu);
                        y32[8 * c + 2 * e + 1] += bf16_bits_to_float(w4[e] >> 16);
                    }
                }
            }
            // the tile's data is in registers: hand the buffers back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&S.acc_empty[buf]);
                mbar_arrive(&S.u_empty[us]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v0 = tile * kBN + wg * 32 + h * 16;
                float* y = y32 + 16 * h;
                if (!(row_ok && v0 + 16 <= p.V)) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (!(row_ok && v0 + i < p.V)) y[i] = -INFINITY;     // edge of the vocabulary
                }
                if (GREEDY) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (y[i] > kb || (y[i] == kb && v0 + i < ib)) {   // ties: the lowest column
                            kb = y[i];
                            ib = v0 + i;
                        }
                    continue;
                }
                // y holds z = U + B; the mass is 2^(z c2 - mref)
                if (mref == -INFINITY) {
                    float zt = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 16; ++i) zt = fmaxf(zt, y[i]);
                    mref = zt * p.c2;
                }
                if (mref != -INFINITY) {
                    const float nm = -mref;
                    float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < 16; ++i) sp[i & 3] += ex2_approx(fmaf(y[i], p.c2, nm));
                    const float st = (sp[0] + sp[1]) + (sp[2] + sp[3]);
                    if (st <= 1.0e30f) {
                        csum += st;
                    } else {
                        // a column far above the reference: move it up and fold the sum
                        float zt = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 16; ++i) zt = fmaxf(zt, y[i]);
                        const float mt = zt * p.c2;
                        float s2 = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) s2 += ex2_approx(fmaf(y[i], p.c2, -mt));
                        csum = fmaf(csum, ex2_approx(mref - mt), s2);
                        mref = mt;
                    }
                }
            }
            if (!GREEDY && ((tile & 1) || tile == p.ntiles - 1)) {
                // end of a 256-column chunk (or of the vocabulary)
                if (row_ok && !abort_flag->abort)
                    p.cmass[((size_t)row * p.nchunk + (tile >> 1)) * 4 + wg] = make_float2(mref, csum);
                csum = 0.f;
            }
        }
        if (GREEDY && row_ok && !abort_flag->abort) {
            DraftPartial part;
            part.m = -INFINITY;
            part.s = 0.0;
            part.kb = kb;
            part.zb = kb;
            part.ib = ib;
            p.parts[((size_t)row * p.nslices + slice) * kEpiWG + wg] = part;
        }
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
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const cuuint64_t* dims,
              const cuuint64_t* strides_bytes, const cuuint32_t* box,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    // host-side guard: a swizzled box row must fit the 128-byte swizzle span
    const cuuint32_t es = (dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ? 4u : 2u;
    if (swz != CU_TENSOR_MAP_SWIZZLE_NONE && box[0] * es > 128u) return false;
    if ((box[0] * es) % 16u) return false;
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, (cuuint32_t)rank, base, dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// M-groups per cluster: pairs when the number of M-groups is even, else one.
// Clusters of four placed 36 at a time on a 152-SM GB300 (144 CTAs, against
// 76 pairs), and the 512-request sweep took 64.6 us per launch with them
// against 61.9 us with pairs.
int cluster_size_for(int n_mg) { return n_mg % 2 == 0 ? 2 : 1; }

// Clusters of two sweep CTAs (U storage UT) that fit on the device at once
// (0 if unknown), per device.
template <int UT>
int active_clusters(int cs) {
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev] = {};
    int dev = 0;
    if (cs != 2 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (cache[dev]) return cache[dev];
    const size_t smem = smem_bytes_for<UT>();
    auto kern = draft_sweep_tc<UT, false, 2>;
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
    cache[dev] = n;
    return n;
}

struct TcPlan {
    int cs;        // CTAs per cluster
    int nslices;   // column slices (grid.x); grid.y = M-groups
};

// One wave: as many column slices as co-resident clusters allow.
template <int UT>
TcPlan plan_for(const DraftArgs& a) {
    const int n_mg = (a.R + kBM - 1) / kBM;
    const int nchunk = (a.V + 255) / 256;
    TcPlan pl;
    pl.cs = cluster_size_for(n_mg);
    int ctas = num_sms();
    if (pl.cs > 1) {
        const int nc = active_clusters<UT>(pl.cs);
        if (nc > 0)
            ctas = nc * pl.cs;
        else
            pl.cs = 1;
    }
    int ns = ctas / n_mg;
    if (ns < 1) ns = 1;
    if (ns > nchunk) ns = nchunk;
    if (ns > 256) ns = 256;          // 4 partials per slice must fit the 1024 slots per row
    pl.nslices = ns;
    return pl;
}

template <int UT, bool GREEDY>
cudaError_t launch_typed(DraftArgs& a, int k, cudaStream_t s) {
    CUtensorMap tmB;
    const TcPlan pl = plan_for<UT>(a);
    if (pl.nslices * kEpiWG != a.n_slices) return cudaErrorInvalidValue;
    // B: W2 [r rows x V]; a copy is one 64-column swizzle atom of 64 K rows,
    // or the piece of it one CTA of a cluster loads (64 / (cs / 2) rows)
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.V, (cuuint64_t)a.r};
        cuuint64_t str[1] = {(cuuint64_t)a.V * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)(pl.cs > 1 ? 128 / pl.cs : 64)};
        if (!make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W2), dims, str, box))
            return cudaErrorInvalidValue;
    }
    TcParams p;
    p.U = a.U;
    p.gamma = a.gamma;
    p.ebf = a.ebf;
    // Markov codes are W1 rows (bf16); RNN codes tanh(out) are f32: three
    // bf16 terms hi + mid + lo (exact) when they fit in tensor memory beside
    // two accumulators (r <= 128), else hi + mid, which keep 16 significant
    // bits of every code element (the dropped term is below 2^-16 of it)
    // and keep the MMA of tile t + 1 overlapping the epilogue of tile t
    p.nsplit = a.rnn ? ((3 * (a.r / 2) + kNACC * kBN <= (int)kTmemCols) ? 3 : 2) : 1;
    p.nacc = (p.nsplit * (a.r / 2) + kNACC * kBN <= (int)kTmemCols) ? kNACC : 1;
    p.parts = a.parts + (size_t)(k & 1) * a.parts_stride;
    p.cmass = a.cmass;
    p.nchunk = a.nchunk;
    p.req_ids = a.req_ids;
    p.ws = a.ws;
    p.R = a.R;
    p.V = a.V;
    p.r = a.r;
    p.k = k;
    p.ntiles = (a.V + kBN - 1) / kBN;
    p.nslices = pl.nslices;
    p.c2 = a.T > 0.f ? kLog2e / a.T : 1.f;
    const size_t smem = smem_bytes_for<UT>();
    auto kern = pl.cs == 2 ? draft_sweep_tc<UT, GREEDY, 2> : draft_sweep_tc<UT, GREEDY, 1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.nslices, (a.R + kBM - 1) / kBM, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)pl.cs;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    prof_begin(kPDraftSweepTc, s);
    e = cudaLaunchKernelEx(&cfg, kern, tmB, p);
    prof_end(s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool draft_tc_encode_available() { return encode_fn() != nullptr; }

bool draft_tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const cuuint64_t* dims,
                       const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    return make_map(m, dt, rank, base, dims, strides_bytes, box);
}

bool draft_tc_supported(const DraftArgs& a) {
    if (a.w_dtype != DSPARK_BF16) return false;
    if (a.r % 64 != 0 || a.r > 256) return false;
    if (a.V % 8 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(a.U) & 15) || (reinterpret_cast<uintptr_t>(a.W2) & 15)) return false;
    if (smem_bytes_for<DSPARK_F32>() > 232448 || smem_bytes_for<DSPARK_BF16>() > 232448) return false;
    return encode_fn() != nullptr;
}

int draft_tc_slices(const DraftArgs& a) {
    return (a.u_dtype == DSPARK_F32 ? plan_for<DSPARK_F32>(a) : plan_for<DSPARK_BF16>(a)).nslices * kEpiWG;
}

cudaError_t launch_draft_tc_sweep(DraftArgs& a, int k, cudaStream_t s) {
    const bool greedy = !(a.T > 0.f);
    if (a.u_dtype == DSPARK_F32)
        return greedy ? launch_typed<DSPARK_F32, true>(a, k, s) : launch_typed<DSPARK_F32, false>(a, k, s);
    return greedy ? launch_typed<DSPARK_BF16, true>(a, k, s) : launch_typed<DSPARK_BF16, false>(a, k, s);
}

}  // namespace dspark
