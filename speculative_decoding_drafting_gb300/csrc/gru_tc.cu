// gru_tc.cu -- the RNN head's GRU step (blog section 3.2 RNNHead.step) on the
// tensor cores:
//   G = z Wgco,  z = [s_{k-1}, W1[x_{k-1}], h_k],  G = (gate | cand | out),
//   s_k = sigmoid(gate) s_{k-1} + (1 - sigmoid(gate)) tanh(cand),  e_k = tanh(out).
//
// z enters as bf16: W1 rows and h are bf16 already; the float32 state s is
// split into three bf16 terms hi + mid + lo (each rounds the remainder of the
// previous ones, so their sum is s exactly).  The A operand of the product is
// therefore the row [s_hi | s_mid | s_lo | W1[x] | h] (4r + d values, padded
// with zeros to a multiple of 64), written by the RNN prep kernel, and every
// 64-row block of Wgco that meets s is multiplied three times, once per term,
// into the same float32 accumulator.
//
// gru_tc: one CTA per (64 state columns j0 .., 128 requests, one part of the
// K range).  Its N = 192 accumulator columns are the gate, candidate and
// output columns of those 64 j (three 64-column boxes of Wgco), so one tile
// holds everything the update needs.  Warp 0 loads stages by TMA (Wgco boxes
// MN-major, z boxes K-major, both 128-byte swizzled), warp 1 issues
// tcgen05.mma (M = 128, N = 192, K = 16, A and B from shared memory), warps
// 2..5 copy the accumulator to the K-part's slice of the workspace.
// gru_finish (draft.cu): one thread per (request, j): the K parts added in
// order, the GRU update, the code e_k and its bf16 terms.
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

constexpr int kGM = 128;                   // requests per CTA
constexpr int kGJ = 64;                    // state columns per CTA
constexpr int kGN = 3 * kGJ;               // accumulator columns: gate, cand, out
constexpr int kGStages = 3;
constexpr int kGBStage = 3 * 8192;         // three 64 x 64 Wgco boxes
constexpr int kGAStage = 3 * 16384;        // up to three 128 x 64 z boxes
constexpr int kGStageBytes = kGBStage + kGAStage;
constexpr int kGThreads = 192;
constexpr uint32_t kGTmemCols = 256;
constexpr int kGTargetCtas = 96;           // K parts are chosen to give about this many CTAs

struct GruParams {
    float* gpart;       // [parts][R][3r]
    void* ws;
    int R, r, kblocks, per_part, sblocks;  // sblocks = r / 64 (Wgco row blocks that meet s)
};

struct GruSmem {
    uint8_t* st;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint32_t* tmem_holder;
    WaitState* wst;
};

__device__ __forceinline__ GruSmem gru_carve(uint8_t* raw) {
    GruSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.st = base;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + (size_t)kGStages * kGStageBytes);
    s.full = bars;
    s.empty = bars + kGStages;
    s.acc_full = bars + 2 * kGStages;
    s.wst = reinterpret_cast<WaitState*>(bars + 2 * kGStages + 1);
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.wst + 1);
    return s;
}

constexpr size_t gru_smem_bytes() { return 1024 + (size_t)kGStages * kGStageBytes + 256; }

__global__ void __launch_bounds__(kGThreads, 1)
    gru_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GruParams p) {
    extern __shared__ uint8_t smem_raw[];
    const GruSmem S = gru_carve(smem_raw);
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j0 = blockIdx.x * kGJ, m0 = blockIdx.y * kGM, part = blockIdx.z;
    const int kb0 = part * p.per_part, kb1 = min(kb0 + p.per_part, p.kblocks);
    const int nkb = kb1 - kb0;
    volatile WaitState* abort_flag = S.wst;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kGStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        mbar_init(S.acc_full, 1);
        S.wst->abort = 0;
        S.wst->limit = ws_wait_limit(p.ws);
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) tmem_alloc(S.tmem_holder, kGTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *S.tmem_holder;
    // z comes from the prep kernel just before this one
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            const uint64_t pol = policy_evict_last();
            int issued = 0;
            for (int i = 0; i < nkb; ++i) {
                const int kb = kb0 + i, st = i % kGStages;
                const uint32_t ph = (uint32_t)(i / kGStages) & 1u;
                if (!mbar_wait(&S.empty[st], ph ^ 1u, abort_flag)) break;
                const bool split = kb < p.sblocks;
                mbar_expect_tx(&S.full[st], (uint32_t)(kGBStage + (split ? 3 : 1) * 16384));
                uint8_t* b = S.st + (size_t)st * kGStageBytes;
                uint8_t* a = b + kGBStage;
#pragma unroll
                for (int g = 0; g < 3; ++g) tma_load_2d(b + g * 8192, &tmB, &S.full[st], g * p.r + j0, kb * 64, pol);
                if (split) {
#pragma unroll
                    for (int t = 0; t < 3; ++t)
                        tma_load_2d(a + t * 16384, &tmA, &S.full[st], kb * 64 + t * p.r, m0, pol);
                } else {
                    // Wgco rows r .. (W1[x] and h) meet z columns 2r further on
                    tma_load_2d(a, &tmA, &S.full[st], kb * 64 + 2 * p.r, m0, pol);
                }
                issued = i + 1;
            }
            if (abort_flag->abort)   // wind down: let the copies this thread issued land
                for (int i = (issued > kGStages ? issued - kGStages : 0); i < issued; ++i)
                    mbar_wait_for(&S.full[i % kGStages], (uint32_t)(i / kGStages) & 1u, abort_flag->limit);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(kGM, kGN, true);
            for (int i = 0; i < nkb; ++i) {
                const int kb = kb0 + i, st = i % kGStages;
                if (!mbar_wait(&S.full[st], (uint32_t)(i / kGStages) & 1u, abort_flag)) break;
                tc_fence_after();
                const uint8_t* b = S.st + (size_t)st * kGStageBytes;
                const uint8_t* a = b + kGBStage;
                // B MN-major: 8-row K groups 1 KB apart, the three 64-column boxes 8 KB apart;
                // A K-major: 16 K values = 32 bytes along the swizzled 128-byte rows
                if (kb < p.sblocks) {
                    // the state's three bf16 terms against the same Wgco rows
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = smem_desc_sw128(b + kk * 2048, 8192, 1024);
#pragma unroll
                        for (int t = 0; t < 3; ++t)
                            umma_bf16(tmem, smem_desc_sw128(a + t * 16384 + kk * 32, 16, 1024), bd, idesc,
                                      (i | kk | t) ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem, smem_desc_sw128(a + kk * 32, 16, 1024), smem_desc_sw128(b + kk * 2048, 8192, 1024),
                                  idesc, (i | kk) ? 1u : 0u);
                }
                umma_commit(&S.empty[st]);
            }
            umma_commit(S.acc_full);
        }
    } else {
        // ---------------- epilogue: TMEM lane quarter (warp % 4) = 32 request rows
        const int q = warp & 3;
        const int row = m0 + q * 32 + lane;
        const bool ok = nkb > 0 && mbar_wait(S.acc_full, 0u, abort_flag);
        tc_fence_after();
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < kGN / 32; ++c) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
                if (row < p.R) {
                    const int g = c >> 1, jj = (c & 1) * 32;
                    float4* dst = reinterpret_cast<float4*>(p.gpart + ((size_t)part * p.R + row) * 3 * p.r +
                                                            (size_t)g * p.r + j0 + jj);
#pragma unroll
                    for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag->abort) {
        // tensor-core work may still be in flight: give it a millisecond
        // before the tensor memory is released
        if (threadIdx.x == 0) raise_status(p.ws, kStatTimeout);
        spin_about_1ms();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kGTmemCols);
    }
}

}  // namespace

int gru_tc_parts(int R, int r, int d) {
    const int kblocks = (2 * r + d + 63) / 64;
    const int base = (r / kGJ) * ((R + kGM - 1) / kGM);
    int parts = kGTargetCtas / (base > 0 ? base : 1);
    if (parts < 1) parts = 1;
    if (parts > kblocks) parts = kblocks;
    const int per = (kblocks + parts - 1) / parts;
    return (kblocks + per - 1) / per;
}

bool gru_tc_supported(const DraftArgs& a) {
    if (a.w_dtype != DSPARK_BF16) return false;
    if (a.r % 64 != 0 || a.r > 1024 || a.d < 1) return false;
    if (reinterpret_cast<uintptr_t>(a.Wgco) & 15) return false;
    if (gru_smem_bytes() > 232448) return false;
    return draft_tc_encode_available();
}

cudaError_t launch_gru_tc(DraftArgs& a, int k, cudaStream_t s) {
    const int kblocks = (2 * a.r + a.d + 63) / 64;
    const int parts = gru_tc_parts(a.R, a.r, a.d);
    const int per = (kblocks + parts - 1) / parts;
    CUtensorMap tmA, tmB;
    {
        // z planes [R rows x ldzb] bf16; a box is 64 columns x 128 rows
        const int ldzb = gru_ldzb(a.r, a.d);
        cuuint64_t dims[2] = {(cuuint64_t)ldzb, (cuuint64_t)a.R};
        cuuint64_t str[1] = {(cuuint64_t)ldzb * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kGM};
        if (!draft_tc_make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.zb, dims, str, box))
            return cudaErrorInvalidValue;
    }
    {
        // Wgco [2r + d rows x 3r] bf16; a box is 64 columns x 64 rows
        cuuint64_t dims[2] = {(cuuint64_t)(3 * a.r), (cuuint64_t)(2 * a.r + a.d)};
        cuuint64_t str[1] = {(cuuint64_t)(3 * a.r) * 2};
        cuuint32_t box[2] = {64, 64};
        if (!draft_tc_make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.Wgco), dims, str, box))
            return cudaErrorInvalidValue;
    }
    GruParams p;
    p.gpart = a.gpart;
    p.ws = a.ws;
    p.R = a.R;
    p.r = a.r;
    p.kblocks = kblocks;
    p.per_part = per;
    p.sblocks = a.r / 64;
    const size_t smem = gru_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(gru_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    (void)k;
    prof_begin(kPDraftRnnGru, s);
    e = launch_kernel(gru_tc, dim3(a.r / kGJ, (a.R + kGM - 1) / kGM, parts), dim3(kGThreads), smem, s, true, tmA,
                      tmB, p);
    prof_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
