// kernels.h -- internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dspark {

// Per-(request, step, V-slice) partial state of the draft's reduction over V:
// running max and sum for the log-sum-exp, and the best race key so far.
struct DraftPartial {
    float m;       // max of z over the slice (-inf if empty)
    float kb;      // best key (z - ln E, or the logit itself at T = 0)
    float zb;      // z of the best element
    int ib;        // its vocabulary index (INT_MAX if empty)
    double s;      // sum of exp(z - m) over the slice
};

struct DraftArgs {
    const void* U;
    int u_dtype;
    const int32_t* anchor;
    const void* W1;
    const void* W2;
    const void* Wgco;   // RNN only
    const void* H;      // RNN only (bf16)
    int w_dtype;
    int R, gamma, V, r, d;
    uint64_t seed;
    const uint32_t* req_ids;
    float T;
    int32_t* tokens;
    float* q_tok;
    double* lse;
    float* code;
    float* state_out;
    // confidence head c_k = sigmoid(wc . [h_k, W1[x_{k-1}]]) (conf == nullptr: off)
    const void* Hc;           // [R, gamma, dc] bf16
    const float* wc;          // [dc + r]
    int dc;
    float* conf;              // [R, gamma]
    const double* tc;         // [gamma] per-position temperatures (STS), nullptr: none
    // workspace carve-up
    void* ws;
    DraftPartial* parts;      // [2][R][n_slices]
    uint16_t* ebf;            // [3][R][r] bf16 bits of e_k = hi + mid + lo (exact for f32 e_k)
    float* rnn_state;         // [R][r]
    float* zbuf;              // RNN head: [R][2r + d] GRU input z of the current step (CUDA-core GRU)
    uint16_t* zb;             // RNN head: [R][ldzb] bf16 z = [s_hi | s_mid | s_lo | W1[x] | h | 0] (tensor-core GRU)
    float* gpart;             // RNN head: [parts][R][3r] partial G of the K parts (tensor-core GRU)
    int gru_tc;               // 1: the GRU step runs on the tensor cores
    int gru_parts;            // K parts of the tensor-core GRU
    uint32_t* best;           // [R] best race key of the current step (order-preserving bits)
    float2* cmass;            // [R][nchunk][4] (reference m, sum 2^(y - m)) per 256-column chunk
    int nchunk;               // ceil(V / 256)
    int rnn;                  // 1 for the RNN head
    int n_slices;             // V-slices per request in the active sweep
    int parts_stride;         // R * n_slices_max
};

struct VerifyArgs {
    const void* P;
    int p_dtype;
    void* P_stage;      // optional device copy of P that pass 1 fills with the rows it reads
    int unit_waves;     // 1: one target row per verification wave (set with P_stage)
    const void* Pv;     // where the passes after pass 1 read P: P_stage, or P itself
    const void* U;
    int u_dtype;
    const void* W2;
    int w_dtype;
    const int32_t* tokens;
    const float* q_tok;
    const double* lse;
    const float* code;
    const int32_t* verify_len;
    int R, gamma, V, r;
    uint64_t seed;
    const uint32_t* req_ids;
    float T;
    int32_t* out_tokens;
    int32_t* accept_len;
    int32_t* n_out;
    float* p_tok;
    double* lse_p;
    // workspace
    void* ws;
    float2* vparts;     // [R][gamma+1][NCH]  (m, s) or (max, idx bits)
    double* lsep_ws;    // [R][gamma+1]
    int2* vstate;       // [R] (mode, position)
    int nch;            // number of 1024-wide chunks of V (target-row partials)
    int nch256;         // number of 256-wide chunks of V (residual masses)
    float* rpart;       // [R][nch256][4] partial residual masses
    int* rej_count;     // number of requests that rejected a draft
    int* wcount_alive;  // [6] requests live at each verification wave (index = wave)
    int* alive;         // [2][R] live requests of the current and the next wave
    int* live_mark;     // [R] the wave a request is still undecided in (0: decided); written by every acceptance pass
    int* rej_list;      // [R] those requests, in arrival order
    uint16_t* a_res;    // [3][rpad][r] bf16 terms hi, mid, lo of the rejecting requests' codes e_j (compact order; rpad = R rounded up to 128)
    uint32_t* vflags;   // bit 0: some rejecting code is not bf16-exact
    int tc;             // 1 if the tensor-core residual pass is launched
};

constexpr int kChunk = 1024;          // chunk of the target-row partials (bonus draws)
constexpr int kChunkLog2 = 10;
constexpr int kRChunk = 256;          // chunk of the residual masses and of the draft's first Gumbel level
constexpr int kRChunkLog2 = 8;
constexpr int kGenericSlice = 4096;   // V-slice of the generic draft sweep

enum VerifyMode : int { kModeDone = 0, kModeResidual = 1, kModeBonus = 2 };

size_t draft_workspace_bytes(int R, int gamma, int V, int r, int d);
int draft_carve(DraftArgs& a, size_t ws_bytes);
cudaError_t launch_draft(DraftArgs& a, bool rnn, cudaStream_t s);

size_t verify_workspace_bytes(int R, int gamma, int V, int r);
int verify_carve(VerifyArgs& a, size_t ws_bytes);
cudaError_t launch_verify(VerifyArgs& a, cudaStream_t s);

size_t schedule_smem_bytes(int R, int gamma);
size_t sts_workspace_bytes(int N, int gamma, int G, int M);
cudaError_t launch_sts_fit(const float* c, const int32_t* accept_len, int N, int gamma, const double* grid, int G,
                           int M, double* t_out, int32_t* g_out, double* ece_out, double* gap_out, void* ws,
                           cudaStream_t s);
cudaError_t launch_sts_apply(const float* c, int N, int gamma, const double* t, float* out, cudaStream_t s);
cudaError_t launch_schedule_threshold(const float* c, int R, int gamma, float theta, int mode, int32_t* len,
                                      cudaStream_t s);
cudaError_t launch_schedule(const float* c, const double* sps, int n_sps, int R, int gamma, const int32_t* budget,
                            int32_t* len, double* theta, int32_t* nstar, void* ws, cudaStream_t s);

int num_sms();

// Row length of the tensor-core GRU's bf16 input [s_hi | s_mid | s_lo | W1[x] | h]
// (4r + d values) rounded up to a whole 64-value K block.
__host__ __device__ inline int gru_ldzb(int r, int d) { return (4 * r + d + 63) / 64 * 64; }
int gru_tc_parts(int R, int r, int d);
bool gru_tc_supported(const DraftArgs& a);
cudaError_t launch_gru_tc(DraftArgs& a, int k, cudaStream_t s);

// Launch `kern` on `s`.  With `pdl` set the launch may begin while the
// previous kernel in the stream is still running (programmatic dependent
// launch); such a kernel executes griddepcontrol.wait (pdl_wait) before it
// touches anything that kernel writes or reads.  The first kernel of every
// entry point is launched without it, so work the caller queued before the
// call is complete and visible as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace dspark
