// api.cu -- the C ABI of libdspark.so: argument checks, workspace carve-up and
// kernel dispatch.  See include/dspark.h for the contract of each entry point.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

// SM count of the current device, looked up once per device (a process may
// drive several GPUs; each call sizes its grids for the device it runs on).
int num_sms() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
    if (dev < kMaxDevices) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
    if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// True for device memory of the current device.  The arrays the kernels
// address through tensor maps (U, W2, Wgco) must be: the tensor-core kernels
// share W2 tiles among the CTAs of a thread-block cluster by multicast, which
// is only defined for this GPU's own memory, so a peer device's buffer, a
// mapped host buffer or managed memory is refused before anything is enqueued.
static bool on_current_device(const void* p) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

static bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
// U, P (and its staging copy), W2 and Wgco are read with 16-byte loads and
// tensor-map copies: they must start on a 16-byte boundary
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool dtype_ok(int dt) { return dt == DSPARK_F32 || dt == DSPARK_BF16; }

static int check_vocab(int V, int dt) {
    if (V < 2 || V > (1 << 20)) return DSPARK_ERR_SHAPE;
    if (dt == DSPARK_F32 && V % 4) return DSPARK_ERR_SHAPE;
    if (dt == DSPARK_BF16 && V % 8) return DSPARK_ERR_SHAPE;
    return DSPARK_OK;
}

static int check_common(int R, int gamma, int V, int r, float T, int u_dtype, int w_dtype) {
    if (!dtype_ok(u_dtype) || !dtype_ok(w_dtype)) return DSPARK_ERR_UNSUPPORTED_DTYPE;
    if (R < 1 || gamma < 1 || gamma > 64 || r < 1 || r > 1024) return DSPARK_ERR_SHAPE;
    if (!(T >= 0.f) || !std::isfinite(T)) return DSPARK_ERR_INVALID_ARG;
    int st = check_vocab(V, u_dtype);
    if (st) return st;
    return check_vocab(V, w_dtype);
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

}  // namespace dspark

using namespace dspark;

extern "C" {

const char* dspark_strerror(int status) {
    switch (status) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID_ARG: return "invalid argument";
        case DSPARK_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case DSPARK_ERR_SHAPE: return "unsupported sizes";
        case DSPARK_ERR_CUDA: return "CUDA runtime error";
        case DSPARK_ERR_TIMEOUT: return "bounded device wait ran out";
        case DSPARK_ERR_BAD_TOKEN: return "token id outside [0, V)";
        case DSPARK_ERR_UNIMPLEMENTED: return "not implemented";
        case DSPARK_ERR_WORKSPACE: return "workspace null, misaligned or too small";
        default: return "unknown status";
    }
}

const char* dspark_version(void) { return "dspark-gb300 0.1 (sm_103a)"; }

int dspark_host_pointer(const void* host, void** device) {
    if (!host || !device) return DSPARK_ERR_INVALID_ARG;
    *device = nullptr;
    if (cudaHostGetDevicePointer(device, const_cast<void*>(host), 0) != cudaSuccess) {
        (void)cudaGetLastError();
        *device = nullptr;
        return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}

int dspark_workspace_status(void* ws, void* stream) {
    if (!ws) return DSPARK_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (word) {
        if (cudaMemsetAsync(ws, 0, sizeof word, s) != cudaSuccess) return DSPARK_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
    }
    if (word & kStatBadToken) return DSPARK_ERR_BAD_TOKEN;
    if (word & kStatTimeout) return DSPARK_ERR_TIMEOUT;
    return DSPARK_OK;
}

int dspark_workspace_set_wait(void* ws, uint64_t limit_cycles, int test_withhold, void* stream) {
    if (!ws || !aligned256(ws) || (test_withhold != 0 && test_withhold != 1)) return DSPARK_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // header bytes [4, 20): test_withhold (u32), wait_limit (u64), the marker (u32)
    struct {
        uint32_t withhold;
        uint32_t limit_lo, limit_hi;
        uint32_t marker;
    } h = {(uint32_t)test_withhold, (uint32_t)limit_cycles, (uint32_t)(limit_cycles >> 32), kWaitMarker};
    static_assert(sizeof(h) == 16, "four words");
    if (cudaMemcpyAsync(static_cast<char*>(ws) + 4, &h, sizeof h, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

size_t dspark_draft_workspace_size(int R, int gamma, int V, int r, int d) {
    if (R < 1 || gamma < 1 || gamma > 64 || V < 2 || V > (1 << 20) || r < 1 || r > 1024 || d < 0) return 0;
    return draft_workspace_bytes(R, gamma, V, r, d);
}

// Attach the confidence head's arguments (conf may be null: head off).
static int attach_conf(DraftArgs& a, bool rnn, const dspark_conf_t* conf) {
    if (!conf) return DSPARK_OK;
    if (!conf->w || !conf->c) return DSPARK_ERR_INVALID_ARG;
    if (conf->H) {
        if (conf->d < 0 || conf->d > 16384) return DSPARK_ERR_SHAPE;
        a.Hc = conf->H;
        a.dc = conf->d;
    } else if (rnn) {
        a.Hc = a.H;   // the RNN head's own hidden states
        a.dc = a.d;
    } else {
        if (conf->d != 0) return DSPARK_ERR_INVALID_ARG;
        a.Hc = nullptr;
        a.dc = 0;
    }
    a.wc = conf->w;
    a.conf = conf->c;
    a.tc = conf->t;
    return DSPARK_OK;
}

static int draft_entry(DraftArgs& a, bool rnn, size_t ws_bytes, void* stream) {
    int st = check_common(a.R, a.gamma, a.V, a.r, a.T, a.u_dtype, a.w_dtype);
    if (st) return st;
    if (!a.U || !a.anchor || !a.W1 || !a.W2 || !a.tokens || !a.q_tok || !a.lse || !a.code)
        return DSPARK_ERR_INVALID_ARG;
    if (rnn && (!a.Wgco || !a.H || a.d < 1 || a.d > 16384)) return rnn && (a.d < 1 || a.d > 16384)
                                                                      ? DSPARK_ERR_SHAPE
                                                                      : DSPARK_ERR_INVALID_ARG;
    if (!aligned16(a.U) || !aligned16(a.W2) || (rnn && !aligned16(a.Wgco))) return DSPARK_ERR_INVALID_ARG;
    if (!on_current_device(a.U) || !on_current_device(a.W2) || (rnn && !on_current_device(a.Wgco)))
        return DSPARK_ERR_INVALID_ARG;
    if (!a.ws || !aligned256(a.ws)) return DSPARK_ERR_WORKSPACE;
    st = draft_carve(a, ws_bytes);
    if (st) return st;
    return cuda_status(launch_draft(a, rnn, static_cast<cudaStream_t>(stream)));
}

int dspark_draft_markov_conf(const void* U, int u_dtype, const int32_t* anchor, const void* W1, const void* W2,
                             int w_dtype, int R, int gamma, int V, int r, uint64_t seed, const uint32_t* req_ids,
                             float temperature, int32_t* tokens, float* q_tok, double* lse, float* code,
                             const dspark_conf_t* conf, void* ws, size_t ws_bytes, void* stream) {
    DraftArgs a;
    std::memset(&a, 0, sizeof a);
    a.U = U; a.u_dtype = u_dtype; a.anchor = anchor; a.W1 = W1; a.W2 = W2; a.w_dtype = w_dtype;
    a.R = R; a.gamma = gamma; a.V = V; a.r = r; a.d = 0; a.seed = seed; a.req_ids = req_ids;
    a.T = temperature; a.tokens = tokens; a.q_tok = q_tok; a.lse = lse; a.code = code; a.ws = ws;
    const int st = attach_conf(a, false, conf);
    if (st) return st;
    return draft_entry(a, false, ws_bytes, stream);
}

int dspark_draft_markov(const void* U, int u_dtype, const int32_t* anchor, const void* W1, const void* W2,
                        int w_dtype, int R, int gamma, int V, int r, uint64_t seed, const uint32_t* req_ids,
                        float temperature, int32_t* tokens, float* q_tok, double* lse, float* code, void* ws,
                        size_t ws_bytes, void* stream) {
    return dspark_draft_markov_conf(U, u_dtype, anchor, W1, W2, w_dtype, R, gamma, V, r, seed, req_ids, temperature,
                                    tokens, q_tok, lse, code, nullptr, ws, ws_bytes, stream);
}

int dspark_draft_rnn_conf(const void* U, int u_dtype, const int32_t* anchor, const void* W1, const void* W2,
                          const void* Wgco, int w_dtype, const void* H, int d, int R, int gamma, int V, int r,
                          uint64_t seed, const uint32_t* req_ids, float temperature, int32_t* tokens, float* q_tok,
                          double* lse, float* code, float* state_out, const dspark_conf_t* conf, void* ws,
                          size_t ws_bytes, void* stream) {
    DraftArgs a;
    std::memset(&a, 0, sizeof a);
    a.U = U; a.u_dtype = u_dtype; a.anchor = anchor; a.W1 = W1; a.W2 = W2; a.Wgco = Wgco; a.H = H;
    a.w_dtype = w_dtype; a.R = R; a.gamma = gamma; a.V = V; a.r = r; a.d = d; a.seed = seed;
    a.req_ids = req_ids; a.T = temperature; a.tokens = tokens; a.q_tok = q_tok; a.lse = lse; a.code = code;
    a.state_out = state_out; a.ws = ws;
    const int st = attach_conf(a, true, conf);
    if (st) return st;
    return draft_entry(a, true, ws_bytes, stream);
}

int dspark_draft_rnn(const void* U, int u_dtype, const int32_t* anchor, const void* W1, const void* W2,
                     const void* Wgco, int w_dtype, const void* H, int d, int R, int gamma, int V, int r,
                     uint64_t seed, const uint32_t* req_ids, float temperature, int32_t* tokens, float* q_tok,
                     double* lse, float* code, float* state_out, void* ws, size_t ws_bytes, void* stream) {
    return dspark_draft_rnn_conf(U, u_dtype, anchor, W1, W2, Wgco, w_dtype, H, d, R, gamma, V, r, seed, req_ids,
                                 temperature, tokens, q_tok, lse, code, state_out, nullptr, ws, ws_bytes, stream);
}

size_t dspark_verify_workspace_size(int R, int gamma, int V, int r) {
    if (R < 1 || gamma < 1 || gamma > 64 || V < 2 || V > (1 << 20) || r < 1 || r > 1024) return 0;
    return verify_workspace_bytes(R, gamma, V, r);
}

int dspark_verify_staged(const void* P, int p_dtype, const void* U, int u_dtype, const void* W2, int w_dtype,
                         const int32_t* tokens, const float* q_tok, const double* lse, const float* code,
                         const int32_t* verify_len, int R, int gamma, int V, int r, uint64_t seed,
                         const uint32_t* req_ids, float temperature, int32_t* out_tokens, int32_t* accept_len,
                         int32_t* n_out, float* p_tok, double* lse_p, void* p_stage, void* ws, size_t ws_bytes,
                         void* stream) {
    if (!dtype_ok(p_dtype)) return DSPARK_ERR_UNSUPPORTED_DTYPE;
    int st = check_common(R, gamma, V, r, temperature, u_dtype, w_dtype);
    if (st) return st;
    st = check_vocab(V, p_dtype);
    if (st) return st;
    if (!P || !tokens || !out_tokens || !accept_len || !n_out) return DSPARK_ERR_INVALID_ARG;
    if (temperature > 0.f && (!U || !W2 || !q_tok || !lse || !code)) return DSPARK_ERR_INVALID_ARG;
    if (!aligned16(P) || (p_stage && !aligned16(p_stage))) return DSPARK_ERR_INVALID_ARG;
    if (temperature > 0.f && (!aligned16(U) || !aligned16(W2))) return DSPARK_ERR_INVALID_ARG;
    if (temperature > 0.f && (!on_current_device(U) || !on_current_device(W2))) return DSPARK_ERR_INVALID_ARG;
    if (!ws || !aligned256(ws)) return DSPARK_ERR_WORKSPACE;
    VerifyArgs a;
    std::memset(&a, 0, sizeof a);
    a.P = P; a.p_dtype = p_dtype; a.U = U; a.u_dtype = u_dtype; a.W2 = W2; a.w_dtype = w_dtype;
    a.tokens = tokens; a.q_tok = q_tok; a.lse = lse; a.code = code; a.verify_len = verify_len;
    a.R = R; a.gamma = gamma; a.V = V; a.r = r; a.seed = seed; a.req_ids = req_ids; a.T = temperature;
    a.out_tokens = out_tokens; a.accept_len = accept_len; a.n_out = n_out; a.p_tok = p_tok; a.lse_p = lse_p;
    a.ws = ws;
    a.P_stage = p_stage;
    a.Pv = p_stage ? p_stage : P;
    st = verify_carve(a, ws_bytes);
    if (st) return st;
    return cuda_status(launch_verify(a, static_cast<cudaStream_t>(stream)));
}

int dspark_verify(const void* P, int p_dtype, const void* U, int u_dtype, const void* W2, int w_dtype,
                  const int32_t* tokens, const float* q_tok, const double* lse, const float* code,
                  const int32_t* verify_len, int R, int gamma, int V, int r, uint64_t seed,
                  const uint32_t* req_ids, float temperature, int32_t* out_tokens, int32_t* accept_len,
                  int32_t* n_out, float* p_tok, double* lse_p, void* ws, size_t ws_bytes, void* stream) {
    return dspark_verify_staged(P, p_dtype, U, u_dtype, W2, w_dtype, tokens, q_tok, lse, code, verify_len, R, gamma,
                                V, r, seed, req_ids, temperature, out_tokens, accept_len, n_out, p_tok, lse_p,
                                nullptr, ws, ws_bytes, stream);
}

size_t dspark_schedule_workspace_size(int R, int gamma) {
    if (R < 1 || gamma < 1 || gamma > 64 || (long long)R * gamma > 8192) return 0;
    return sizeof(WsHeader);
}

int dspark_schedule(const float* c, const double* sps, int n_sps, int R, int gamma, int32_t* verify_len,
                    double* theta, int32_t* n_star, void* ws, size_t ws_bytes, void* stream) {
    if (R < 1 || gamma < 1 || gamma > 64 || (long long)R * gamma > 8192 || n_sps < 1) return DSPARK_ERR_SHAPE;
    if (!c || !sps || !verify_len || !theta || !n_star) return DSPARK_ERR_INVALID_ARG;
    if (!ws || !aligned256(ws)) return DSPARK_ERR_WORKSPACE;
    if (ws_bytes < sizeof(WsHeader)) return DSPARK_ERR_WORKSPACE;
    return cuda_status(launch_schedule(c, sps, n_sps, R, gamma, nullptr, verify_len, theta, n_star, ws,
                                       static_cast<cudaStream_t>(stream)));
}

int dspark_schedule_async(const float* c, const double* sps, int n_sps, int R, int gamma, const int32_t* budget,
                          int32_t* verify_len, double* theta, int32_t* n_star, void* ws, size_t ws_bytes,
                          void* stream) {
    if (R < 1 || gamma < 1 || gamma > 64 || (long long)R * gamma > 8192 || n_sps < 1) return DSPARK_ERR_SHAPE;
    if (!c || !sps || !budget || !verify_len || !theta || !n_star) return DSPARK_ERR_INVALID_ARG;
    if (!ws || !aligned256(ws)) return DSPARK_ERR_WORKSPACE;
    if (ws_bytes < sizeof(WsHeader)) return DSPARK_ERR_WORKSPACE;
    return cuda_status(launch_schedule(c, sps, n_sps, R, gamma, budget, verify_len, theta, n_star, ws,
                                       static_cast<cudaStream_t>(stream)));
}

size_t dspark_sts_workspace_size(int N, int gamma, int G, int M) {
    if (N < 1 || N > (1 << 24) || gamma < 1 || gamma > 64 || G < 1 || G > 4096 || M < 1 || M > 32) return 0;
    return sts_workspace_bytes(N, gamma, G, M);
}

int dspark_sts_fit(const float* c, const int32_t* accept_len, int N, int gamma, const double* grid, int G, int M,
                   double* t_out, int32_t* g_out, double* ece_out, double* gap_out, void* ws, size_t ws_bytes,
                   void* stream) {
    if (N < 1 || N > (1 << 24) || gamma < 1 || gamma > 64 || G < 1 || G > 4096 || M < 1 || M > 32)
        return DSPARK_ERR_SHAPE;
    if (!c || !accept_len || !grid || !t_out || !g_out || !ece_out || !gap_out) return DSPARK_ERR_INVALID_ARG;
    if (!ws || !aligned256(ws) || ws_bytes < sts_workspace_bytes(N, gamma, G, M)) return DSPARK_ERR_WORKSPACE;
    return cuda_status(launch_sts_fit(c, accept_len, N, gamma, grid, G, M, t_out, g_out, ece_out, gap_out, ws,
                                      static_cast<cudaStream_t>(stream)));
}

int dspark_sts_apply(const float* c, int N, int gamma, const double* t, float* out, void* stream) {
    if (N < 1 || gamma < 1 || gamma > 64 || (long long)N * gamma > (1ll << 31)) return DSPARK_ERR_SHAPE;
    if (!c || !t || !out) return DSPARK_ERR_INVALID_ARG;
    return cuda_status(launch_sts_apply(c, N, gamma, t, out, static_cast<cudaStream_t>(stream)));
}

int dspark_schedule_threshold(const float* c, int R, int gamma, float theta, int mode, int32_t* verify_len,
                              void* stream) {
    if (R < 1 || gamma < 1 || gamma > 64) return DSPARK_ERR_SHAPE;
    if (!c || !verify_len || (mode != 0 && mode != 1)) return DSPARK_ERR_INVALID_ARG;
    return cuda_status(launch_schedule_threshold(c, R, gamma, theta, mode, verify_len,
                                                 static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
