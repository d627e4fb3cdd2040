// verify_static.cu -- dspark_verify_noalloc: verification with library-owned scratch.
//
// Some callers cannot hand the library a workspace: a plugin that is given
// only its input and output tensors, a serving engine whose memory planner
// owns every byte of the device and forbids allocations it did not plan, or a
// latency-critical path that must not pay for (or synchronise on) an
// allocation.  For them this entry point runs the same kernels as
// dspark_verify, with the scratch taken from a fixed array compiled into the
// library instead of from the caller.
//
// The array is a file-scope __device__ object of kNoallocScratchBytes: every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; make that first call before capturing a stream.
// All calls share the one array and each leaves its contents behind: calls
// whose work overlaps on the GPU (different streams, or different host
// threads without ordering) race on it and must be serialised by the caller.
// The status word at the start of the array is cleared by every call.  The
// stream must belong to the current device (the array's address is the
// current device's); a stream of another device is refused.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

constexpr size_t kNoallocScratchBytes = 8u << 20;   // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSPARK_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DSPARK_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return DSPARK_OK;
}
}  // namespace

}  // namespace dspark

using namespace dspark;

extern "C" int dspark_verify_noalloc(const void* P, int p_dtype, const void* U, int u_dtype, const void* W2,
                                     int w_dtype, const int32_t* tokens, const float* q_tok, const double* lse,
                                     const float* code, const int32_t* verify_len, int R, int gamma, int V, int r,
                                     uint64_t seed, const uint32_t* req_ids, float temperature,
                                     int32_t* out_tokens, int32_t* accept_len, int32_t* n_out, float* p_tok,
                                     double* lse_p, void* stream) {
    if (R < 1 || gamma < 1 || gamma > 64 || V < 2 || V > (1 << 20) || r < 1 || r > 1024) return DSPARK_ERR_SHAPE;
    if (verify_workspace_bytes(R, gamma, V, r) > kNoallocScratchBytes) return DSPARK_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scratch address belongs to the current device: a stream of another
    // device would hand its kernels memory they cannot address
    int dev = 0, sdev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess) {
        (void)cudaGetLastError();
        return DSPARK_ERR_CUDA;
    }
    if (sdev != dev) return DSPARK_ERR_INVALID_ARG;
    void* ws = nullptr;
    int st = noalloc_scratch(&ws);
    if (st) return st;
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), s) != cudaSuccess) return DSPARK_ERR_CUDA;
    return dspark_verify(P, p_dtype, U, u_dtype, W2, w_dtype, tokens, q_tok, lse, code, verify_len, R, gamma, V, r,
                         seed, req_ids, temperature, out_tokens, accept_len, n_out, p_tok, lse_p, ws,
                         kNoallocScratchBytes, stream);
}
