// rng.cu -- the device's Philox4x32-10 block function behind the C ABI, so that
// known-answer vectors of the generator (Salmon et al., "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11) can check the copy every kernel draws
// from (common.cuh), not only its effect on sampled tokens.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace {

__global__ void __launch_bounds__(256) philox_blocks(const uint4* ctr, const uint2* key, uint4* out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint2 k = key[i];
    out[i] = philox4x32_10(ctr[i], PhiloxKey{k.x, k.y});
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" int dspark_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int n, void* stream) {
    if (n < 1) return DSPARK_ERR_SHAPE;
    if (!ctr || !key || !out) return DSPARK_ERR_INVALID_ARG;
    // uint4 / uint2 loads: the arrays must be 16- and 8-byte aligned
    if ((reinterpret_cast<uintptr_t>(ctr) & 15) || (reinterpret_cast<uintptr_t>(out) & 15) ||
        (reinterpret_cast<uintptr_t>(key) & 7))
        return DSPARK_ERR_INVALID_ARG;
    const int blocks = (n + 255) / 256;
    cudaError_t e = launch_kernel(philox_blocks, dim3(blocks), dim3(256), 0, static_cast<cudaStream_t>(stream), false,
                                  reinterpret_cast<const uint4*>(ctr), reinterpret_cast<const uint2*>(key),
                                  reinterpret_cast<uint4*>(out), n);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
