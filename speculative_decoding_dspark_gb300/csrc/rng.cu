// rng.cu -- batch evaluation of the device Philox4x32-10 (common.cuh).
#include "kernels.cuh"

namespace dspark {
namespace {

__global__ void philox_batch_kernel(const uint4* ctr, const uint64_t* keys, int n, uint4* out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint64_t k = keys[i];
    out[i] = philox4x32_10(ctr[i], (uint32_t)(k & 0xFFFFFFFFu), (uint32_t)(k >> 32));
}

}  // namespace

cudaError_t launch_philox_batch(const uint32_t* ctr, const uint64_t* keys, int n, uint32_t* out,
                                cudaStream_t stream) {
    if (n > 0)
        philox_batch_kernel<<<(n + 255) / 256, 256, 0, stream>>>(
            reinterpret_cast<const uint4*>(ctr), keys, n, reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace dspark
