// verify_static.cu -- dspark_verify with its scratch in a static device array.
//
// Some callers cannot hand the library a workspace: a plugin running inside a
// serving engine whose device memory all belongs to the engine's own pool (an
// extra cudaMalloc there is not allowed -- it can synchronise the device and
// escapes the engine's memory accounting), or code that has no spare buffer
// to pass down.  This entry point needs no workspace and allocates nothing:
// its scratch is the array below, compiled into the library.  Every GPU that
// loads the library holds the array until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it; the verify prologue clears the counters, flags and
// per-request rows at the start of each call, so nothing has to be zeroed
// beforehand.  Two calls
// whose kernels overlap on the GPU (for example on two streams) use the same
// array and race: serialise them.
#include <mutex>

#include "dspark.h"
#include "kernels.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The scratch area itself.
__device__ __align__(256) unsigned char g_verify_scratch[DSPARK_VERIFY_STATIC_SCRATCH_BYTES];

// Device addresses of the array, looked up once per device.  In host code the
// array's name only stands in for the device object, so the address has to
// come from cudaGetSymbolAddress with the device current.  The address kept
// here belongs to the device's primary context; after cudaDeviceReset the
// module is loaded anew (possibly elsewhere), which is why the header asks
// callers not to use this entry point across a reset.
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DSPARK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return DSPARK_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DSPARK_OK;
}

}  // namespace

extern "C" int dspark_verify_static_scratch(const float* target_logits, const int32_t* cu_seqlens,
                                            const int32_t* draft_tokens, const float* q_logits,
                                            const float* q_lse, const float* q_tok,
                                            const uint64_t* seeds, uint32_t cycle, float temperature,
                                            int R, int gamma, int V, int max_rows,
                                            int32_t* n_accepted, int32_t* out_tokens, float* p_tok,
                                            int32_t* dev_status, dspark_stream_t stream) {
    const size_t need = dspark_workspace_size(DSPARK_OP_VERIFY, R, gamma, V, 0, max_rows, 0, 0);
    if (need == 0) return DSPARK_ERR_INVALID_ARG;
    if (need > (size_t)DSPARK_VERIFY_STATIC_SCRATCH_BYTES) return DSPARK_ERR_CAPACITY;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != DSPARK_OK) return st;
    return dspark_verify(target_logits, cu_seqlens, draft_tokens, q_logits, q_lse, q_tok, seeds, cycle,
                         temperature, R, gamma, V, max_rows, n_accepted, out_tokens, p_tok, scratch,
                         (size_t)DSPARK_VERIFY_STATIC_SCRATCH_BYTES, dev_status, stream);
}
