// noalloc.cu -- a Dion step whose scratch memory is a fixed array inside
// libdion, for callers that cannot allocate device memory themselves.
//
// The scratch is one file-scope __device__ array.  Every GPU that loads the
// library holds it (DION_STATIC_SCRATCH_BYTES) until the process exits.  Host
// code must not pass the array's name to a kernel: on the host that name is a
// stand-in, not a device address.  The device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made while it is current, and cached.
#include "internal.h"

namespace dion {
namespace {

constexpr size_t kStaticScratch = (size_t)DION_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratch];

void* g_scratch_addr[kMaxDevices];   // device address of g_static_scratch, per device

}  // namespace
}  // namespace dion

using namespace dion;

extern "C" dion_status dion_step_batched_static(int batch, int m, int n, int r, dion_dtype dt, void* X, const void* G,
                                                float* M, float* Q, float mu, float lr, float weight_decay,
                                                void* cuda_stream)
{
    size_t need = 0;
    const dion_status sz = dion_workspace_size(batch, m, n, r, dt, &need);
    if (sz != DION_OK) return sz;
    if (!X || !G || !M || !Q) return DION_ERR_INVALID_ARG;
    if (((uintptr_t)X | (uintptr_t)G | (uintptr_t)M | (uintptr_t)Q) & 15u) return DION_ERR_INVALID_ARG;
    if (need > kStaticScratch) return DION_ERR_WORKSPACE;   // shape too large for the fixed scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DION_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DION_ERR_UNSUPPORTED;
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return DION_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    // The same step as dion_step_batched, with the fixed array as its workspace.
    return dion_step_batched(batch, m, n, r, dt, X, G, M, Q, mu, lr, weight_decay, g_scratch_addr[dev], kStaticScratch,
                             cuda_stream);
}
