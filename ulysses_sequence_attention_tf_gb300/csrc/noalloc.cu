// noalloc.cu -- the fixed device scratch behind tf_ulysses_scatter_qkv_noalloc.
//
// The fp32 cos/sin table that the fused scatter reads lives here, in a
// file-scope device array, instead of in memory the library allocates.  Every
// GPU that loads the library holds these 16 MiB until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current.
#include <mutex>

#include "noalloc.h"

namespace tfu {

static __device__ __align__(256) float g_noalloc_table[kNoAllocTableFloats];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
float* g_addr[kMaxDevices] = {};
}  // namespace

cudaError_t noalloc_table_address(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_addr_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_table);
        if (e != cudaSuccess) return e;
        g_addr[dev] = static_cast<float*>(p);
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace tfu
