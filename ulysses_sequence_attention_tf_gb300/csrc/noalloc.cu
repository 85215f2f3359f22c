// noalloc.cu -- the fixed device scratch behind tf_ulysses_scatter_qkv_noalloc.
//
// The fp32 cos/sin table that the fused scatter reads lives here, in a
// file-scope device array, instead of in memory the library allocates.  Every
// GPU that loads the library holds these 16 MiB until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current.  The array keeps the last table built into it; a call whose
// (theta, rows, D) it already holds uses it as it is.
#include <cmath>
#include <cstring>
#include <mutex>

#include "noalloc.h"
#include "relayout.h"

namespace tfu {

static __device__ __align__(256) float g_noalloc_table[kNoAllocTableFloats];

namespace {
constexpr int kMaxDevices = 64;

struct DeviceScratch {
    float* ptr = nullptr;            // device address of g_noalloc_table on this device
    cudaEvent_t built = nullptr;     // recorded after each build
    bool held = false;               // the array holds the table of (theta, S rows, D) below
    float theta = 0.f;
    int S = 0, D = 0;
};
std::mutex g_scratch_mu;
DeviceScratch g_scratch[kMaxDevices];
}  // namespace

cudaError_t noalloc_table(float theta, int S, int D, cudaStream_t stream, bool capturing, float** out, bool* built) {
    *built = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    DeviceScratch& d = g_scratch[dev];
    if (d.ptr == nullptr) {  // set-up, once per device
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_table);
        if (e != cudaSuccess) return e;
        e = cudaEventCreateWithFlags(&d.built, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        d.ptr = static_cast<float*>(p);
    }
    *out = d.ptr;
    if (d.held && d.D == D && d.S >= S && std::memcmp(&d.theta, &theta, sizeof theta) == 0)
        return cudaStreamWaitEvent(stream, d.built, capturing ? cudaEventWaitExternal : 0);
    // frequencies of the pairs, theta^(-2i/D), in double on the host (D <= 256)
    double inv_freq[128];
    for (int i = 0; i < D / 2; ++i) inv_freq[i] = std::pow(double(theta), -2.0 * i / D);
    d.held = false;
    e = launch_rope_table(d.ptr, inv_freq, S, D, stream);
    if (e != cudaSuccess) return e;
    e = capturing ? cudaEventRecordWithFlags(d.built, stream, cudaEventRecordExternal) : cudaEventRecord(d.built, stream);
    if (e != cudaSuccess) return e;
    d.held = true;
    d.theta = theta;
    d.S = S;
    d.D = D;
    *built = S > 0;
    return cudaSuccess;
}

}  // namespace tfu
