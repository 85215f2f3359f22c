// noalloc.h -- internal: the fixed device scratch of tf_ulysses_scatter_qkv_noalloc.
#pragma once

#include <cstddef>

#include <cuda_runtime.h>

namespace tfu {

// Capacity of the fixed cos/sin table scratch, in floats: S * D <= 4 Mi
// (16 MiB), enough for S = 32760 tokens at D = 128.
constexpr size_t kNoAllocTableFloats = size_t(4) << 20;

// Device address of the fixed scratch on the current device.  The first call on
// a device looks it up (cudaGetSymbolAddress) and caches it; later calls only
// read the cache.
cudaError_t noalloc_table_address(float** out);

}  // namespace tfu
