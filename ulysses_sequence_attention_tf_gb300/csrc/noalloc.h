// noalloc.h -- internal: the fixed device scratch of tf_ulysses_scatter_qkv_noalloc.
#pragma once

#include <cstddef>

#include <cuda_runtime.h>

namespace tfu {

// Capacity of the fixed cos/sin table scratch, in floats: S * D <= 4 Mi
// (16 MiB), enough for S = 32760 tokens at D = 128.
constexpr size_t kNoAllocTableFloats = size_t(4) << 20;

// The fixed scratch of the current device holding the (cos, sin) table of
// (theta, >= S rows, D) in stream order on `stream`; *out receives its device
// address.  The first call on a device sets the device up (looks up the array's
// address with cudaGetSymbolAddress and creates the event that marks the end of
// each build).  The table is rebuilt on `stream` only when the array does not
// already hold (theta, >= S rows, D) (*built = true); otherwise `stream` waits on
// the end of the last build (*built = false).  capturing: `stream` is capturing
// a graph (the event is then recorded and waited on as an external node).
// S * D must not exceed kNoAllocTableFloats.
cudaError_t noalloc_table(float theta, int S, int D, cudaStream_t stream, bool capturing, float** out, bool* built);

}  // namespace tfu
