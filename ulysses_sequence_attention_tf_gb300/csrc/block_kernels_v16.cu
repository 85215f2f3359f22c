// block_kernels_v16.cu -- the block kernel (block_kernel.cuh) for fused scatters
// whose sources or targets are only 16-byte aligned: each lane still holds 32
// bytes of a head row, moved as two 16-byte vectors.
#include "block_kernel.cuh"

namespace tfu {

cudaError_t launch_blocks_v16(const RelayoutParams& p, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.vec_bytes != 16 || p.rpu == 0) return cudaErrorInvalidValue;
    switch (fused) {
        case Fused::kBF16: return launch_block_style<Fused::kBF16, true>(p, stream);
        case Fused::kFP16: return launch_block_style<Fused::kFP16, true>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_block_status_v16(unsigned* out, bool clear) { return read_this_block_status(out, clear); }

}  // namespace tfu
