// block_kernels.cu -- the block kernel (block_kernel.cuh) for rows whose every
// address is 32-byte aligned: fused scatters and the copy scatters the planner
// gives it.  Fused scatters of rows only 16-byte aligned go to
// block_kernels_v16.cu (a separate translation unit, so the two sets of
// instantiations compile in parallel).
#include "block_kernel.cuh"

namespace tfu {

cudaError_t launch_blocks(const RelayoutParams& p, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.rpu == 0) return cudaErrorInvalidValue;
    if (p.vec_bytes == 16) return fused == Fused::kNone ? cudaErrorInvalidValue : launch_blocks_v16(p, fused, stream);
    if (p.vec_bytes != 32) return cudaErrorInvalidValue;
    switch (fused) {
        case Fused::kNone:
            if (p.fused_mask != 0) return cudaErrorInvalidValue;
            switch (p.nx) {
                case 1: return launch_block_lanes<Fused::kNone, 1, 0, false, false>(p, stream);
                case 2: return launch_block_lanes<Fused::kNone, 2, 0, false, false>(p, stream);
                case 3: return launch_block_lanes<Fused::kNone, 3, 0, false, false>(p, stream);
                default: return cudaErrorInvalidValue;
            }
        case Fused::kBF16: return launch_block_style<Fused::kBF16, false>(p, stream);
        case Fused::kFP16: return launch_block_style<Fused::kFP16, false>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t read_block_status(unsigned* out, bool clear) { return read_this_block_status(out, clear); }

}  // namespace tfu
