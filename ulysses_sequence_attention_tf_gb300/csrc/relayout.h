// relayout.h -- internal interface between the C-ABI host code and the CUDA kernels.
// Not part of the public ABI (that is include/tf_ulysses.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tfu {

constexpr int kMaxShards = 8;
constexpr int kMaxSlots = 3;      // Q, K, V
#ifndef TFU_CHECKED
#define TFU_CHECKED 0  // 1: block kernels test their accesses against the planned buffers
#endif

constexpr int kThreads = 256;          // threads per CTA
#ifndef TFU_CHUNK_BYTES
#define TFU_CHUNK_BYTES 32768
#endif
constexpr int kChunkBytes = TFU_CHUNK_BYTES;  // payload bytes per work unit of the register kernel
__host__ __device__ constexpr int chunk_vecs(int vec_bytes) { return kChunkBytes / vec_bytes; }

// Block kernel pipeline: rows (of every slot) each lane keeps loaded ahead of the
// one it computes, with and without fused slots.
#ifndef TFU_BLOCK_DEPTH
#define TFU_BLOCK_DEPTH 2
#endif
#ifndef TFU_COPY_BLOCK_DEPTH
#define TFU_COPY_BLOCK_DEPTH 4
#endif
#ifndef TFU_QK_BLOCK_DEPTH
// fused launches without a copied slot (Q/K only): a third row in flight fits the
// registers once the RMSNorm weights sit in shared memory (124, no spill) and
// measured 5304 GB/s against 5158-5163 at depth 2 (depth 4: 5126-5128)
#define TFU_QK_BLOCK_DEPTH 3
#endif
constexpr int kBlockDepth = TFU_BLOCK_DEPTH;
constexpr int kCopyBlockDepth = TFU_COPY_BLOCK_DEPTH;
constexpr int kQkBlockDepth = TFU_QK_BLOCK_DEPTH;

// Unsigned 32-bit division by an invariant divisor as multiply-high, add and
// shift (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, section 4, figure 4.1).  Exact for every n < 2^32.
struct FastDiv {
    uint32_t d, m, s1, s2;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{};
    f.d = d;
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;  // l = ceil(log2 d)
    uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    f.m = uint32_t(m);
    f.s1 = l < 1 ? l : 1;
    f.s2 = l > 1 ? l - 1 : 0;
    return f;
}

__host__ __device__ inline uint32_t fastdiv(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
    uint32_t t = __umulhi(n, f.m);
#else
    uint32_t t = uint32_t((uint64_t(n) * f.m) >> 32);
#endif
    return (t + ((n - t) >> f.s1)) >> f.s2;
}

enum class Dir : int { kScatter = 0, kGather = 1 };
enum class Fused : int { kNone = 0, kBF16 = 1, kFP16 = 2 };

// One grouped launch.  A "slot" is one tensor (V, Q, K in that order when present);
// a "plane" is one (batch b, shard r, slot x, head group g) block of
// S_local * Hl * D elements; a "unit" is one 32 KiB chunk of a plane.
struct RelayoutParams {
    // scatter: src[x][r] = shard r, dst[x][g] = head-group target g
    // gather:  src[x][g] = head-group buffer g, dst[x][r] = shard output r
    const uint8_t* src[kMaxSlots][kMaxShards];
    uint8_t* dst[kMaxSlots][kMaxShards];
    int64_t s_b[kMaxSlots], s_t[kMaxSlots], s_h[kMaxSlots];  // byte strides
    int64_t d_b[kMaxSlots], d_t[kMaxSlots], d_h[kMaxSlots];  // byte strides (a scatter's slots share them)
    const void* weight[kMaxSlots];  // per slot RMSNorm weight [D] (fused slots only)
    const float* table;             // [>= P*S_local][D/2][2] fp32 (fused only)
    float eps;
    uint32_t fused_mask;  // bit x set: slot x gets RMSNorm + RoPE
    uint32_t nx, P, B, Sl, Hl;
    uint32_t vec_bytes;  // bytes each lane moves per access: 32, or 16 when rows/strides/bases are
                         // only 16-byte aligned
    uint32_t vpr;        // vectors per head row = D * esize / vec_bytes
    uint32_t nv;         // vectors per plane = Sl * Hl * vpr
    uint32_t n_planes;   // B * P * nx * P
    uint32_t n_chunks;   // ceil(nv / chunk_vecs(vec_bytes))
    uint32_t n_units;   // n_chunks * n_planes
    FastDiv div_vpr, div_hl, div_planes;
    // shared-memory-staged kernel: units are row ranges of a plane
    uint32_t row_bytes;   // D * esize
    uint32_t rpu;         // rows per unit (tma_rows_per_unit)
    uint32_t plane_rows;  // Sl * Hl
    uint32_t rope_neox;   // fused slots: 0 interleaved pairs (2i, 2i+1), 1 half-split pairs (i, i + D/2)
    uint32_t Hg;          // heads between consecutive head groups on the head-major side (scatter
                          // source, gather destination): Hl, or the whole band when a launch moves
                          // a head chunk of Hl heads out of every band
#if TFU_CHECKED
    // checked builds: one past the last byte each slot's buffers may be accessed
    // at (from the plan's shapes and strides), and the table's; the block kernel
    // tests every row and table access against [base, end) and skips any outside
    const uint8_t* src_end[kMaxSlots][kMaxShards];
    const uint8_t* dst_end[kMaxSlots][kMaxShards];
    const float* table_end;
#endif
};
// Field order is part of the staged kernel's speed: inserting one 4-byte field
// before `nx` (shifting every later field by 4 bytes) measured ~1.3 % slower
// bulk copies on the video-DiT shape.  New fields go at the end.

// Launch `kernel` allowed to overlap the kernel before it in the stream
// (programmatic dependent launch): its CTAs may be scheduled while that kernel's
// last CTAs drain, and wait at grid_dependency_wait() (device_common.cuh) until
// it has completed and its writes are visible, so stream order is kept.  Before
// an operation that is not such a kernel the launch is an ordinary one.
template <typename... Params, typename... Args>
inline cudaError_t launch_overlapped(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                                     cudaStream_t stream, const Args&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Checked builds (TFU_CHECKED=1): the block kernels' bounds status -- nonzero
// once a row or table access of a block kernel fell outside the ranges in
// RelayoutParams (the access was skipped); optionally cleared.  Always 0 in
// other builds.  One word per translation unit: 32-byte and 16-byte forms.
cudaError_t read_block_status(unsigned* out, bool clear);
cudaError_t read_block_status_v16(unsigned* out, bool clear);

// Launch the relayout of every plane in `p` with the register kernel (vector
// width p.vec_bytes); pure relayouts only (fused scatters take the block
// kernel).  Scatter destination rows of a plane are d_h bytes apart.
cudaError_t launch_relayout(const RelayoutParams& p, Dir dir, cudaStream_t stream);

// Launch the shared-memory-staged (bulk-copy) relayout of a pure relayout
// (no fused rows).  Requires rpu > 0; units are counted in rows
// (n_chunks = ceil(plane_rows / rpu), n_units = n_chunks * n_planes).
cudaError_t launch_relayout_staged(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream);

// Launch the scatter over token blocks of all slots together (copied slots
// first, then the fused ones, normalised and rotated in the same pass).
// Requires vpr = D * esize / 32 in {2, 4, 8, 16} (lanes per head row, 32 bytes
// each), vec_bytes == 32 -- or 16 for a fused scatter whose rows are only
// 16-byte aligned -- and units counted in rows of one (b, r, g) block:
// n_planes = B * P * P, rpu = rows per unit, n_chunks = ceil(plane_rows / rpu).
// Destination rows are d_h bytes apart.
cudaError_t launch_blocks(const RelayoutParams& p, Fused fused, cudaStream_t stream);
// The fused scatters of launch_blocks with vec_bytes == 16.
cudaError_t launch_blocks_v16(const RelayoutParams& p, Fused fused, cudaStream_t stream);

// Device status word of the staged kernel: 0, or 1 when a bounded wait for a
// bulk load gave up.  read_staged_status optionally clears it.
cudaError_t read_staged_status(unsigned* out, bool clear);

// Fill table[S][D/2][2] with (cos, sin) of p * inv_freq[i] evaluated in double.
cudaError_t launch_rope_table(float* table, const double* inv_freq_host, int S, int D, cudaStream_t stream);

}  // namespace tfu
