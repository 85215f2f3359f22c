// relayout_kernels.cu -- sm_103a register kernel of the pure Ulysses
// sequence<->head relayout (the cases the block and bulk-copy kernels do not
// take), and the builder of the resident RoPE table.
//
// What is computed (TeleFuser docs, "Communication Architecture", section
// "Sequence Parallel Communication / Ulysses"; head bands and rank-order
// concatenation as in flashinfer PR #6332, "Assumptions / Exchange algorithm"):
//   scatter:  T_g[b, r*Sl + t, h, :] = S_r[b, t, g*Hl + h, :]
//   gather:   O_r[b, t, g*Hl + h, :] = A_g[b, r*Sl + t, h, :]
// as bit copies.
//
// Design (HBM-bound data movement; no tensor cores):
//  * One grouped launch per call.  Work is split into units of 32 KiB of one
//    plane = (batch b, shard r, tensor slot x, head group g).  Units are ordered
//    chunk-major with g innermost, so CTAs running at the same time read whole
//    source token rows (all head groups) and write the P head groups of one
//    token block.
//  * A persistent grid (SM count x resident CTAs) walks the units.  Each lane
//    moves 32-byte vectors (16-byte when rows, strides or bases are only 16-byte
//    aligned) and issues all of its loads of a batch before any store.  Loads
//    skip L1 allocation (read once); stores are evict-first (not re-read here).
#include "device_common.cuh"
#include "relayout.h"

namespace tfu {
namespace {

using namespace dev;

int device_sms() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

// vector v of a plane -> (token t, head h, vector-in-row dv) -> byte offset
template <int VW>
__device__ __forceinline__ int64_t vec_offset(const RelayoutParams& p, uint32_t v, int64_t st, int64_t sh) {
    const uint32_t row = fastdiv(v, p.div_vpr);
    const uint32_t dv = v - row * p.vpr;
    const uint32_t t = fastdiv(row, p.div_hl);
    const uint32_t h = row - t * p.Hl;
    return int64_t(t) * st + int64_t(h) * sh + int64_t(dv) * VW;
}

// Destination offset of vector v of a plane: row (t, h) at t*dt + h*dh on
// either side (scatter targets may be the fused receive layout or a head chunk
// of wider targets).
template <Dir kDir, int VW>
__device__ __forceinline__ int64_t dst_offset(const RelayoutParams& p, const Plane& pl, uint32_t v) {
    return vec_offset<VW>(p, v, pl.dt, pl.dh);
}

template <Dir kDir, int VW, int VB>
__device__ __forceinline__ void copy_range(const RelayoutParams& p, const Plane& pl, uint32_t v0, uint32_t v1) {
#pragma unroll 1
    for (uint32_t base = v0; base < v1; base += kThreads * VB) {
        Vec<VW> buf[VB];
#pragma unroll
        for (int i = 0; i < VB; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            if (v < v1) buf[i] = ld_stream<VW>(pl.src + vec_offset<VW>(p, v, pl.st, pl.sh));
        }
#pragma unroll
        for (int i = 0; i < VB; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            if (v < v1) st_stream<VW>(pl.dst + dst_offset<kDir, VW>(p, pl, v), buf[i]);
        }
    }
}

// Tuning constants (compile-time; overridable with -D for measurement sweeps).
// TFU_COPY_MIN_BLOCKS: resident 256-thread CTAs per SM the register budget is
// sized for.  TFU_COPY_BATCH: 32-byte vectors each lane loads before storing
// (twice as many 16-byte vectors).
#ifndef TFU_COPY_MIN_BLOCKS
#define TFU_COPY_MIN_BLOCKS 4
#endif
#ifndef TFU_COPY_BATCH
#define TFU_COPY_BATCH 4
#endif

template <int VW>
__host__ __device__ constexpr int copy_batch() {
    return VW == 32 ? TFU_COPY_BATCH : 2 * TFU_COPY_BATCH;
}

template <Dir kDir, int VW>
__global__ void __launch_bounds__(kThreads, TFU_COPY_MIN_BLOCKS) relayout_kernel(const __grid_constant__ RelayoutParams p) {
    constexpr uint32_t kChunk = uint32_t(chunk_vecs(VW));
    grid_dependency_wait();
#pragma unroll 1
    for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const uint32_t c = fastdiv(u, p.div_planes);
        const uint32_t q = u - c * p.n_planes;
        const Plane pl = decode_plane<kDir>(p, q);
        const uint32_t v0 = c * kChunk;
        copy_range<kDir, VW, copy_batch<VW>()>(p, pl, v0, min(v0 + kChunk, p.nv));
    }
}

struct RopeTableParams {
    double inv_freq[128];
    float* out;
    int S, half;
};

__global__ void __launch_bounds__(256) rope_table_kernel(const __grid_constant__ RopeTableParams p) {
    grid_dependency_wait();
    const int64_t n = int64_t(p.S) * p.half;
    for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < n; idx += int64_t(gridDim.x) * blockDim.x) {
        const int64_t pos = idx / p.half;
        const int i = int(idx - pos * p.half);
        const double angle = double(pos) * p.inv_freq[i];
        double s, c;
        sincos(angle, &s, &c);  // one argument reduction for both
        reinterpret_cast<float2*>(p.out)[idx] = make_float2(__double2float_rn(c), __double2float_rn(s));
    }
}

template <Dir kDir, int VW>
cudaError_t launch_one(const RelayoutParams& p, cudaStream_t stream) {
    static int blocks_per_sm = 0;  // same for every device of one architecture
    if (blocks_per_sm == 0) {
        int b = 0;
        cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, relayout_kernel<kDir, VW>, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm = b > 0 ? b : 1;
    }
    const int64_t want = int64_t(device_sms()) * blocks_per_sm;
    const unsigned grid = unsigned(want < int64_t(p.n_units) ? want : int64_t(p.n_units));
    return launch_overlapped(relayout_kernel<kDir, VW>, grid, kThreads, 0, stream, p);
}

template <int VW>
cudaError_t launch_width(const RelayoutParams& p, Dir dir, cudaStream_t stream) {
    return dir == Dir::kGather ? launch_one<Dir::kGather, VW>(p, stream) : launch_one<Dir::kScatter, VW>(p, stream);
}

}  // namespace

cudaError_t launch_relayout(const RelayoutParams& p, Dir dir, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.fused_mask != 0) return cudaErrorInvalidValue;
    if (p.vec_bytes == 32) return launch_width<32>(p, dir, stream);
    if (p.vec_bytes == 16) return launch_width<16>(p, dir, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_rope_table(float* table, const double* inv_freq_host, int S, int D, cudaStream_t stream) {
    RopeTableParams rp{};
    const int half = D / 2;
    if (half < 1 || half > 128) return cudaErrorInvalidValue;
    for (int i = 0; i < half; ++i) rp.inv_freq[i] = inv_freq_host[i];
    rp.out = table;
    rp.S = S;
    rp.half = half;
    const int64_t n = int64_t(S) * half;
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    const unsigned grid = unsigned(blocks < int64_t(device_sms()) * 8 ? blocks : int64_t(device_sms()) * 8);
    return launch_overlapped(rope_table_kernel, grid, 256, 0, stream, rp);
}

}  // namespace tfu
