// relayout_kernels.cu -- sm_103a kernels of the Ulysses sequence<->head relayout.
//
// What is computed (TeleFuser docs, "Communication Architecture", section
// "Sequence Parallel Communication / Ulysses"; head bands and rank-order
// concatenation as in flashinfer PR #6332, "Assumptions / Exchange algorithm"):
//   scatter:  T_g[b, r*Sl + t, h, :] = f_x(S_r[b, t, g*Hl + h, :], p = r*Sl + t)
//   gather:   O_r[b, t, g*Hl + h, :] = A_g[b, r*Sl + t, h, :]
// f_x is the identity (bit copy) for V and for plain scatters, and for Q/K in the
// fused mode the per-head RMSNorm + interleaved RoPE of flashinfer PR #6332,
// "Assumptions / Operator math" (see tf_ulysses.h for the formula).
//
// Design (HBM-bound data movement plus light fp32 math; no tensor cores):
//  * One grouped launch per call.  Work is split into units of 32 KiB of one
//    plane = (batch b, shard r, tensor slot x, head group g).  Units are ordered
//    chunk-major with g innermost, so CTAs running at the same time read whole
//    source token rows (all head groups), write the P head groups of one token
//    block, and in the fused mode share the same RoPE table rows through L2.
//    V (slot 0) comes first within each token block.
//  * A persistent grid (SM count x resident CTAs) walks the units.  Each lane
//    moves 32-byte vectors (16-byte when rows, strides or bases are only 16-byte
//    aligned) and issues all of its loads of a batch before any store.  Loads
//    skip L1 allocation (read once); stores are evict-first (not re-read here).
//  * Fused rows: a head row of D 16-bit values is spread over D*2/VW consecutive
//    lanes.  The sum of squares is carried as an unevaluated float pair (TwoSum)
//    through the lane and an xor-shuffle tree, so the fp32 mean is the correctly
//    rounded mean for ordinary inputs; then 1/sqrt(ms + eps) with IEEE-rounded
//    sqrt and reciprocal, the product rounded to the 16-bit type, the weight
//    scale as a packed 16-bit multiply (exactly the rounded product), and the
//    rotation with separately rounded fp32 products (no contraction), as a
//    step-by-step fp32 evaluation does.
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

// Fused Q/K rows of one unit, row-major: the CTA's kThreads / kLanes row groups
// each take a contiguous run of the unit's rows and walk it with four rows' loads
// in flight (software pipeline).  Consecutive rows of a run mostly belong to the
// same token (Hl heads per token), so a lane reloads its (cos, sin) entries only
// when the token changes.
// kExact = false: pipelined, the fast mean (a row whose sum of squares is not
// finite sets *redo); kExact = true: one row at a time with the complete mean
// (row_mean_sq), same rows per lane group.
template <Fused kF, int VW, int kLanes, bool kNeox, bool kExact>
__device__ __forceinline__ void norm_rope_rows(const RelayoutParams& p, const Plane& pl, uint32_t v0, uint32_t v1,
                                               volatile int* redo) {
    constexpr int NP = VW / 4;                    // element pairs per lane
    constexpr int kRowFloats = kLanes * NP * 2;  // D floats per table row: D/2 (cos, sin) pairs
    constexpr int kCs = cs_vecs<kNeox, NP>();
    constexpr uint32_t kGroups = kThreads / kLanes;
    const uint32_t g = threadIdx.x / kLanes, dv = threadIdx.x % kLanes;
    const uint32_t row0 = v0 / kLanes;  // first plane row of the unit (v0 is a multiple of kLanes)
    const uint32_t n_rows = (v1 - v0) / kLanes;
    const uint32_t per = (n_rows + kGroups - 1) / kGroups;  // rows per group, the same for every lane
    const uint32_t r_beg = g * per;
    uint32_t wpk[NP];
    {
        const Vec<VW> wv = *reinterpret_cast<const Vec<VW>*>(static_cast<const uint8_t*>(p.weight[pl.x]) + dv * VW);
#pragma unroll
        for (int j = 0; j < NP; ++j) wpk[j] = wv.w[j];
    }
    const float* tab_lane = p.table + size_t(pl.pos0) * kRowFloats + cs_lane_offset<kNeox, kLanes, NP>(dv);
    float4 cs[kCs];
#pragma unroll
    for (int k = 0; k < kCs; ++k) cs[k] = make_float4(1.f, 0.f, 1.f, 0.f);
    uint32_t t_cached = 0xffffffffu;
    auto load = [&](Vec<VW>& buf, uint32_t j) {
        const uint32_t i = r_beg + j;
#pragma unroll
        for (int w = 0; w < NP; ++w) buf.w[w] = 0u;
        if (j < per && i < n_rows) {
            const uint32_t R = row0 + i;
            const uint32_t t = fastdiv(R, p.div_hl);
            const uint32_t h = R - t * p.Hl;
            buf = ld_stream<VW>(pl.src + int64_t(t) * pl.st + int64_t(h) * pl.sh + int64_t(dv) * VW);
        }
    };
    auto compute_store = [&](Vec<VW>& buf, uint32_t j) {
        const uint32_t i = r_beg + j;
        const bool valid = j < per && i < n_rows;
        const uint32_t t = fastdiv(row0 + i, p.div_hl);
        const uint32_t h = row0 + i - t * p.Hl;
        if (valid && t != t_cached) {
            const float* tab = tab_lane + size_t(t) * kRowFloats;
#pragma unroll
            for (int k = 0; k < kCs; ++k) cs[k] = ld_table(tab + 4 * k);
            t_cached = t;
        }
        // every lane runs the row reduction (it shuffles); only valid rows are written
        norm_rope_core<kF, kLanes, NP, kNeox, kExact>(buf.w, wpk, cs, p.eps, redo);
        if (valid) st_stream<VW>(pl.dst + int64_t(t) * pl.dt + int64_t(h) * pl.dh + int64_t(dv) * VW, buf);
    };
    if constexpr (kExact) {
#pragma unroll 1
        for (uint32_t j = 0; j < per; ++j) {
            Vec<VW> b;
            load(b, j);
            compute_store(b, j);
        }
        return;
    }
    Vec<VW> b0, b1, b2, b3;
    load(b0, 0);
    load(b1, 1);
    load(b2, 2);
    load(b3, 3);
#pragma unroll 1
    for (uint32_t j = 0; j < per; j += 4) {
        compute_store(b0, j);
        load(b0, j + 4);
        compute_store(b1, j + 1);
        load(b1, j + 5);
        compute_store(b2, j + 2);
        load(b2, j + 6);
        compute_store(b3, j + 3);
        load(b3, j + 7);
    }
}

// Tuning constants (compile-time; overridable with -D for measurement sweeps).
// TFU_COPY_MIN_BLOCKS / TFU_FUSED_MIN_BLOCKS: resident 256-thread CTAs per SM the
// register budget is sized for.  TFU_COPY_BATCH: 32-byte vectors each lane
// loads before storing (twice as many 16-byte vectors).
#ifndef TFU_COPY_MIN_BLOCKS
#define TFU_COPY_MIN_BLOCKS 4
#endif
#ifndef TFU_FUSED_MIN_BLOCKS
#define TFU_FUSED_MIN_BLOCKS 2
#endif
#ifndef TFU_COPY_BATCH
#define TFU_COPY_BATCH 4
#endif

template <Fused kF>
__host__ __device__ constexpr int min_blocks() {
    return kF == Fused::kNone ? TFU_COPY_MIN_BLOCKS : TFU_FUSED_MIN_BLOCKS;
}
template <int VW>
__host__ __device__ constexpr int copy_batch() {
    return VW == 32 ? TFU_COPY_BATCH : 2 * TFU_COPY_BATCH;
}

template <Dir kDir, Fused kF, int VW, int kLanes, bool kNeox>
__global__ void __launch_bounds__(kThreads, min_blocks<kF>()) relayout_kernel(const __grid_constant__ RelayoutParams p) {
    constexpr uint32_t kChunk = uint32_t(chunk_vecs(VW));
    __shared__ int redo;  // set when a fused row's sum of squares was not finite
    if constexpr (kF != Fused::kNone) {
        if (threadIdx.x == 0) redo = 0;
        __syncthreads();
    }
#pragma unroll 1
    for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const uint32_t c = fastdiv(u, p.div_planes);
        const uint32_t q = u - c * p.n_planes;
        const Plane pl = decode_plane<kDir>(p, q);
        const uint32_t v0 = c * kChunk;
        const uint32_t v1 = min(v0 + kChunk, p.nv);
        if constexpr (kF != Fused::kNone) {
            if ((p.fused_mask >> pl.x) & 1u) {
                norm_rope_rows<kF, VW, kLanes, kNeox, false>(p, pl, v0, v1, &redo);
                continue;
            }
        }
        copy_range<kDir, VW, copy_batch<VW>()>(p, pl, v0, v1);
    }
    if constexpr (kF != Fused::kNone) {
        // A fused row whose sum of squares was not finite (an element of magnitude
        // >= 2^64, an infinite one or a NaN) was stored with the fast mean: if the
        // CTA met one, its fused rows are computed again with the complete mean,
        // each row by the lanes that stored it, after their first store.
        __syncthreads();
        if (redo) {
#pragma unroll 1
            for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
                const uint32_t c = fastdiv(u, p.div_planes);
                const Plane pl = decode_plane<kDir>(p, u - c * p.n_planes);
                if ((p.fused_mask >> pl.x) & 1u)
                    norm_rope_rows<kF, VW, kLanes, kNeox, true>(p, pl, c * kChunk, min(c * kChunk + kChunk, p.nv),
                                                                &redo);
            }
        }
    }
}

struct RopeTableParams {
    double inv_freq[128];
    float* out;
    int S, half;
};

__global__ void __launch_bounds__(256) rope_table_kernel(const __grid_constant__ RopeTableParams p) {
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

template <Dir kDir, Fused kF, int VW, int kLanes, bool kNeox>
cudaError_t launch_one(const RelayoutParams& p, cudaStream_t stream) {
    static int blocks_per_sm = 0;  // same for every device of one architecture
    if (blocks_per_sm == 0) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &b, relayout_kernel<kDir, kF, VW, kLanes, kNeox>, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm = b > 0 ? b : 1;
    }
    const int64_t want = int64_t(device_sms()) * blocks_per_sm;
    const unsigned grid = unsigned(want < int64_t(p.n_units) ? want : int64_t(p.n_units));
    relayout_kernel<kDir, kF, VW, kLanes, kNeox><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// Fused scatters reach this kernel only with 16-byte vectors (the block kernel
// takes the 32-byte ones): a head row of D in {32, 64, 128, 256} over D/8 lanes.
template <Fused kF, bool kNeox>
cudaError_t launch_fused(const RelayoutParams& p, cudaStream_t stream) {
    switch (p.vpr) {  // lanes per head row
        case 4: return launch_one<Dir::kScatter, kF, 16, 4, kNeox>(p, stream);
        case 8: return launch_one<Dir::kScatter, kF, 16, 8, kNeox>(p, stream);
        case 16: return launch_one<Dir::kScatter, kF, 16, 16, kNeox>(p, stream);
        case 32: return launch_one<Dir::kScatter, kF, 16, 32, kNeox>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int VW>
cudaError_t launch_width(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream) {
    if (dir == Dir::kGather) {
        if (fused != Fused::kNone) return cudaErrorInvalidValue;
        return launch_one<Dir::kGather, Fused::kNone, VW, 0, false>(p, stream);
    }
    if (fused == Fused::kNone) return launch_one<Dir::kScatter, Fused::kNone, VW, 0, false>(p, stream);
    if constexpr (VW == 16) {
        if (fused == Fused::kBF16)
            return p.rope_neox ? launch_fused<Fused::kBF16, true>(p, stream) : launch_fused<Fused::kBF16, false>(p, stream);
        if (fused == Fused::kFP16)
            return p.rope_neox ? launch_fused<Fused::kFP16, true>(p, stream) : launch_fused<Fused::kFP16, false>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_relayout(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.vec_bytes == 32) return launch_width<32>(p, dir, fused, stream);
    if (p.vec_bytes == 16) return launch_width<16>(p, dir, fused, stream);
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
    rope_table_kernel<<<grid, 256, 0, stream>>>(rp);
    return cudaGetLastError();
}

}  // namespace tfu
