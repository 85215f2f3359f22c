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

// Scatter targets are contiguous [B, S, Hl, D]: vector v of a plane lands at v * VW.
template <Dir kDir, int VW>
__device__ __forceinline__ int64_t dst_offset(const RelayoutParams& p, const Plane& pl, uint32_t v) {
    if constexpr (kDir == Dir::kScatter) {
        return int64_t(v) * VW;
    } else {
        return vec_offset<VW>(p, v, pl.dt, pl.dh);
    }
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

#ifndef TFU_FUSED_PIPELINE
#define TFU_FUSED_PIPELINE 1  // 1: software-pipelined half batches, 0: load-all-then-compute batches
#endif

// Fused Q/K rows of one unit.  VB slots per thread; pipelined as two half
// batches of VB/2 slots: the loads of one half are in flight while the other
// half is normalised, rotated and stored, so a warp never computes with no
// loads outstanding.
template <Fused kF, int VW, int kLanes, int VB>
__device__ __forceinline__ void norm_rope_range(const RelayoutParams& p, const Plane& pl, uint32_t v0, uint32_t v1) {
    constexpr int NP = VW / 4;                    // element pairs per lane
    constexpr int kRowFloats = kLanes * NP * 2;  // D floats per table row: D/2 (cos, sin) pairs
    constexpr int H = TFU_FUSED_PIPELINE ? VB / 2 : VB;
    constexpr uint32_t kStep = uint32_t(kThreads) * H;  // vectors per half batch
    const uint32_t dv = threadIdx.x % kLanes;    // v0 and kThreads are multiples of kLanes
    uint32_t wpk[NP];
    {
        const Vec<VW> wv = *reinterpret_cast<const Vec<VW>*>(static_cast<const uint8_t*>(p.weight[pl.x]) + dv * VW);
#pragma unroll
        for (int j = 0; j < NP; ++j) wpk[j] = wv.w[j];
    }
    const float* tab_lane = p.table + size_t(pl.pos0) * kRowFloats + dv * (2 * NP);
    auto load = [&](Vec<VW>(&buf)[H], uint32_t base) {
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
#pragma unroll
            for (int j = 0; j < NP; ++j) buf[i].w[j] = 0u;
            if (v < v1) {
                const uint32_t row = v / kLanes;
                const uint32_t t = fastdiv(row, p.div_hl);
                const uint32_t h = row - t * p.Hl;
                buf[i] = ld_stream<VW>(pl.src + int64_t(t) * pl.st + int64_t(h) * pl.sh + int64_t(dv) * VW);
            }
        }
    };
    auto compute_store = [&](Vec<VW>(&buf)[H], uint32_t base) {
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            const uint32_t t = fastdiv(v / kLanes, p.div_hl);
            // every lane runs the row reduction (it shuffles); only valid lanes load and store
            norm_rope_lane<kF, kLanes, NP>(buf[i].w, wpk, tab_lane + size_t(t) * kRowFloats, v < v1, p.eps);
            if (v < v1) st_stream<VW>(pl.dst + int64_t(v) * VW, buf[i]);
        }
    };
    Vec<VW> a[H];
    if constexpr (TFU_FUSED_PIPELINE) {
        Vec<VW> b[H];
        load(a, v0);
#pragma unroll 1
        for (uint32_t base = v0; base < v1; base += 2 * kStep) {
            load(b, base + kStep);  // fully masked past the end of the range
            compute_store(a, base);
            load(a, base + 2 * kStep);
            compute_store(b, base + kStep);
        }
    } else {
#pragma unroll 1
        for (uint32_t base = v0; base < v1; base += kStep) {
            load(a, base);
            compute_store(a, base);
        }
    }
}

#ifndef TFU_FUSED_ROWMAJOR
#define TFU_FUSED_ROWMAJOR 1  // 1: row runs per lane group (norm_rope_rows), 0: norm_rope_range
#endif

// Fused Q/K rows of one unit, row-major: the CTA's kThreads / kLanes row groups
// each take a contiguous run of the unit's rows and walk it with four rows' loads
// in flight (software pipeline).  Consecutive rows of a run mostly belong to the
// same token (Hl heads per token), so a lane reloads its (cos, sin) pairs only
// when the token changes.
template <Fused kF, int VW, int kLanes>
__device__ __forceinline__ void norm_rope_rows(const RelayoutParams& p, const Plane& pl, uint32_t v0, uint32_t v1) {
    constexpr int NP = VW / 4;                    // element pairs per lane
    constexpr int kRowFloats = kLanes * NP * 2;  // D floats per table row: D/2 (cos, sin) pairs
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
    const float* tab_lane = p.table + size_t(pl.pos0) * kRowFloats + dv * (2 * NP);
    float4 cs[NP / 2];
#pragma unroll
    for (int k = 0; k < NP / 2; ++k) cs[k] = make_float4(1.f, 0.f, 1.f, 0.f);
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
        if (valid && t != t_cached) {
            const float* tab = tab_lane + size_t(t) * kRowFloats;
#pragma unroll
            for (int k = 0; k < NP / 2; ++k) cs[k] = ld_table(tab + 4 * k);
            t_cached = t;
        }
        // every lane runs the row reduction (it shuffles); only valid rows are written
        norm_rope_core<kF, kLanes, NP>(buf.w, wpk, cs, p.eps);
        if (valid) st_stream<VW>(pl.dst + int64_t(row0 + i) * (kLanes * VW) + int64_t(dv) * VW, buf);
    };
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
// register budget is sized for.  TFU_COPY_BATCH / TFU_FUSED_BATCH: 32-byte
// vectors each lane loads before storing (twice as many 16-byte vectors).
#ifndef TFU_COPY_MIN_BLOCKS
#define TFU_COPY_MIN_BLOCKS 4
#endif
#ifndef TFU_FUSED_MIN_BLOCKS
#define TFU_FUSED_MIN_BLOCKS 2
#endif
#ifndef TFU_COPY_BATCH
#define TFU_COPY_BATCH 4
#endif
#ifndef TFU_FUSED_BATCH
#define TFU_FUSED_BATCH 4
#endif

template <Fused kF>
__host__ __device__ constexpr int min_blocks() {
    return kF == Fused::kNone ? TFU_COPY_MIN_BLOCKS : TFU_FUSED_MIN_BLOCKS;
}
template <int VW>
__host__ __device__ constexpr int copy_batch() {
    return VW == 32 ? TFU_COPY_BATCH : 2 * TFU_COPY_BATCH;
}
template <int VW>
__host__ __device__ constexpr int fused_batch() {
    return VW == 32 ? TFU_FUSED_BATCH : 2 * TFU_FUSED_BATCH;
}

template <Dir kDir, Fused kF, int VW, int kLanes>
__global__ void __launch_bounds__(kThreads, min_blocks<kF>()) relayout_kernel(const __grid_constant__ RelayoutParams p) {
    constexpr uint32_t kChunk = uint32_t(chunk_vecs(VW));
#pragma unroll 1
    for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const uint32_t c = fastdiv(u, p.div_planes);
        const uint32_t q = u - c * p.n_planes;
        const Plane pl = decode_plane<kDir>(p, q);
        const uint32_t v0 = c * kChunk;
        const uint32_t v1 = min(v0 + kChunk, p.nv);
        if constexpr (kF != Fused::kNone) {
            if ((p.fused_mask >> pl.x) & 1u) {
                if constexpr (TFU_FUSED_ROWMAJOR) {
                    norm_rope_rows<kF, VW, kLanes>(p, pl, v0, v1);
                } else {
                    norm_rope_range<kF, VW, kLanes, fused_batch<VW>()>(p, pl, v0, v1);
                }
                continue;
            }
        }
        copy_range<kDir, VW, copy_batch<VW>()>(p, pl, v0, v1);
    }
}

#ifndef TFU_BLOCK_DEPTH
#define TFU_BLOCK_DEPTH 2  // rows (of every slot) each lane has loaded ahead of the one it computes
#endif
#ifndef TFU_COPY_BLOCK_DEPTH
#define TFU_COPY_BLOCK_DEPTH 4  // the same for block launches without fused slots
#endif
#ifndef TFU_COPY_BLOCK_MIN_BLOCKS
#define TFU_COPY_BLOCK_MIN_BLOCKS 2  // resident CTAs per SM the copy block kernel's registers allow
#endif

// Scatter over token blocks of all tensors together.  A unit is the row range
// [c * rpu, ...) of one (batch b, shard r, head group g) block for every slot:
// kCopy copied slots (V first) followed by kNF fused ones (Q, then K).  Each lane
// group of kLanes lanes walks a contiguous run of the unit's rows; for each row
// it loads its 32-byte chunk from every slot, normalises and rotates the fused
// ones with one (cos, sin) load that both share and that is reused across the
// heads of a token, and stores every slot.  So V's loads and stores are in
// flight while the same warps compute Q/K, and no SM idles in a copy-only or a
// math-only phase.  Destination rows of a block are d_h bytes apart.
template <Fused kF, int kLanes, int kCopy, int kNF>
__global__ void __launch_bounds__(kThreads, kNF > 0 ? TFU_FUSED_MIN_BLOCKS : TFU_COPY_BLOCK_MIN_BLOCKS)
    block_kernel(const __grid_constant__ RelayoutParams p) {
    constexpr int VW = 32, NP = 8;                // 32 bytes = 8 element pairs per lane
    constexpr int kSlots = kCopy + kNF;
    constexpr int kDepth = kNF > 0 ? TFU_BLOCK_DEPTH : TFU_COPY_BLOCK_DEPTH;
    constexpr int kRowFloats = kLanes * NP * 2;  // D floats per table row
    constexpr uint32_t kGroups = kThreads / kLanes;
    static_assert(kSlots >= 1 && kSlots <= kMaxSlots && (kNF == 0) == (kF == Fused::kNone), "slot pattern");
    const uint32_t g_row = threadIdx.x / kLanes, dv = threadIdx.x % kLanes;
    uint32_t w[kNF > 0 ? kNF : 1][NP];  // this lane's weight pairs of each fused slot
#pragma unroll
    for (int f = 0; f < kNF; ++f) {
        const Vec<VW> wv =
            *reinterpret_cast<const Vec<VW>*>(static_cast<const uint8_t*>(p.weight[kCopy + f]) + dv * VW);
#pragma unroll
        for (int j = 0; j < NP; ++j) w[f][j] = wv.w[j];
    }
#pragma unroll 1
    for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const uint32_t c = fastdiv(u, p.div_planes);
        const uint32_t q = u - c * p.n_planes;  // q = (b * P + r) * P + g
        const uint32_t g = q % p.P;
        const uint32_t r = (q / p.P) % p.P;
        const uint32_t b = q / (p.P * p.P);
        const uint8_t* src[kSlots];
        uint8_t* dst[kSlots];
#pragma unroll
        for (int x = 0; x < kSlots; ++x) {
            src[x] = p.src[x][r] + int64_t(b) * p.s_b[x] + int64_t(g) * p.Hl * p.s_h[x] + int64_t(dv) * VW;
            dst[x] = p.dst[x][g] + int64_t(b) * p.d_b[x] + int64_t(r) * p.Sl * p.d_t[x] + int64_t(dv) * VW;
        }
        const uint32_t R0 = c * p.rpu;
        const uint32_t n_rows = min(R0 + p.rpu, p.plane_rows) - R0;
        const uint32_t per = (n_rows + kGroups - 1) / kGroups;  // rows per group, the same for every lane
        const uint32_t r_beg = R0 + g_row * per;                 // first plane row of this group
        const uint32_t r_end = min(r_beg + per, R0 + n_rows);    // may be <= r_beg for trailing groups
        const float* tab_lane = kNF > 0 ? p.table + size_t(r) * p.Sl * kRowFloats + dv * (2 * NP) : nullptr;
        float4 cs[NP / 2];
#pragma unroll
        for (int k = 0; k < NP / 2; ++k) cs[k] = make_float4(1.f, 0.f, 1.f, 0.f);
        uint32_t t_cached = 0xffffffffu;
        auto load = [&](Vec<VW>(&buf)[kSlots], uint32_t R) {
            const uint32_t t = fastdiv(R, p.div_hl);
            const uint32_t h = R - t * p.Hl;
#pragma unroll
            for (int x = 0; x < kSlots; ++x) {
                if constexpr (kNF > 0) {  // masked rows still go through the row reduction
#pragma unroll
                    for (int k = 0; k < NP; ++k) buf[x].w[k] = 0u;
                }
                if (R < r_end) buf[x] = ld_stream<VW>(src[x] + int64_t(t) * p.s_t[x] + int64_t(h) * p.s_h[x]);
            }
        };
        auto compute_store = [&](Vec<VW>(&buf)[kSlots], uint32_t R) {
            const bool valid = R < r_end;
            if constexpr (kNF > 0) {
                const uint32_t t = fastdiv(R, p.div_hl);
                if (valid && t != t_cached) {
                    const float* tab = tab_lane + size_t(t) * kRowFloats;
#pragma unroll
                    for (int k = 0; k < NP / 2; ++k) cs[k] = ld_table(tab + 4 * k);
                    t_cached = t;
                }
                // every lane runs the row reductions (they shuffle); only valid rows are written
#pragma unroll
                for (int f = 0; f < kNF; ++f) norm_rope_core<kF, kLanes, NP>(buf[kCopy + f].w, w[f], cs, p.eps);
            }
            if (valid) {
#pragma unroll
                for (int x = 0; x < kSlots; ++x) st_stream<VW>(dst[x] + int64_t(R) * p.d_h[x], buf[x]);
            }
        };
        Vec<VW> bufs[kDepth][kSlots];
#pragma unroll
        for (int d = 0; d < kDepth; ++d) load(bufs[d], r_beg + d);
#pragma unroll 1
        for (uint32_t R = r_beg; R < r_beg + per; R += kDepth) {
#pragma unroll
            for (int d = 0; d < kDepth; ++d) {
                compute_store(bufs[d], R + d);
                load(bufs[d], R + d + kDepth);
            }
        }
    }
}

template <Fused kF, int kLanes, int kCopy, int kNF>
cudaError_t launch_block(const RelayoutParams& p, cudaStream_t stream) {
    static int blocks_per_sm = 0;  // same for every device of one architecture
    if (blocks_per_sm == 0) {
        int bps = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, block_kernel<kF, kLanes, kCopy, kNF>,
                                                                      kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm = bps > 0 ? bps : 1;
    }
    const int64_t want = int64_t(device_sms()) * blocks_per_sm;
    const unsigned grid = unsigned(want < int64_t(p.n_units) ? want : int64_t(p.n_units));
    block_kernel<kF, kLanes, kCopy, kNF><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <Fused kF, int kCopy, int kNF>
cudaError_t launch_block_lanes(const RelayoutParams& p, cudaStream_t stream) {
    switch (p.vpr) {  // lanes per head row = D * esize / 32
        case 2: return launch_block<kF, 2, kCopy, kNF>(p, stream);
        case 4: return launch_block<kF, 4, kCopy, kNF>(p, stream);
        case 8: return launch_block<kF, 8, kCopy, kNF>(p, stream);
        case 16: return launch_block<kF, 16, kCopy, kNF>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <Fused kF>
cudaError_t launch_block_fused(const RelayoutParams& p, cudaStream_t stream) {
    const uint32_t n_copy = (p.fused_mask & 1u) ? 0u : 1u;  // V (unfused) can only be slot 0
    const uint32_t nf = p.nx - n_copy;
    if (nf < 1 || nf > 2 || p.fused_mask != ((1u << nf) - 1u) << n_copy) return cudaErrorInvalidValue;
    if (n_copy) return nf == 2 ? launch_block_lanes<kF, 1, 2>(p, stream) : launch_block_lanes<kF, 1, 1>(p, stream);
    return nf == 2 ? launch_block_lanes<kF, 0, 2>(p, stream) : launch_block_lanes<kF, 0, 1>(p, stream);
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
        const float c = __double2float_rn(cos(angle));
        const float s = __double2float_rn(sin(angle));
        reinterpret_cast<float2*>(p.out)[idx] = make_float2(c, s);
    }
}

template <Dir kDir, Fused kF, int VW, int kLanes>
cudaError_t launch_one(const RelayoutParams& p, cudaStream_t stream) {
    static int blocks_per_sm = 0;  // same for every device of one architecture
    if (blocks_per_sm == 0) {
        int b = 0;
        cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, relayout_kernel<kDir, kF, VW, kLanes>, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm = b > 0 ? b : 1;
    }
    const int64_t want = int64_t(device_sms()) * blocks_per_sm;
    const unsigned grid = unsigned(want < int64_t(p.n_units) ? want : int64_t(p.n_units));
    relayout_kernel<kDir, kF, VW, kLanes><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <Fused kF, int VW>
cudaError_t launch_fused(const RelayoutParams& p, cudaStream_t stream) {
    switch (p.vpr) {  // lanes per head row
        case 2: return launch_one<Dir::kScatter, kF, VW, 2>(p, stream);
        case 4: return launch_one<Dir::kScatter, kF, VW, 4>(p, stream);
        case 8: return launch_one<Dir::kScatter, kF, VW, 8>(p, stream);
        case 16: return launch_one<Dir::kScatter, kF, VW, 16>(p, stream);
        case 32: return launch_one<Dir::kScatter, kF, VW, 32>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int VW>
cudaError_t launch_width(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream) {
    if (dir == Dir::kGather) {
        if (fused != Fused::kNone) return cudaErrorInvalidValue;
        return launch_one<Dir::kGather, Fused::kNone, VW, 0>(p, stream);
    }
    switch (fused) {
        case Fused::kNone: return launch_one<Dir::kScatter, Fused::kNone, VW, 0>(p, stream);
        case Fused::kBF16: return launch_fused<Fused::kBF16, VW>(p, stream);
        case Fused::kFP16: return launch_fused<Fused::kFP16, VW>(p, stream);
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

cudaError_t launch_blocks(const RelayoutParams& p, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.vec_bytes != 32 || p.rpu == 0) return cudaErrorInvalidValue;
    switch (fused) {
        case Fused::kNone:
            if (p.fused_mask != 0) return cudaErrorInvalidValue;
            switch (p.nx) {
                case 1: return launch_block_lanes<Fused::kNone, 1, 0>(p, stream);
                case 2: return launch_block_lanes<Fused::kNone, 2, 0>(p, stream);
                case 3: return launch_block_lanes<Fused::kNone, 3, 0>(p, stream);
                default: return cudaErrorInvalidValue;
            }
        case Fused::kBF16: return p.table ? launch_block_fused<Fused::kBF16>(p, stream) : cudaErrorInvalidValue;
        case Fused::kFP16: return p.table ? launch_block_fused<Fused::kFP16>(p, stream) : cudaErrorInvalidValue;
    }
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
