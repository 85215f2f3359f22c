// block_kernel.cuh -- the scatter over token blocks of all tensors together
// (sm_103a), used for every fused scatter; block_kernels.cu instantiates it for
// 32-byte-aligned rows, block_kernels_v16.cu for rows only 16-byte aligned.
//
// What is computed (TeleFuser docs, "Communication Architecture", section
// "Sequence Parallel Communication / Ulysses"; head bands and rank order as in
// flashinfer PR #6332 commit message, "Assumptions / Exchange algorithm"):
//   T^x_g[b, r*Sl + t, h, :] = f_x(S^x_r[b, t, g*Hl + h, :], p = r*Sl + t)
// with f_x the bit copy for V (and every tensor of a plain scatter) and, for Q/K
// of a fused scatter, RMSNorm + weight + RoPE (flashinfer PR #6332,
// "Assumptions / Operator math"; interleaved pairs, or half-split pairs).
// TeleFuser PR #27 overlaps V's transfer with the Q/K norm/RoPE ("Changes
// Made"); on one GPU both are SM work, so here they share every warp: a unit
// carries V's rows and Q/K's rows of the same token block.
//
// Design:
//  * A unit is the row range [c*rpu, (c+1)*rpu) of one (batch b, shard r, head
//    group g) block, for every slot: kCopy copied slots (V first) and kNF fused
//    ones (Q, then K).  A persistent grid walks the units, chunk-major with g
//    innermost, so CTAs running together read whole source token rows and
//    write all P head groups of a token block.
//  * Each lane group of kLanes = D*2/32 lanes takes a contiguous run of the
//    unit's rows and keeps kDepth rows (of every slot) loaded ahead of the one it
//    computes, across unit boundaries too: the last pass over a unit's rows
//    already loads the group's rows of its next unit (V+Q+K launches of many
//    rounds of units keep to one unit at a time, which measured faster there).
//    32 bytes per lane per row and slot, moved as one 32-byte vector or, when
//    sources or targets are only 16-byte aligned (kV16), as two 16-byte ones
//    (the lane layout is the same); loads bypass L1, stores are evict-first.
//  * The (cos, sin) entries are loaded once per token and reused across its
//    heads and by Q and K; launches without a copied slot bring them into a
//    per-thread shared-memory ring with the row loads, so that the arithmetic
//    never waits on them.  Q/K-only launches compute the Q and K rows of a
//    position together (norm_rope_qk).  Destination row (t, h) sits at t*d_t + h*d_h, so the
//    same code writes the separate [B, S, Hl, D] targets, the fused receive
//    layout [B, S, Hl, 3*D] (d_h = 3*D*esize, slot offsets 0, D, 2D) and a head
//    chunk of wider targets (d_t > Hl*d_h; source bands Hg heads apart).
#pragma once

#include <atomic>
#include <type_traits>

#include "device_common.cuh"
#include "relayout.h"

#ifndef TFU_FUSED_MIN_BLOCKS
#define TFU_FUSED_MIN_BLOCKS 2  // resident 256-thread CTAs per SM the fused register budget is sized for
#endif
#ifndef TFU_COPY_BLOCK_MIN_BLOCKS
#define TFU_COPY_BLOCK_MIN_BLOCKS 2  // resident CTAs per SM the copy block kernel's registers allow
#endif

namespace tfu {
namespace {

using namespace dev;

// 16 bytes of a half-split head row, read-only, allocating in L1
__device__ __forceinline__ Vec<16> ld_half(const uint8_t* p) {
    Vec<16> v;
    asm("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
        : "l"(p));
    return v;
}

// The (cos, sin) ring of launches without a copied slot (block_tab_ring): each
// thread's own entries, 16 bytes per cp.async, read back by the same thread after
// its copies have landed (cp.async.wait_group), so no barrier is involved.
__device__ __forceinline__ void tab_cp16(uint32_t saddr, const float* g) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void tab_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void tab_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ float4 tab_lds(uint32_t saddr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}
// Table rows in flight per thread: at most one per row loaded ahead, and one more
// so that a slot is rewritten only a full row after it was read.
constexpr int kTabSlots = 4;
// Q/K-only video DiT: 248 against 254 us with the ring (DRAM waits 1.33 against
// 2.29 stalls per issue); V+Q+K launches measured slower with it (311.0 against
// 307.4 us, the FLUX-like scatter 31.5 against 29.6 us) and load the entries
// directly.
template <int kCopy, int kNF>
__host__ __device__ constexpr bool block_tab_ring() {
    return kCopy == 0 && kNF > 0;
}
// dynamic shared memory: kTabSlots slots x 4 float4s x kThreads threads
template <int kCopy, int kNF>
__host__ __device__ constexpr size_t block_tab_smem() {
    return block_tab_ring<kCopy, kNF>() ? size_t(kTabSlots) * 4 * kThreads * 16 : 0;
}

#if TFU_CHECKED
// checked builds: nonzero once an access fell outside its planned buffer
__device__ unsigned g_block_status;
#endif

// Whether [ptr, ptr + bytes) lies in [lo, end).  Checked builds test it and
// record a failure in g_block_status (the caller then skips the access); other
// builds compile it to `true`.
__device__ __forceinline__ bool access_ok(const void* ptr, uint32_t bytes, const void* lo, const void* end) {
#if TFU_CHECKED
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    if (lo && a >= reinterpret_cast<uintptr_t>(lo) && a + bytes <= reinterpret_cast<uintptr_t>(end)) return true;
    atomicOr(&g_block_status, 1u);
    return false;
#else
    (void)ptr, (void)bytes, (void)lo, (void)end;
    return true;
#endif
}

// g_block_status of this translation unit (always 0 in unchecked builds)
inline cudaError_t read_this_block_status(unsigned* out, bool clear) {
#if TFU_CHECKED
    cudaError_t e = cudaMemcpyFromSymbol(out, g_block_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_block_status, &zero, sizeof(unsigned));
#else
    (void)clear;
    *out = 0;
    return cudaSuccess;
#endif
}

inline int block_device_sms() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

#ifndef TFU_QK_MIN_BLOCKS
#define TFU_QK_MIN_BLOCKS TFU_FUSED_MIN_BLOCKS  // resident CTAs per SM for fused launches without a copied slot
#endif

template <int kCopy, int kNF>
__host__ __device__ constexpr int block_min_blocks() {
    return kNF == 0 ? TFU_COPY_BLOCK_MIN_BLOCKS : (kCopy == 0 ? TFU_QK_MIN_BLOCKS : TFU_FUSED_MIN_BLOCKS);
}

#ifndef TFU_BLOCK_STREAM
// 1: each row group streams the rows of all its units (next unit's loads during
// the last pass of the one before); 0: one unit at a time
#define TFU_BLOCK_STREAM 1
#endif
#ifndef TFU_STREAM_MAX_ROUNDS
// V+Q+K fused launches stream only while the grid walks at most this many rounds
// of units.  Streaming measured (P=4, H=24, D=128, read-flushed fractions of the
// copy peak) +7 % at 5 and 10 rounds, +4 % at 20, +2 % at 25-35 and nothing at
// 40-60; but -1.3 to -2 % at 40-81 rounds with wider head bands (the video DiT,
// 67 rounds; S=32760 at H=48).  Copy and Q/K-only launches gained at every size
// (video-DiT copy scatter +2.6 %).
#define TFU_STREAM_MAX_ROUNDS 36
#endif

template <Fused kF, int kLanes, int kCopy, int kNF, bool kNeox, bool kStream, bool kV16>
__global__ void __launch_bounds__(kThreads, block_min_blocks<kCopy, kNF>())
    block_kernel(const __grid_constant__ RelayoutParams p) {
    constexpr int VW = 32, NP = 8;                // 32 bytes = 8 element pairs per lane
    constexpr int kSlots = kCopy + kNF;
    constexpr int kDepth = kNF == 0 ? kCopyBlockDepth : (kCopy == 0 ? kQkBlockDepth : kBlockDepth);
    constexpr int kRowFloats = kLanes * NP * 2;  // D floats per table row
    constexpr int kCs = NP / 2;                   // (cos, sin) float4s of the lane's element pairs
    constexpr uint32_t kGroups = kThreads / kLanes;
    constexpr uint32_t kHalf = kLanes * 16;       // bytes in half a head row
    static_assert(kSlots >= 1 && kSlots <= kMaxSlots && (kNF == 0) == (kF == Fused::kNone), "slot pattern");
    static_assert(!block_tab_ring<kCopy, kNF>() || kTabSlots >= kDepth + 1,
                  "the table ring holds a slot for every row in flight and one more");
    const uint32_t g_row = threadIdx.x / kLanes, dv = threadIdx.x % kLanes;
    // Lane dv's bytes of a head row: one 32-byte vector at dv*32 -- or, for the
    // fused slots of half-split RoPE, 16 bytes at dv*16 of each half, so that
    // both elements of every rotation pair sit in the same lane.
    auto is_split = [](int x) { return kNeox && x >= kCopy; };
    const uint32_t lane_off[2] = {dv * VW, dv * 16};  // whole-vector slots, split slots
    // checked builds: a lane's row (holding its lane offset) of slot x against
    // the planned bounds of shard/head-group i's buffer; the whole head row is tested
    constexpr uint32_t kRowBytes = kLanes * VW;
    auto src_ok = [&](const uint8_t* row, int x, uint32_t i) {
#if TFU_CHECKED
        return access_ok(row - lane_off[is_split(x) ? 1 : 0], kRowBytes, p.src[x][i], p.src_end[x][i]);
#else
        (void)row, (void)x, (void)i;
        return true;
#endif
    };
    auto dst_ok = [&](const uint8_t* row, int x, uint32_t i) {
#if TFU_CHECKED
        return access_ok(row - lane_off[is_split(x) ? 1 : 0], kRowBytes, p.dst[x][i], p.dst_end[x][i]);
#else
        (void)row, (void)x, (void)i;
        return true;
#endif
    };
    // a lane's (cos, sin) entries of one token: 2 * NP floats
    auto tab_ok = [&](const float* t) {
#if TFU_CHECKED
        return access_ok(t, 2 * NP * sizeof(float), p.table, p.table_end);
#else
        (void)t;
        return true;
#endif
    };
    // `row` already holds the lane's offset (lane_off)
    auto ld_lane = [&](const uint8_t* row, int x) {
        if (!is_split(x)) {
            if constexpr (!kV16) {
                return ld_stream<VW>(row);
            } else {
                const Vec<16> lo = ld_stream<16>(row), hi = ld_stream<16>(row + 16);
                Vec<VW> v;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v.w[k] = lo.w[k];
                    v.w[4 + k] = hi.w[k];
                }
                return v;
            }
        }
        // the two 16-byte halves go through L1: the video-DiT half-split scatter
        // measured 6389 GB/s against 6314 with L1::no_allocate on these loads
        const Vec<16> lo = ld_half(row), hi = ld_half(row + kHalf);
        Vec<VW> v;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v.w[k] = lo.w[k];
            v.w[4 + k] = hi.w[k];
        }
        return v;
    };
    auto st_lane = [&](uint8_t* row, int x, const Vec<VW>& v) {
        if (!is_split(x) && !kV16) {
            st_stream<VW>(row, v);
            return;
        }
        Vec<16> lo, hi;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            lo.w[k] = v.w[k];
            hi.w[k] = v.w[4 + k];
        }
        st_stream<16>(row, lo);
        st_stream<16>(row + (is_split(x) ? kHalf : 16u), hi);
    };
    // the weight pairs of each fused slot by lane position, in shared memory
    __shared__ uint32_t w_all[kNF > 0 ? kNF : 1][kLanes][NP];
    // set when a row's sum of squares was not finite: the fused rows are computed again below
    __shared__ int redo;
    if (threadIdx.x == 0) redo = 0;
    grid_dependency_wait();  // nothing global is touched before this
    if (threadIdx.x < kLanes) {
        const uint32_t lp = threadIdx.x;
#pragma unroll
        for (int f = 0; f < kNF; ++f) {
            const uint8_t* wrow = static_cast<const uint8_t*>(p.weight[kCopy + f]);
            const uint4 a = *reinterpret_cast<const uint4*>(wrow + (kNeox ? lp * 16 : lp * VW));
            const uint4 b = *reinterpret_cast<const uint4*>(wrow + (kNeox ? kHalf + lp * 16 : lp * VW + 16));
            w_all[f][lp][0] = a.x, w_all[f][lp][1] = a.y, w_all[f][lp][2] = a.z, w_all[f][lp][3] = a.w;
            w_all[f][lp][4] = b.x, w_all[f][lp][5] = b.y, w_all[f][lp][6] = b.z, w_all[f][lp][7] = b.w;
        }
    }
    // Q/K only: the (Q, K) weight pairs of each of the lane's elements (norm_rope_qk)
    __shared__ uint32_t wqk_all[kLanes][kNF == 2 ? 2 * NP : 1];
    if constexpr (kNF == 2 && kCopy == 0) {
        __syncthreads();
        if (threadIdx.x < kLanes * NP) {
            const uint32_t lp = threadIdx.x / NP, j = threadIdx.x % NP;
            const uint32_t wq = w_all[0][lp][j], wk = w_all[1][lp][j];
            wqk_all[lp][2 * j] = __byte_perm(wq, wk, 0x5410);
            wqk_all[lp][2 * j + 1] = __byte_perm(wq, wk, 0x7632);
        }
    }
    __syncthreads();
    auto w = [&](int f) -> const uint32_t(&)[NP] { return w_all[f][dv]; };
    // A group's rows of one unit: plane rows [beg, end) (empty for trailing
    // groups) and the pipeline slots that walk them (a multiple of kDepth)
    struct Span {
        uint32_t beg, end, slots;
    };
    auto span_of = [&](uint32_t c) -> Span {
        const uint32_t R0 = c * p.rpu;
        const uint32_t n_rows = min(R0 + p.rpu, p.plane_rows) - R0;
        const uint32_t per = (n_rows + kGroups - 1) / kGroups;  // rows per group, the same for every lane
        const uint32_t beg = R0 + g_row * per;
        return Span{beg, min(beg + per, R0 + n_rows), (per + kDepth - 1) / kDepth * kDepth};
    };
    uint32_t g, r, b;  // the (head group, shard, batch) of the unit located last
    uint32_t g_st = 0;  // the head group of the unit being stored (set_dst)
    auto locate = [&](uint32_t u) -> Span {
        const uint32_t c = fastdiv(u, p.div_planes);
        const uint32_t q = u - c * p.n_planes;  // q = (b * P + r) * P + g
        g = q % p.P;
        r = (q / p.P) % p.P;
        b = q / (p.P * p.P);
        return span_of(c);
    };
    const uint8_t* src[kSlots];  // each slot's source block of the unit being loaded
    uint8_t* dst[kSlots];        // each slot's target block of the unit being stored
    const float* tab_lane = nullptr;
    float4 cs[kCs];              // the lane's (cos, sin) entries of token t_cached
#pragma unroll
    for (int k = 0; k < kCs; ++k) cs[k] = make_float4(1.f, 0.f, 1.f, 0.f);
    uint32_t t_cached = 0xffffffffu;
    // Each thread's (cos, sin) entries travel through its own slots of a small
    // shared-memory ring: copied (cp.async) when a row of a new token is loaded,
    // read back when that row is computed.  Slot s, float4 k of thread i at
    // ((s * kCs + k) * kThreads + i) * 16.
    extern __shared__ __align__(16) uint8_t tab_ring[];
    const uint32_t ring0 = uint32_t(__cvta_generic_to_shared(tab_ring)) + threadIdx.x * 16u;
    auto ring_at = [&](uint32_t slot, int k) { return ring0 + (slot * kCs + uint32_t(k)) * kThreads * 16u; };
    uint32_t t_loaded = 0xffffffffu, n_loaded = 0, n_read = 0;
    // RMSNorm + weight + RoPE of the lane's part of one row of fused slot f
    auto fused_row = [&](auto exact, uint32_t(&xw)[NP], int f) {
        constexpr bool kExact = decltype(exact)::value;
        if constexpr (kNeox) {
            norm_rope_core_split<kF, kLanes, NP, kExact>(xw, w(f), cs, p.eps, &redo);
        } else {
            norm_rope_core<kF, kLanes, NP, kExact>(xw, w(f), cs, p.eps, &redo);
        }
    };
    auto set_src = [&]() {
#pragma unroll
        for (int x = 0; x < kSlots; ++x) {
            const uint32_t lo = lane_off[is_split(x) ? 1 : 0];
            src[x] = p.src[x][r] + int64_t(b) * p.s_b[x] + int64_t(g) * p.Hg * p.s_h[x] + lo;
        }
        t_loaded = 0xffffffffu;  // a new unit on the load side
    };
    auto set_dst = [&]() {
#pragma unroll
        for (int x = 0; x < kSlots; ++x) {
            const uint32_t lo = lane_off[is_split(x) ? 1 : 0];
            dst[x] = p.dst[x][g] + int64_t(b) * p.d_b[x] + int64_t(r) * p.Sl * p.d_t[x] + lo;
        }
        g_st = g;
        // the lane's element pairs use table entries [dv*NP, dv*NP + NP) in both mappings
        if constexpr (kNF > 0) tab_lane = p.table + size_t(r) * p.Sl * kRowFloats + dv * (2 * NP);
        t_cached = 0xffffffffu;  // a new shard r: another table block
    };
    auto load = [&](Vec<VW>(&buf)[kSlots], uint32_t R, uint32_t end) {
        const uint32_t t = fastdiv(R, p.div_hl);
        const uint32_t h = R - t * p.Hl;
        if constexpr (block_tab_ring<kCopy, kNF>()) {
            if (R < end && t != t_loaded) {  // the compute side sees the same tokens in the same order
                const float* tab = p.table + (size_t(r) * p.Sl + t) * kRowFloats + dv * (2 * NP);
                const uint32_t slot = n_loaded % kTabSlots;
                if (tab_ok(tab)) {
#pragma unroll
                    for (int k = 0; k < kCs; ++k) tab_cp16(ring_at(slot, k), tab + 4 * k);
                }
                t_loaded = t;
                ++n_loaded;
            }
            tab_commit();  // one group per load call, possibly empty
        }
#pragma unroll
        for (int x = 0; x < kSlots; ++x) {
            if constexpr (kNF > 0) {  // masked rows still go through the row reduction
#pragma unroll
                for (int k = 0; k < NP; ++k) buf[x].w[k] = 0u;
            }
            if (R < end) {
                const uint8_t* row = src[x] + int64_t(t) * p.s_t[x] + int64_t(h) * p.s_h[x];
                if (src_ok(row, x, r)) buf[x] = ld_lane(row, x);
            }
        }
    };
    auto compute_store = [&](Vec<VW>(&buf)[kSlots], uint32_t R, uint32_t end) {
        const bool valid = R < end;
        const uint32_t t = fastdiv(R, p.div_hl);
        const uint32_t h = R - t * p.Hl;
        if constexpr (kNF > 0) {
            if (valid && t != t_cached) {
                if constexpr (block_tab_ring<kCopy, kNF>()) {
                    tab_wait<kDepth - 1>();  // this row's load call was kDepth calls ago
                    const uint32_t slot = n_read % kTabSlots;
#pragma unroll
                    for (int k = 0; k < kCs; ++k) cs[k] = tab_lds(ring_at(slot, k));
                    ++n_read;
                } else {
                    const float* tab = tab_lane + size_t(t) * kRowFloats;
                    if (tab_ok(tab)) {
#pragma unroll
                        for (int k = 0; k < kCs; ++k) cs[k] = ld_table(tab + 4 * k);
                    }
                    if constexpr (!kStream) {
                        if (t + 1 < p.Sl) asm volatile("prefetch.global.L1 [%0];" ::"l"(tab + kRowFloats));
                    }
                }
                t_cached = t;
            }
            // every lane runs the row reductions (they shuffle); only valid rows are written.
            // Q/K only: both rows as fp32 pairs (video DiT 231.7 against 247.7 us with
            // the ring alone).  V+Q+K one unit at a time: Q and K share the cross-lane
            // work (311.5 against 316.1 us); streamed V+Q+K launches keep the per-row
            // form (the FLUX-like scatter 29.9-31.0 us with the shared form, 29.6 without)
            if constexpr (kNF == 2 && kCopy == 0) {
                norm_rope_qk<kF, kLanes, NP, kNeox>(buf[0].w, buf[1].w, wqk_all[dv], cs, p.eps, &redo);
            } else if constexpr (kNF == 2 && kCopy == 1 && !kStream) {
                norm_rope_pair<kF, kLanes, NP, kNeox>(buf[kCopy].w, buf[kCopy + 1].w, w(0), w(1), cs, p.eps, &redo);
            } else {
#pragma unroll
                for (int f = 0; f < kNF; ++f) fused_row(std::false_type{}, buf[kCopy + f].w, f);
            }
        }
        if (valid) {  // the scatter targets of one launch share their strides (slot 0's)
            const int64_t off = int64_t(t) * p.d_t[0] + int64_t(h) * p.d_h[0];
#pragma unroll
            for (int x = 0; x < kSlots; ++x)
                if (dst_ok(dst[x] + off, x, g_st)) st_lane(dst[x] + off, x, buf[x]);
        }
    };
    Vec<VW> bufs[kDepth][kSlots];
    if constexpr (kStream) {
        // Each row group walks the rows of all its units as one stream: during the
        // last pipeline pass of a unit its loads already fetch the first rows of the
        // group's next unit, so the loads of a new unit overlap the arithmetic of the
        // one before.  (g, r, b) and src then hold the unit being loaded, dst the
        // unit being stored.
        uint32_t u = blockIdx.x;  // the grid never exceeds the unit count
        Span ld = locate(u), st = ld;
        set_src();
        set_dst();
#pragma unroll
        for (int d = 0; d < kDepth; ++d) load(bufs[d], ld.beg + d, ld.end);
#pragma unroll 1
        for (;;) {
#pragma unroll 1
            for (uint32_t j = 0; j < st.slots; j += kDepth) {
                uint32_t ld_row = ld.beg + j + kDepth;
                if (j + kDepth >= st.slots) {  // last pass: load the next unit's first rows
                    const uint32_t un = u + gridDim.x;
                    if (un < p.n_units) {
                        ld = locate(un);
                        set_src();
                    } else {
                        ld.beg = ld.end = 0;  // nothing left: the loads below are masked
                    }
                    ld_row = ld.beg;
                }
#pragma unroll
                for (int d = 0; d < kDepth; ++d) {
                    compute_store(bufs[d], st.beg + j + d, st.end);
                    load(bufs[d], ld_row + d, ld.end);
                }
            }
            u += gridDim.x;
            if (u >= p.n_units) break;
            st = ld;
            set_dst();
        }
    } else {
        // one unit at a time: its rows are loaded, computed and stored before the
        // next unit's first loads
#pragma unroll 1
        for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const Span sp = locate(u);
            set_src();
            set_dst();
#pragma unroll
            for (int d = 0; d < kDepth; ++d) load(bufs[d], sp.beg + d, sp.end);
#pragma unroll 1
            for (uint32_t R = sp.beg; R < sp.beg + sp.slots; R += kDepth) {
#pragma unroll
                for (int d = 0; d < kDepth; ++d) {
                    compute_store(bufs[d], R + d, sp.end);
                    load(bufs[d], R + d + kDepth, sp.end);
                }
            }
        }
    }
    if constexpr (kNF > 0) {
        if constexpr (block_tab_ring<kCopy, kNF>()) tab_wait<0>();
        // A row whose sum of squares was not finite (an element of magnitude >=
        // 2^64, an infinite one or a NaN) was stored with the fast mean.  If the
        // CTA met one, every row group walks its rows of the fused slots once
        // more, one row at a time, with the complete mean; each row is rewritten
        // by the lanes that stored it, after their first store.
        __syncthreads();
        if (redo) {
#pragma unroll 1
            for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
                const Span sp = locate(u);
                set_src();
                set_dst();
#pragma unroll 1
                for (uint32_t R = sp.beg; R < sp.beg + sp.slots; ++R) {
                    const bool valid = R < sp.end;
                    const uint32_t t = fastdiv(R, p.div_hl);
                    const uint32_t h = R - t * p.Hl;
                    if (valid && t != t_cached) {
                        const float* tab = tab_lane + size_t(t) * kRowFloats;
                        if (tab_ok(tab)) {
#pragma unroll
                            for (int k = 0; k < kCs; ++k) cs[k] = ld_table(tab + 4 * k);
                        }
                        t_cached = t;
                    }
#pragma unroll
                    for (int f = 0; f < kNF; ++f) {
                        constexpr int x0 = kCopy;
                        Vec<VW> v;
#pragma unroll
                        for (int k = 0; k < NP; ++k) v.w[k] = 0u;
                        const uint8_t* srow = src[x0 + f] + int64_t(t) * p.s_t[x0 + f] + int64_t(h) * p.s_h[x0 + f];
                        uint8_t* drow = dst[x0 + f] + int64_t(t) * p.d_t[0] + int64_t(h) * p.d_h[0];
                        if (valid && src_ok(srow, x0 + f, r)) v = ld_lane(srow, x0 + f);
                        fused_row(std::true_type{}, v.w, f);
                        if (valid && dst_ok(drow, x0 + f, g)) st_lane(drow, x0 + f, v);
                    }
                }
            }
        }
    }
}

template <Fused kF, int kLanes, int kCopy, int kNF, bool kNeox, bool kStream, bool kV16>
cudaError_t launch_block_as(const RelayoutParams& p, cudaStream_t stream) {
    auto* kernel = block_kernel<kF, kLanes, kCopy, kNF, kNeox, kStream, kV16>;
    constexpr size_t kSmem = block_tab_smem<kCopy, kNF>();
    if constexpr (kSmem > 0) {
        // per device: the opt-in to more than 48 KiB of dynamic shared memory
        // (setting it twice is harmless)
        static std::atomic<bool> attr_done[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= 64 || !attr_done[dev].load()) {
            const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_done[dev].store(true);
        }
    }
    static std::atomic<int> blocks_per_sm{0};  // same for every device of one architecture
    if (blocks_per_sm.load() == 0) {
        int bps = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, kThreads, kSmem);
        if (e != cudaSuccess) return e;
        blocks_per_sm.store(bps > 0 ? bps : 1);
    }
    const int64_t want = int64_t(block_device_sms()) * blocks_per_sm.load();
    const unsigned grid = unsigned(want < int64_t(p.n_units) ? want : int64_t(p.n_units));
    return launch_overlapped(kernel, grid, kThreads, kSmem, stream, p);
}

template <Fused kF, int kLanes, int kCopy, int kNF, bool kNeox, bool kV16>
cudaError_t launch_block(const RelayoutParams& p, cudaStream_t stream) {
    if constexpr (kCopy == 1 && kNF == 2 && TFU_BLOCK_STREAM) {
        // rounds of units = units / resident CTAs
        const uint64_t resident = uint64_t(block_device_sms()) * block_min_blocks<kCopy, kNF>();
        if (p.n_units > uint64_t(TFU_STREAM_MAX_ROUNDS) * resident)
            return launch_block_as<kF, kLanes, kCopy, kNF, kNeox, false, kV16>(p, stream);
    }
    constexpr bool kStreamed = TFU_BLOCK_STREAM != 0;
    return launch_block_as<kF, kLanes, kCopy, kNF, kNeox, kStreamed, kV16>(p, stream);
}

template <Fused kF, int kCopy, int kNF, bool kNeox, bool kV16>
cudaError_t launch_block_lanes(const RelayoutParams& p, cudaStream_t stream) {
    switch (p.vpr) {  // lanes per head row = D * esize / 32
        case 2: return launch_block<kF, 2, kCopy, kNF, kNeox, kV16>(p, stream);
        case 4: return launch_block<kF, 4, kCopy, kNF, kNeox, kV16>(p, stream);
        case 8: return launch_block<kF, 8, kCopy, kNF, kNeox, kV16>(p, stream);
        case 16: return launch_block<kF, 16, kCopy, kNF, kNeox, kV16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <Fused kF, bool kNeox, bool kV16>
cudaError_t launch_block_fused(const RelayoutParams& p, cudaStream_t stream) {
    const uint32_t n_copy = (p.fused_mask & 1u) ? 0u : 1u;  // V (unfused) can only be slot 0
    const uint32_t nf = p.nx - n_copy;
    if (nf < 1 || nf > 2 || p.fused_mask != ((1u << nf) - 1u) << n_copy) return cudaErrorInvalidValue;
    if (n_copy)
        return nf == 2 ? launch_block_lanes<kF, 1, 2, kNeox, kV16>(p, stream)
                       : launch_block_lanes<kF, 1, 1, kNeox, kV16>(p, stream);
    return nf == 2 ? launch_block_lanes<kF, 0, 2, kNeox, kV16>(p, stream)
                   : launch_block_lanes<kF, 0, 1, kNeox, kV16>(p, stream);
}

template <Fused kF, bool kV16>
cudaError_t launch_block_style(const RelayoutParams& p, cudaStream_t stream) {
    if (!p.table) return cudaErrorInvalidValue;
    return p.rope_neox ? launch_block_fused<kF, true, kV16>(p, stream) : launch_block_fused<kF, false, kV16>(p, stream);
}

}  // namespace
}  // namespace tfu
