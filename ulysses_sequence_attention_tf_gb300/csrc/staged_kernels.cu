// staged_kernels.cu -- shared-memory-staged relayout kernel for sm_103a.
//
// Same computation as relayout_kernels.cu (TeleFuser docs, "Communication
// Architecture", "Sequence Parallel Communication / Ulysses"; fused Q/K math of
// flashinfer PR #6332, "Assumptions / Operator math"), organised around the
// Blackwell bulk-copy engine instead of per-lane loads:
//
//  * Persistent grid, one CTA per SM.  Warp 0 is the data-movement warp: one
//    elected lane issues cp.async.bulk global->shared loads for a unit (a row
//    range of one plane, <= 32 KiB, see tma_plan.h; fused units also their
//    tokens' cos/sin rows) into a ring of shared-memory stages, a few units
//    ahead, each completing on the stage's mbarrier with a transaction count;
//    it then issues the unit's bulk
//    shared->global stores, and reuses a stage only after the store's reads of
//    it have finished (cp.async.bulk.wait_group.read).
//  * In the fused kernels the other warps (compute warps) follow the units in
//    order: for Q/K units (RMSNorm + RoPE) they rewrite the staged head rows in
//    place, fence the generic-proxy writes for the async proxy and arrive on the
//    stage's "done" mbarrier, which the store waits for; V units they only pass
//    on.  Staged data of V and plain units never enters registers.
//  * Every wait is bounded (clock64 budget).  A wait that gives up sets a bit in
//    a device status word and a shared abort flag; the kernel then drains the
//    copies it issued (bounded as well) and returns.  No trap, no endless loop.
#include "device_common.cuh"
#include "relayout.h"
#include "tma_plan.h"

// Tuning constants (compile-time; overridable with -D for measurement sweeps).
#ifndef TFU_STAGES
#define TFU_STAGES 6  // copy kernels: stages of 32 KiB
#endif
#ifndef TFU_LAG
#define TFU_LAG 2  // copy kernels: units loaded ahead of the store
#endif
#ifndef TFU_FUSED_STAGES
#define TFU_FUSED_STAGES 4  // fused kernels: stages of 32 KiB payload + 16 KiB cos/sin rows
#endif
#ifndef TFU_FUSED_LAG
#define TFU_FUSED_LAG 2
#endif
#ifndef TFU_COMPUTE_WARPS
#define TFU_COMPUTE_WARPS 16
#endif
#ifndef TFU_COMPUTE_SLOTS
#define TFU_COMPUTE_SLOTS 1
#endif

namespace tfu {

// Reasons a bounded wait gave up (bitwise OR); zero when the library loads.
__device__ unsigned g_staged_status;

namespace {

using namespace dev;

constexpr int kComputeWarps = TFU_COMPUTE_WARPS;
constexpr int kSlots = TFU_COMPUTE_SLOTS;  // row groups a compute warp works on at once
constexpr int kStagedThreads = 32 * (1 + kComputeWarps);
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

// Stage ring of one kernel configuration: copy kernels stage payload only; fused
// kernels also stage the unit's cos/sin rows behind the payload.
template <bool kFusedCfg>
struct Ring {
    static constexpr int kStages = kFusedCfg ? TFU_FUSED_STAGES : TFU_STAGES;
    static constexpr int kLag = kFusedCfg ? TFU_FUSED_LAG : TFU_LAG;
    static constexpr uint32_t kTable = kFusedCfg ? kStageTableBytes : 0u;
    static constexpr uint32_t kStride = kStageBytes + kTable;  // bytes per stage
    static constexpr size_t kSmem = size_t(kStages) * kStride + 2 * kStages * sizeof(uint64_t) + 16;
    static_assert(kLag >= 1 && kLag < kStages, "loads ahead must leave a stage for the store");
    static_assert(kSmem <= 227 * 1024, "stage ring exceeds shared memory");
};

constexpr unsigned kStatusLoadWait = 1u, kStatusComputeWait = 2u, kStatusWarpLoadWait = 4u;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(smem_src)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Wait for the phase of `bar` with parity `parity`.  Gives up (returns false)
// when the shared abort flag is raised or after kWaitCycles; a give-up records
// `code` in the status word and raises the abort flag.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned code) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kWaitCycles) {
                atomicOr(&g_staged_status, code);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Drain wait after an abort: same budget, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) return;
    }
}

struct Unit {
    Plane pl;
    uint32_t R0, R1;  // plane rows [R0, R1)
    bool fused;
};

// unit u = c * n_planes + q: row chunk c of plane q (chunk-major, as in the
// register kernel, so CTAs running together share token blocks)
template <Dir kDir>
__device__ __forceinline__ Unit decode_unit(const RelayoutParams& p, uint32_t u) {
    const uint32_t c = fastdiv(u, p.div_planes);
    const uint32_t q = u - c * p.n_planes;
    Unit un;
    un.pl = decode_plane<kDir>(p, q);
    un.R0 = c * p.rpu;
    un.R1 = min(un.R0 + p.rpu, p.plane_rows);
    un.fused = ((p.fused_mask >> un.pl.x) & 1u) != 0;
    return un;
}

// The data-movement lane: loads kLag units ahead, stores behind.
//
// Barrier protocol (every phase of every stage barrier is observed in order, so
// a parity wait can never match a phase that is one use ahead or behind):
//  * full[s] completes once per unit loaded into stage s (arrive + bytes).
//  * With compute warps (fused kernels), every compute warp waits full[s] for
//    every unit in order -- rewriting the rows of fused units only -- and then
//    arrives on done[s]; the store waits done[s].  Without compute warps the
//    store waits full[s].
//  * A stage is reloaded only after the previous store's reads of it finished
//    (bulk wait_group.read), and that store waited for every compute warp.
// Fused units also load their tokens' cos/sin rows behind the payload.
template <Dir kDir, bool kHasCompute>
__device__ void dma_loop(const RelayoutParams& p, uint8_t* stages, uint64_t* full, uint64_t* done,
                         volatile int* abort_flag, uint32_t n_my) {
    using R = Ring<kHasCompute>;
    const uint32_t rb = p.row_bytes;
    const uint32_t table_row_bytes = rb * 2;  // D fp32 values per token row (16-bit payload)
    uint32_t issued = 0, consumed = 0;
    bool ok = true;
    for (uint32_t k = 0; ok && k < n_my + R::kLag; ++k) {
        if (k < n_my) {
            const uint32_t s = k % R::kStages;
            const Unit un = decode_unit<kDir>(p, blockIdx.x + k * gridDim.x);
            // stage s last held unit k - kStages, whose store was committed
            // kStages - kLag - 1 groups ago: wait until it has read the stage
            if (k >= uint32_t(R::kStages)) bulk_wait_read<R::kStages - R::kLag - 1>();
            uint8_t* stage = stages + size_t(s) * R::kStride;
            uint32_t bytes = (un.R1 - un.R0) * rb;
            uint32_t t0 = 0, t1 = 0;
            const bool with_table = kHasCompute && un.fused;
            if (with_table) {
                unit_tokens(un.R0, un.R1, p.Hl, t0, t1);
                bytes += (t1 - t0 + 1) * table_row_bytes;
            }
            mbar_arrive_expect_tx(&full[s], bytes);
            for_each_run(un.R0, un.R1, p.Hl, un.pl.st, un.pl.sh, rb, [&](uint32_t i, uint32_t n, int64_t off) {
                bulk_load(stage + size_t(i) * rb, un.pl.src + off, n * rb, &full[s]);
            });
            if (with_table)
                bulk_load(stage + kStageBytes, p.table + size_t(un.pl.pos0 + t0) * (table_row_bytes / 4),
                          (t1 - t0 + 1) * table_row_bytes, &full[s]);
            issued = k + 1;
        }
        if (k >= uint32_t(R::kLag)) {
            const uint32_t j = k - R::kLag;
            const uint32_t s = j % R::kStages;
            const uint32_t parity = (j / R::kStages) & 1u;
            const Unit un = decode_unit<kDir>(p, blockIdx.x + j * gridDim.x);
            if constexpr (kHasCompute) {
                ok = bounded_wait(&done[s], parity, abort_flag, kStatusComputeWait);
            } else {
                ok = bounded_wait(&full[s], parity, abort_flag, kStatusLoadWait);
            }
            if (!ok) break;
            const uint8_t* stage = stages + size_t(s) * R::kStride;
            for_each_run(un.R0, un.R1, p.Hl, un.pl.dt, un.pl.dh, rb, [&](uint32_t i, uint32_t n, int64_t off) {
                bulk_store(un.pl.dst + off, stage + size_t(i) * rb, n * rb);
            });
            bulk_commit();
            consumed = j + 1;
        }
    }
    bulk_wait_all();
    if (!ok) {  // drain the loads still in flight into this CTA's shared memory
        for (uint32_t j = consumed; j < issued; ++j) drain_wait(&full[j % R::kStages], (j / R::kStages) & 1u);
    }
}

// A compute warp: for every unit, wait for its load; for fused units normalise
// and rotate the head rows in place (kLanes lanes x 32 bytes per row) with the
// staged cos/sin rows; then signal the stage done.
template <Fused kF, int kLanes>
__device__ void compute_loop(const RelayoutParams& p, uint8_t* stages, uint64_t* full, uint64_t* done,
                             volatile int* abort_flag, uint32_t n_my, uint32_t cw, uint32_t lane) {
    using R = Ring<true>;
    constexpr int NP = 8;                         // element pairs in a lane's 32 bytes
    constexpr uint32_t kRowsPerIter = 32 / kLanes;
    constexpr uint32_t kRowFloats = kLanes * 16;  // D floats per table row
    constexpr uint32_t kRowBytes = kLanes * 32;
    constexpr uint32_t kGroupStride = kComputeWarps * kRowsPerIter;  // rows between a warp's row groups
    const uint32_t dv = lane % kLanes;
    for (uint32_t k = 0; k < n_my; ++k) {
        const Unit un = decode_unit<Dir::kScatter>(p, blockIdx.x + k * gridDim.x);
        const uint32_t s = k % R::kStages;
        if (!bounded_wait(&full[s], (k / R::kStages) & 1u, abort_flag, kStatusWarpLoadWait)) return;
        if (!un.fused) {  // V / plain unit: nothing to rewrite, just pass the stage on
            __syncwarp();
            if (lane == 0) mbar_arrive(&done[s]);
            continue;
        }
        uint8_t* stage = stages + size_t(s) * R::kStride;
        const float* tab = reinterpret_cast<const float*>(stage + kStageBytes) + dv * 16;
        const uint32_t t_first = fastdiv(un.R0, p.div_hl);
        uint32_t wpk[NP];
        {
            const uint4* wp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.weight[un.pl.x]) + dv * 32);
            const uint4 w0 = __ldg(wp), w1 = __ldg(wp + 1);
            wpk[0] = w0.x; wpk[1] = w0.y; wpk[2] = w0.z; wpk[3] = w0.w;
            wpk[4] = w1.x; wpk[5] = w1.y; wpk[6] = w1.z; wpk[7] = w1.w;
        }
        const uint32_t n_rows = un.R1 - un.R0;
        // kSlots independent row groups per iteration (their dependent chains interleave)
#pragma unroll 1
        for (uint32_t base = cw * kRowsPerIter; base < n_rows; base += kSlots * kGroupStride) {
            uint32_t xw[kSlots][NP];
            bool valid[kSlots];
#pragma unroll
            for (int sl = 0; sl < kSlots; ++sl) {
                const uint32_t i = base + sl * kGroupStride + lane / kLanes;
                valid[sl] = i < n_rows;
#pragma unroll
                for (int j = 0; j < NP; ++j) xw[sl][j] = 0u;
                if (valid[sl]) {
                    const uint4* rowp = reinterpret_cast<const uint4*>(stage + size_t(i) * kRowBytes + dv * 32);
                    const uint4 a = rowp[0], b = rowp[1];
                    xw[sl][0] = a.x; xw[sl][1] = a.y; xw[sl][2] = a.z; xw[sl][3] = a.w;
                    xw[sl][4] = b.x; xw[sl][5] = b.y; xw[sl][6] = b.z; xw[sl][7] = b.w;
                }
            }
#pragma unroll
            for (int sl = 0; sl < kSlots; ++sl) {
                const uint32_t i = base + sl * kGroupStride + lane / kLanes;
                const uint32_t t = fastdiv(un.R0 + i, p.div_hl) - t_first;  // token within the unit
                // every lane runs the row reduction (it shuffles); only valid rows are written
                norm_rope_lane<kF, kLanes, NP, true>(xw[sl], wpk, tab + size_t(t) * kRowFloats, valid[sl], p.eps);
            }
#pragma unroll
            for (int sl = 0; sl < kSlots; ++sl) {
                const uint32_t i = base + sl * kGroupStride + lane / kLanes;
                if (valid[sl]) {
                    uint4* rowp = reinterpret_cast<uint4*>(stage + size_t(i) * kRowBytes + dv * 32);
                    rowp[0] = make_uint4(xw[sl][0], xw[sl][1], xw[sl][2], xw[sl][3]);
                    rowp[1] = make_uint4(xw[sl][4], xw[sl][5], xw[sl][6], xw[sl][7]);
                }
            }
        }
        fence_proxy_async_smem();  // make the rewritten rows visible to the bulk store
        __syncwarp();
        if (lane == 0) mbar_arrive(&done[s]);
    }
}

template <Dir kDir, Fused kF, int kLanes>
__global__ void __launch_bounds__(kStagedThreads, 1) staged_kernel(const __grid_constant__ RelayoutParams p) {
    using R = Ring<kF != Fused::kNone>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(R::kStages) * R::kStride);
    uint64_t* done = full + R::kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(done + R::kStages);
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < R::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&done[s], kComputeWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const uint32_t n_my = blockIdx.x < p.n_units ? (p.n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (warp == 0) {
        if (lane == 0) dma_loop<kDir, kF != Fused::kNone>(p, stages, full, done, abort_flag, n_my);
        return;
    }
    if constexpr (kF != Fused::kNone) compute_loop<kF, kLanes>(p, stages, full, done, abort_flag, n_my, warp - 1, lane);
}

int staged_device_sms(int* dev_out) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *dev_out = dev;
    return sms > 0 ? sms : 1;
}

template <Dir kDir, Fused kF, int kLanes>
cudaError_t launch_staged_one(const RelayoutParams& p, cudaStream_t stream) {
    using R = Ring<kF != Fused::kNone>;
    static bool attr_done[64] = {};  // per device: the shared-memory opt-in
    int dev = 0;
    const int sms = staged_device_sms(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(staged_kernel<kDir, kF, kLanes>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(R::kSmem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const unsigned grid = unsigned(p.n_units < uint32_t(sms) ? p.n_units : uint32_t(sms));
    staged_kernel<kDir, kF, kLanes><<<grid, kStagedThreads, R::kSmem, stream>>>(p);
    return cudaGetLastError();
}

template <Fused kF>
cudaError_t launch_staged_fused(const RelayoutParams& p, cudaStream_t stream) {
    switch (p.row_bytes / 32) {  // lanes per head row
        case 2: return launch_staged_one<Dir::kScatter, kF, 2>(p, stream);
        case 4: return launch_staged_one<Dir::kScatter, kF, 4>(p, stream);
        case 8: return launch_staged_one<Dir::kScatter, kF, 8>(p, stream);
        case 16: return launch_staged_one<Dir::kScatter, kF, 16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_relayout_staged(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.rpu == 0) return cudaErrorInvalidValue;
    if (dir == Dir::kGather) {
        if (fused != Fused::kNone) return cudaErrorInvalidValue;
        return launch_staged_one<Dir::kGather, Fused::kNone, 0>(p, stream);
    }
    if (fused != Fused::kNone && p.row_bytes % 32 != 0) return cudaErrorInvalidValue;
    switch (fused) {
        case Fused::kNone: return launch_staged_one<Dir::kScatter, Fused::kNone, 0>(p, stream);
        case Fused::kBF16: return launch_staged_fused<Fused::kBF16>(p, stream);
        case Fused::kFP16: return launch_staged_fused<Fused::kFP16>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t read_staged_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_staged_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_staged_status, &zero, sizeof(unsigned));
}

}  // namespace tfu
