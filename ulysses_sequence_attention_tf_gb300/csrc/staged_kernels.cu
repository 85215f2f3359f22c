// staged_kernels.cu -- shared-memory-staged bulk-copy relayout kernel for sm_103a
// (pure relayouts: copy scatters and gathers).
//
// Same computation as the copy path of relayout_kernels.cu (TeleFuser docs,
// "Communication Architecture", "Sequence Parallel Communication / Ulysses"),
// organised around the Blackwell bulk-copy engine instead of per-lane loads:
//
//  * Persistent grid, one CTA (one warp) per SM.  The warp issues
//    cp.async.bulk global->shared loads for a unit (a row range of one plane,
//    <= 64 KiB, see tma_plan.h) into a ring of shared-memory stages (six of
//    32 KiB, two units ahead, or three of 64 KiB, one ahead, as the planner
//    sized the units), each completing on the stage's mbarrier with a transaction count;
//    it then issues the unit's bulk shared->global stores and reuses a stage
//    only after the stores' reads of it have finished
//    (cp.async.bulk.wait_group.read).  A unit's copies (one per contiguous run:
//    a token's head band, a head row, or the whole unit) are spread over the 32
//    lanes.  The data never enters registers.
//  * Every wait is bounded (clock64 budget).  A wait that gives up sets a bit in
//    a device status word and a shared abort flag; the kernel then drains the
//    copies it issued (bounded as well) and returns.  No trap, no endless loop.
#include <atomic>

#include "device_common.cuh"
#include "relayout.h"
#include "tma_plan.h"

// Tuning constants (compile-time; overridable with -D for measurement sweeps).
// The two rings of tma_plan.h: stages, and units loaded ahead of the store.
#ifndef TFU_STAGES
#define TFU_STAGES 3  // large ring: stages of kStageBytes (64 KiB)
#endif
#ifndef TFU_LAG
#define TFU_LAG 1  // large ring (two ahead measured lower with 64 KiB stages)
#endif
#ifndef TFU_STAGES_SMALL
#define TFU_STAGES_SMALL 6  // small ring: stages of kStageBytesSmall (32 KiB)
#endif
#ifndef TFU_LAG_SMALL
#define TFU_LAG_SMALL 2
#endif
namespace tfu {

// Reasons a bounded wait gave up (bitwise OR); zero when the library loads.
__device__ unsigned g_staged_status;

namespace {

using namespace dev;

constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

// Copy kernel: one data-movement warp and a ring of kStages stages of kStride bytes.
template <int kStagesR, int kLagR, uint32_t kStrideR>
struct CopyRing {
    static constexpr int kStages = kStagesR;
    static constexpr int kLag = kLagR;
    static constexpr uint32_t kStride = kStrideR;
    static constexpr size_t kSmem = size_t(kStages) * kStride + kStages * sizeof(uint64_t) + 16;
    static_assert(kLag >= 1 && kLag < kStages, "loads ahead must leave a stage for the store");
    static_assert(kSmem <= 227 * 1024, "stage ring exceeds shared memory");
};
using LargeRing = CopyRing<TFU_STAGES, TFU_LAG, kStageBytes>;
using SmallRing = CopyRing<TFU_STAGES_SMALL, TFU_LAG_SMALL, kStageBytesSmall>;

constexpr unsigned kStatusLoadWait = 1u;

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

// The data-movement loop: for each of this CTA's units k, load it kLag units
// ahead of its store.  kWarp = false: lane 0 alone issues every copy in order.
// kWarp = true: the whole warp runs the loop, and the copies of a unit made of
// many small runs are dealt out to the 32 lanes (for_each_run_lane: one copy per
// token band or row), so they are not bound by one lane's issue rate; `split_st`
// (uniform over the launch) says whether any unit deals out its stores, and only
// then do lanes other than 0 commit and wait on bulk groups.
// Barrier protocol: full[s] completes once per unit loaded into stage s (lane 0's
// arrive + the bytes of every lane's loads); the store of unit j waits
// full[j % kStages] for the phase of j (every active lane observes it), so every
// phase is observed in order; a lane that stores commits one bulk group per unit
// stored, and a stage is reloaded only after every store that last read it has
// finished reading (each storing lane's bulk wait_group.read, then a warp barrier).
template <Dir kDir, bool kWarp, class R>
__device__ void copy_dma_loop(const RelayoutParams& p, uint8_t* ring, uint64_t* full, volatile int* abort_flag,
                              uint32_t n_my, uint32_t lane, bool split_st) {
    const uint32_t rb = p.row_bytes;
    const uint32_t lanes = kWarp ? 32u : 1u;
    const bool stores = !kWarp || split_st || lane == 0;  // this lane may issue stores
    uint32_t issued = 0, consumed = 0;
    bool ok = true;
    for (uint32_t k = 0; ok && k < n_my + R::kLag; ++k) {
        if (k < n_my) {
            const uint32_t s = k % R::kStages;
            const Unit un = decode_unit<kDir>(p, blockIdx.x + k * gridDim.x);
            // stage s last held unit k - kStages, whose stores were committed
            // kStages - kLag - 1 groups ago: wait until they have read the stage
            if (k >= uint32_t(R::kStages) && stores) bulk_wait_read<R::kStages - R::kLag - 1>();
            if constexpr (kWarp) __syncwarp();
            uint8_t* stage = ring + size_t(s) * R::kStride;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], (un.R1 - un.R0) * rb);
            for_each_run_lane(un.R0, un.R1, p.Hl, un.pl.st, un.pl.sh, rb, lane, lanes, kLoadSplitRuns,
                              [&](uint32_t i, uint32_t n, int64_t off) {
                                  bulk_load(stage + size_t(i) * rb, un.pl.src + off, n * rb, &full[s]);
                              });
            issued = k + 1;
        }
        if (k >= uint32_t(R::kLag)) {
            const uint32_t j = k - R::kLag;
            const uint32_t s = j % R::kStages;
            const Unit un = decode_unit<kDir>(p, blockIdx.x + j * gridDim.x);
            ok = bounded_wait(&full[s], (j / R::kStages) & 1u, abort_flag, kStatusLoadWait);
            if constexpr (kWarp) ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint8_t* stage = ring + size_t(s) * R::kStride;
            for_each_run_lane(un.R0, un.R1, p.Hl, un.pl.dt, un.pl.dh, rb, lane, lanes, kStoreSplitRuns,
                              [&](uint32_t i, uint32_t n, int64_t off) {
                                  bulk_store(un.pl.dst + off, stage + size_t(i) * rb, n * rb);
                              });
            if (stores) bulk_commit();
            consumed = j + 1;
        }
    }
    bulk_wait_all();
    if (!ok) {  // drain the loads still in flight into this CTA's shared memory
        for (uint32_t j = consumed; j < issued; ++j) drain_wait(&full[j % R::kStages], (j / R::kStages) & 1u);
    }
    if constexpr (kWarp) __syncwarp();
}

// Pure relayout (copy scatter, gather): one warp, one ring, all units.  The warp
// deals out copies only when some slot's units are made of enough runs (the
// same decision for every CTA of the launch); otherwise lane 0 works alone.
template <Dir kDir, class R>
__global__ void __launch_bounds__(32, 1) copy_staged_kernel(const __grid_constant__ RelayoutParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(R::kStages) * R::kStride);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + R::kStages);
    const uint32_t lane = threadIdx.x;
    if (lane == 0) {
        for (int s = 0; s < R::kStages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    bool split_ld = false, split_st = false;
    for (uint32_t x = 0; x < p.nx; ++x) {
        split_ld = split_ld || unit_split_runs(p.rpu, p.Hl, p.s_t[x], p.s_h[x], p.row_bytes) >= kLoadSplitRuns;
        split_st = split_st || unit_split_runs(p.rpu, p.Hl, p.d_t[x], p.d_h[x], p.row_bytes) >= kStoreSplitRuns;
    }
    const uint32_t n_my = blockIdx.x < p.n_units ? (p.n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    grid_dependency_wait();  // the barriers above are shared memory; nothing global is touched before this
    if (!split_ld && !split_st) {
        if (lane == 0) copy_dma_loop<kDir, false, R>(p, smem, full, abort_flag, n_my, 0, false);
        return;
    }
    __syncwarp();  // the barriers are initialised before any lane uses them
    copy_dma_loop<kDir, true, R>(p, smem, full, abort_flag, n_my, lane, split_st);
}

template <Dir kDir, class R>
cudaError_t launch_copy(const RelayoutParams& p, cudaStream_t stream) {
    static std::atomic<bool> attr_done[64] = {};  // per device: the shared-memory opt-in (setting it twice is harmless)
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
        cudaError_t e = cudaFuncSetAttribute(copy_staged_kernel<kDir, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(R::kSmem));
        if (e != cudaSuccess) return e;
        attr_done[dev].store(true);
    }
    const unsigned grid = unsigned(p.n_units < uint32_t(sms) ? p.n_units : uint32_t(sms));
    return launch_overlapped(copy_staged_kernel<kDir, R>, grid, 32, R::kSmem, stream, p);
}

// The ring whose stages fit the planned units: the small one when a unit fits
// its stage, the large one otherwise (a unit never exceeds the large stage).
template <Dir kDir>
cudaError_t launch_copy_ring(const RelayoutParams& p, cudaStream_t stream) {
    if (uint64_t(p.rpu) * p.row_bytes > kStageBytes) return cudaErrorInvalidValue;
    if (uint64_t(p.rpu) * p.row_bytes <= kStageBytesSmall) return launch_copy<kDir, SmallRing>(p, stream);
    return launch_copy<kDir, LargeRing>(p, stream);
}

}  // namespace

cudaError_t launch_relayout_staged(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (p.rpu == 0 || fused != Fused::kNone) return cudaErrorInvalidValue;
    return dir == Dir::kGather ? launch_copy_ring<Dir::kGather>(p, stream) : launch_copy_ring<Dir::kScatter>(p, stream);
}

cudaError_t read_staged_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_staged_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_staged_status, &zero, sizeof(unsigned));
}

}  // namespace tfu
