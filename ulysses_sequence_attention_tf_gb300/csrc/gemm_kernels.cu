// gemm_kernels.cu -- the QKV projection in front of the Ulysses exchange on the
// 5th-generation tensor cores (sm_103a), with the Q/K RMSNorm + RoPE and the
// scatter into the final-layout targets in the epilogue.
//
// What is computed (flashinfer PR #6332 commit message, "Description": the BF16
// QKV projection, per-head RMSNorm of Q and K, interleaved RoPE from a per-token
// cos/sin table and the head exchange in one call, the exchange stored straight
// from the GEMM epilogue; "Assumptions / Operator math": projection -> QK-norm ->
// RoPE, BF16 operands and outputs).  For shard r, token row m = b*Sl + t,
// feature n:
//     Y[m, n] = round_bf16( sum_k X_r[m, k] * W[n, k] )     (fp32 accumulation)
// Y's feature blocks [0, HD), [HD, 2HD), [2HD, 3HD) are Q, K, V; head h of a block
// lands in head group g = h / Hl at target row r*Sl + t, head h % Hl; Q and K rows
// then get the RMSNorm + RoPE of tf_ulysses.h at global position p = r*Sl + t.
//
// Two forms of one design.  The default, qkv_gemm_pair_kernel (below), runs CTA
// pairs on the 2-SM MMA over 256 x 256 tiles; the single-CTA form described here
// is the fallback (build option TFU_GEMM_PAIR=0, or no pair cluster fits) and
// shares its epilogue, raster and failure handling.
// Single-CTA form (persistent: one CTA of 192 threads per SM walks 128 x 256 output tiles):
//  * warp 0, one lane: TMA producer.  Each stage holds a 128 x 64 tile of X and a
//    256 x 64 tile of W (bf16, 128-byte swizzle), loaded with
//    cp.async.bulk.tensor onto the stage's mbarrier (transaction bytes).
//  * warp 1: allocates 512 TMEM columns (two 128 x 256 fp32 accumulators, so the
//    epilogue of one tile overlaps the MMAs of the next), and one lane issues
//    tcgen05.mma (kind::f16, M = 128, N = 256, K = 16, four per stage) from
//    shared-memory descriptors, committing each stage back to the producer and
//    each finished accumulator to the epilogue, which releases it when read.
//  * warps 2-5: the epilogue.  Warp w reads TMEM lanes 32*(w%4).. with
//    tcgen05.ld, so each thread holds one token row: per head, 128 fp32
//    accumulators are rounded to bf16 (the projection's output), and for Q/K
//    normalised (exact sum of squares, in-thread), scaled and rotated, then
//    stored as one 256-byte row of the head-group target.
//  * Tiles are rasterised in passes over n_group column tiles, so the weight
//    columns of a pass stay in L2 while every row tile streams past.
//  * Every mbarrier wait is bounded; a wait that gives up records a status bit,
//    raises a shared abort flag, and the CTA drains its copies and MMAs (bounded)
//    and frees its TMEM before returning.
#include <atomic>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "gemm.h"

namespace tfu {

__device__ unsigned g_gemm_status;

namespace {

using namespace dev;

constexpr int kStagesG = 4;                            // stages of 48 KiB (a fifth does not fit)
constexpr uint32_t kRowBytesG = kGemmBK * 2;          // one operand row of a stage: 128 bytes
constexpr uint32_t kABytes = kGemmBM * kRowBytesG;     // 16 KiB
constexpr uint32_t kBBytes = kGemmBN * kRowBytesG;     // 32 KiB
constexpr uint32_t kStageBytesG = kABytes + kBBytes;
constexpr int kThreadsG = 192;
constexpr uint32_t kTmemCols = 256;
constexpr size_t kSmemG = size_t(kStagesG) * kStageBytesG + 256 + 1024;  // stages, barriers, alignment slack
constexpr long long kWaitCyclesG = 4000000000LL;                           // ~2 s at 2 GHz
constexpr unsigned kStatusWait = 1u;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kGemmBN >> 3) << 17) |
                            (uint32_t(kGemmBM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// kCS: acquire at cluster scope (arrivals and copies of the other CTA of a pair).
template <bool kCS = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if constexpr (kCS) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    }
    return ok != 0;
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Wait for the phase of `bar` with parity `parity`; false if the abort flag is
// raised or the budget runs out (then records the status and raises the flag,
// and also the flag at shared::cluster address `peer_flag` of the other CTA of a
// pair when it is not 0).
template <bool kCS = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           long long budget = kWaitCyclesG, uint32_t peer_flag = 0) {
    if (mbar_try_wait<kCS>(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait<kCS>(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > budget) {
                atomicOr(&g_gemm_status, kStatusWait);
                *abort_flag = 1;
                if (peer_flag) asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_flag), "r"(1u) : "memory");
                return false;
            }
        }
    }
}

// The same without the abort flag (draining after an abort): bounded only.
template <bool kCS = false>
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait<kCS>(bar, parity)) {
        if (clock64() - t0 > kWaitCyclesG) return;
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_result), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, one M=128 x N=256 x K=16 step.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 128 bytes with the 128-byte swizzle, 8-row groups 1024 bytes apart: start
// address >> 4 (bits 0-13), leading byte offset (unused by this layout, 1) at
// bits 16-29, stride byte offset at bits 32-45, descriptor version 1 at bits
// 46-47, base offset 0 (tiles are aligned to the swizzle pattern), swizzle mode
// 2 (128-byte) at bits 61-63.  A K step of 16 elements advances the start by 32
// bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    constexpr uint64_t kMode = 2;
    return uint64_t((smem_addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t((8 * kRowBytesG) >> 4) << 32) |
           (uint64_t(1) << 46) | (kMode << 61);
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane (warp-collective:
// the warp is reconverged first).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- epilogue
// 16 packed bf16 pairs of 32 accumulator columns: the projection's output rounding.
__device__ __forceinline__ void round_chunk(const uint32_t (&r)[32], uint32_t (&z)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = pack2<Fused::kBF16>(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
}

// y = round(x * inv), z = round(y * w) for 16 pairs; wp: the chunk's weight pairs.
__device__ __forceinline__ void scale_chunk(uint32_t (&z)[16], float inv, const uint32_t* wp) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float a, b;
        unpack2<Fused::kBF16>(z[i], a, b);
        z[i] = mul2<Fused::kBF16>(pack2<Fused::kBF16>(__fmul_rn(a, inv), __fmul_rn(b, inv)), __ldg(wp + i));
    }
}

__device__ __forceinline__ void store_chunk(uint8_t* dst, const uint32_t (&z)[16]) {
    Vec<32> v0, v1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v0.w[k] = z[k];
        v1.w[k] = z[8 + k];
    }
    st_stream<32>(dst, v0);
    st_stream<32>(dst + 32, v1);
}

// One head of this thread's token row, TMEM columns [taddr, taddr + 128): the
// projection rounded to bf16, then for a Q/K head the RMSNorm (exact in-thread
// sum of squares, first pass over TMEM), the bf16 weight scale and RoPE
// (interleaved pairs (2i, 2i+1), or half-split pairs (i, i + 64)) in a second
// pass, 32 columns (64 output bytes) at a time.  tcgen05.ld is warp-collective:
// every lane loads, only valid rows store.
template <bool kFusedT, bool kNeox>
__device__ __forceinline__ void epilogue_head(uint32_t taddr, bool valid, bool norm, const uint32_t* wpairs,
                                              const float* tab, float eps, uint8_t* dst_row) {
    if (!(kFusedT && norm)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32], z[16];
            tc_ld32(taddr + uint32_t(c * 32), r);
            tc_wait_ld();
            round_chunk(r, z);
            if (valid) store_chunk(dst_row + c * 64, z);
        }
        return;
    }
    constexpr float kInvD = 1.0f / kGemmHeadDim;
    // sum of squares of the rounded row (each value scaled by `scale`, a power of
    // two): hi + lo exact unless it overflows
    auto sumsq = [&](float scale, float& hi, float& lo) {
        hi = 0.f;
        lo = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32], z[16];
            tc_ld32(taddr + uint32_t(c * 32), r);
            tc_wait_ld();
            round_chunk(r, z);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float a, b, s, e;
                unpack2<Fused::kBF16>(z[i], a, b);
                a = __fmul_rn(a, scale);
                b = __fmul_rn(b, scale);
                two_sum(hi, __fmul_rn(a, a), s, e);  // squares of bf16 values are exact in fp32
                lo = __fadd_rn(lo, e);
                hi = s;
                two_sum(hi, __fmul_rn(b, b), s, e);
                lo = __fadd_rn(lo, e);
                hi = s;
            }
        }
    };
    float hi, lo;
    sumsq(1.0f, hi, lo);
    float ms = __fmul_rn(__fadd_rn(hi, lo), kInvD);
    // A sum that is not finite (an element of magnitude >= 2^64, an infinite one or
    // a NaN): the row scaled by 2^-96 (exact) gives the mean, scaled back by 2^192
    // in two exact steps (+inf when the mean exceeds the fp32 range).  TMEM loads
    // are warp-collective, so the warp rescans when any of its rows needs it.
    if (__any_sync(0xffffffffu, !(hi <= 3.40282347e38f))) {
        float hs, ls;
        sumsq(0x1p-96f, hs, ls);
        if (!(hi <= 3.40282347e38f))
            ms = hs <= 3.40282347e38f ? __fmul_rn(__fmul_rn(__fmul_rn(__fadd_rn(hs, ls), kInvD), 0x1p96f), 0x1p96f)
                                      : hs;
    }
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
    if constexpr (!kNeox) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {  // pairs 16c .. 16c + 15, table entries likewise
            uint32_t r[32], z[16];
            tc_ld32(taddr + uint32_t(c * 32), r);
            tc_wait_ld();
            round_chunk(r, z);  // rows past the end compute on zeros and store nothing
            scale_chunk(z, inv, wpairs + c * 16);
            const float4* t4 = reinterpret_cast<const float4*>(tab) + c * 8;  // two pairs per float4
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float4 cs = __ldg(t4 + i / 2);
                float a, b;
                unpack2<Fused::kBF16>(z[i], a, b);
                z[i] = pack2<Fused::kBF16>(__fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y)),
                                           __fadd_rn(__fmul_rn(a, cs.y), __fmul_rn(b, cs.x)));
                unpack2<Fused::kBF16>(z[i + 1], a, b);
                z[i + 1] = pack2<Fused::kBF16>(__fsub_rn(__fmul_rn(a, cs.z), __fmul_rn(b, cs.w)),
                                               __fadd_rn(__fmul_rn(a, cs.w), __fmul_rn(b, cs.z)));
            }
            if (valid) store_chunk(dst_row + c * 64, z);
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {  // columns 32c.. pair with 32c + 64..; entries 32c .. 32c + 31
            uint32_t r[32], zl[16], zh[16];
            tc_ld32(taddr + uint32_t(c * 32), r);
            tc_wait_ld();
            round_chunk(r, zl);
            tc_ld32(taddr + uint32_t(c * 32 + 64), r);
            tc_wait_ld();
            round_chunk(r, zh);
            scale_chunk(zl, inv, wpairs + c * 16);
            scale_chunk(zh, inv, wpairs + c * 16 + 32);
            const float4* t4 = reinterpret_cast<const float4*>(tab) + c * 16;  // entries 2i, 2i+1 per float4
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 cs = __ldg(t4 + i);
                float a0, a1, b0, b1;
                unpack2<Fused::kBF16>(zl[i], a0, a1);
                unpack2<Fused::kBF16>(zh[i], b0, b1);
                zl[i] = pack2<Fused::kBF16>(__fsub_rn(__fmul_rn(a0, cs.x), __fmul_rn(b0, cs.y)),
                                            __fsub_rn(__fmul_rn(a1, cs.z), __fmul_rn(b1, cs.w)));
                zh[i] = pack2<Fused::kBF16>(__fadd_rn(__fmul_rn(a0, cs.y), __fmul_rn(b0, cs.x)),
                                            __fadd_rn(__fmul_rn(a1, cs.w), __fmul_rn(b1, cs.z)));
            }
            if (valid) {
                store_chunk(dst_row + c * 64, zl);
                store_chunk(dst_row + c * 64 + 128, zh);
            }
        }
    }
}

// ---------------------------------------------------------------- the kernel
using Tile = GemmTile;

template <int kCluster>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, uint32_t t, uint32_t rank) {
    return gemm_tile<kCluster>(p.P, p.m_tiles, p.n_tiles, p.n_group, t, rank);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr uint32_t kAccBufs = 2;  // TMEM accumulators: the epilogue of tile i overlaps the MMAs of tile i+1

// Persistent: CTA c takes tiles c, c + gridDim.x, ...; the shared-memory stage
// ring and the two TMEM accumulators carry on from tile to tile.
template <bool kFusedT, bool kNeox>
__global__ void __launch_bounds__(kThreadsG, 1) qkv_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kStagesG) * kStageBytesG);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStagesG);
    const uint32_t acc_full0 = smem_u32(bars + 2 * kStagesG), acc_empty0 = smem_u32(bars + 2 * kStagesG + kAccBufs);
    const uint32_t mma_done = smem_u32(bars + 2 * kStagesG + 2 * kAccBufs);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStagesG + 2 * kAccBufs + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t cid = blockIdx.x, ctas = gridDim.x;
    const uint32_t units = p.P * p.m_tiles * p.n_tiles;
    const uint32_t KB = p.K / kGemmBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesG; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);  // the MMAs that read the stage release it
        }
        for (uint32_t a = 0; a < kAccBufs; ++a) {
            mbar_init(acc_full0 + 8 * a, 1);
            mbar_init(acc_empty0 + 8 * a, 4);  // one arrival per epilogue warp
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols * kAccBufs);
        tmem_relinquish();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: one continuous stream of k-blocks
        uint32_t q = 0;  // k-blocks issued by this CTA
        bool ok = true;
        for (uint32_t t = cid; ok && t < units; t += ctas) {
            const Tile tl = decode_tile<1>(p, t, 0);
            const CUtensorMap* mx = &p.tmap_x[tl.r];
            for (uint32_t kb = 0; kb < KB; ++kb, ++q) {
                const uint32_t s = q % kStagesG, use = q / kStagesG;
                if (use > 0 && !wait_phase(empty0 + 8 * s, (use - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t a = smem_u32(smem + size_t(s) * kStageBytesG);
                mbar_expect_tx(full0 + 8 * s, kStageBytesG);
                tma_load_2d(a, mx, int(kb * kGemmBK), int(tl.m_tile * kGemmBM), full0 + 8 * s);
                tma_load_2d(a + kABytes, &p.tmap_w, int(kb * kGemmBK), int(tl.n_tile * kGemmBN), full0 + 8 * s);
            }
        }
        // the last load issued into each stage has landed before the CTA exits
        for (uint32_t k = q > uint32_t(kStagesG) ? q - kStagesG : 0; k < q; ++k)
            drain_phase(full0 + 8 * (k % kStagesG), (k / kStagesG) & 1u);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        uint32_t q = 0, i = 0;
        bool ok = true;
        for (uint32_t t = cid; ok && t < units; t += ctas, ++i) {
            const uint32_t a = i % kAccBufs, u = i / kAccBufs;
            if (u > 0 && !wait_phase(acc_empty0 + 8 * a, (u - 1) & 1u, abort_flag)) break;  // epilogue drained it
            tc_fence_after();
            const uint32_t d = tmem + a * kTmemCols;
            for (uint32_t kb = 0; kb < KB; ++kb, ++q) {
                const uint32_t s = q % kStagesG, use = q / kStagesG;
                if (!wait_phase(full0 + 8 * s, use & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + size_t(s) * kStageBytesG);
#pragma unroll
                for (uint32_t kk = 0; kk < kGemmBK / 16; ++kk)
                    tc_mma(d, sw128_desc(sa + kk * 32), sw128_desc(sa + kABytes + kk * 32), (kb | kk) != 0);
                tc_commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
            }
            tc_commit(acc_full0 + 8 * a);  // the tile's accumulator is complete (or abandoned)
        }
        tc_commit(mma_done);
        drain_phase(mma_done, 0);  // every MMA of this CTA has completed
    } else if (warp >= 2) {
        // ---------------- epilogue
        const uint32_t quarter = warp & 3u;
        const uint32_t HD = p.H * kGemmHeadDim;
        uint32_t i = 0;
        for (uint32_t t = cid; t < units; t += ctas, ++i) {
            const uint32_t a = i % kAccBufs, u = i / kAccBufs;
            const bool ok = wait_phase(acc_full0 + 8 * a, u & 1u, abort_flag);
            tc_fence_after();
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;  // warp-uniform: TMEM loads are collective
            const Tile tl = decode_tile<1>(p, t, 0);
            const uint32_t m = tl.m_tile * kGemmBM + quarter * 32 + lane;
            const bool valid = tl.m_tile < p.m_tiles && m < p.rows;
            const uint32_t b = valid ? m / p.Sl : 0, tt = valid ? m - b * p.Sl : 0;
            const uint32_t pos = tl.r * p.Sl + tt;
#pragma unroll 1
            for (uint32_t j = 0; j < kGemmBN / kGemmHeadDim; ++j) {
                const uint32_t f = tl.n_tile * kGemmBN + j * kGemmHeadDim;
                const uint32_t sec = f / HD;
                const uint32_t h = (f - sec * HD) / kGemmHeadDim;
                const uint32_t g = h / p.Hl, hh = h - g * p.Hl;
                uint8_t* dst_row = p.dst[sec][g] + int64_t(b) * p.d_b + int64_t(pos) * p.d_t + int64_t(hh) * p.d_h;
                const bool norm = kFusedT && sec < 2;
                const uint32_t* wp = norm ? static_cast<const uint32_t*>(p.weight[sec]) : nullptr;
                const float* tab = norm ? p.table + size_t(pos) * kGemmHeadDim : nullptr;
                epilogue_head<kFusedT, kNeox>(tmem + a * kTmemCols + ((quarter * 32u) << 16) + j * kGemmHeadDim, valid,
                                              norm, wp, tab, p.eps, dst_row);
            }
            tc_fence_before();  // this warp's TMEM reads are done (tcgen05.wait::ld) before the release
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty0 + 8 * a);
        }
    }
    // teardown: every MMA has completed (warp 1 waited on mma_done) and every TMEM
    // read has finished before the columns are freed
    __syncwarp();  // the single-lane roles rejoin their warps before the CTA barrier
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols * kAccBufs);
    }
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
// The pair form of the projection: the two CTAs of a cluster compute one
// 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256), issued by the even CTA.
// Each CTA stages its own 128 rows of X and one 128-row half of the weight tile
// (the lower CTA the first half), so a stage is 32 KiB instead of 48 KiB and the
// ring holds more k-blocks; the MMA reads both CTAs' stages and writes each CTA's
// 128 rows x 256 columns into that CTA's TMEM, where its own epilogue reads them.
//  * both CTAs' loads complete on the even CTA's stage barrier (cp.async.bulk.tensor
//    .cta_group::2 signals a barrier of either CTA of the pair); the even CTA's
//    producer posts the transaction bytes of the whole pair;
//  * the MMA thread's commits arrive on both CTAs' stage and accumulator barriers
//    (multicast), so each producer refills its stage, and each epilogue starts, on
//    its own barriers;
//  * both CTAs' epilogue warps release an accumulator on the even CTA's barrier;
//  * TMEM is allocated and freed by one warp of each CTA together (cta_group::2).
#ifndef TFU_GEMM_PAIR_STAGES
#define TFU_GEMM_PAIR_STAGES 6
#endif
constexpr int kStagesP = TFU_GEMM_PAIR_STAGES;
constexpr uint32_t kBHalfBytes = kBBytes / 2;
constexpr uint32_t kStageBytesP = kABytes + kBHalfBytes;
constexpr size_t kSmemP = size_t(kStagesP) * kStageBytesP + 256 + 1024;
static_assert(kSmemP <= 232448, "the pair stage ring exceeds 227 KiB of shared memory");
// M = 256 (two CTAs of 128 rows), N = 256, otherwise as kIdesc.
constexpr uint32_t kIdescPair = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kGemmBN >> 3) << 17) |
                                (uint32_t((2 * kGemmBM) >> 4) << 24);

// shared::cluster address of the object at this CTA's shared address `local` in CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// Load into this CTA's shared memory; the transaction bytes complete on `bar`, a
// shared::cluster address of a barrier in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
#ifndef TFU_GEMM_HINTS
// 1: the pair's weight loads carry the L2 evict_last policy, so the weight columns
// of a raster pass outlive the streaming rows and targets in L2 (0: no policy).
#define TFU_GEMM_HINTS 1
#endif
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t smem_dst, const CUtensorMap* map, int x, int y,
                                                      uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_result), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T, one M=256 x N=256 x K=16 step.
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdescPair), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(bar),
                 "h"(mask)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

template <bool kFusedT, bool kNeox>
__global__ void __launch_bounds__(kThreadsG, 1) qkv_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kStagesP) * kStageBytesP);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStagesP);
    const uint32_t acc_full0 = smem_u32(bars + 2 * kStagesP), acc_empty0 = smem_u32(bars + 2 * kStagesP + kAccBufs);
    const uint32_t mma_done = smem_u32(bars + 2 * kStagesP + 2 * kAccBufs);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStagesP + 2 * kAccBufs + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();  // 0: the CTA that issues the pair's MMAs
    const uint32_t cid = blockIdx.x / 2, clusters = gridDim.x / 2;
    const uint32_t units = (p.P * p.m_tiles + 1) / 2 * p.n_tiles;
    const uint32_t KB = p.K / kGemmBK;
    const uint32_t full0_lead = map_rank(full0, 0);            // stage barriers the loads of both CTAs complete on
    const uint32_t acc_empty0_lead = map_rank(acc_empty0, 0);  // accumulator releases of both CTAs
    const uint32_t peer_flag = map_rank(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);
    constexpr uint16_t kBoth = 3;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesP; ++s) {
            mbar_init(full0 + 8 * s, 1);   // the even CTA's producer; bytes of both CTAs
            mbar_init(empty0 + 8 * s, 1);  // the pair's MMA commit
        }
        for (uint32_t a = 0; a < kAccBufs; ++a) {
            mbar_init(acc_full0 + 8 * a, 1);
            mbar_init(acc_empty0 + 8 * a, 8);  // the epilogue warps of both CTAs
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols * kAccBufs);
        tmem_relinquish_pair();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer (both CTAs): this CTA's rows and weight half
        const uint64_t pol_w = TFU_GEMM_HINTS ? l2_policy_evict_last() : 0;
        (void)pol_w;
        uint32_t q = 0;
        bool ok = true;
        for (uint32_t t = cid; ok && t < units; t += clusters) {
            const Tile tl = decode_tile<2>(p, t, rank);
            const CUtensorMap* mx = &p.tmap_x[tl.r];
            for (uint32_t kb = 0; kb < KB; ++kb, ++q) {
                const uint32_t s = q % kStagesP, use = q / kStagesP;
                if (use > 0 && !wait_phase<true>(empty0 + 8 * s, (use - 1) & 1u, abort_flag, kWaitCyclesG, peer_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t a = smem_u32(smem + size_t(s) * kStageBytesP);
                if (rank == 0) mbar_expect_tx(full0 + 8 * s, 2 * kStageBytesP);
                tma_load_2d_pair(a, mx, int(kb * kGemmBK), int(tl.m_tile * kGemmBM), full0_lead + 8 * s);
                const int wy = int(tl.n_tile * kGemmBN + rank * (kGemmBN / 2));
                if constexpr (TFU_GEMM_HINTS != 0) {
                    tma_load_2d_pair_hint(a + kABytes, &p.tmap_w_part, int(kb * kGemmBK), wy, full0_lead + 8 * s, pol_w);
                } else {
                    tma_load_2d_pair(a + kABytes, &p.tmap_w_part, int(kb * kGemmBK), wy, full0_lead + 8 * s);
                }
            }
        }
        // the MMAs that read the last fill of each stage have completed (their commit
        // arrives on this CTA's stage barriers), so this CTA's loads have all landed
        for (uint32_t k = q > uint32_t(kStagesP) ? q - kStagesP : 0; k < q; ++k)
            drain_phase<true>(empty0 + 8 * (k % kStagesP), (k / kStagesP) & 1u);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer (the even CTA)
        if (rank == 0) {
            uint32_t q = 0, i = 0;
            bool ok = true;
            for (uint32_t t = cid; ok && t < units; t += clusters, ++i) {
                const uint32_t a = i % kAccBufs, u = i / kAccBufs;
                if (u > 0 && !wait_phase<true>(acc_empty0 + 8 * a, (u - 1) & 1u, abort_flag, kWaitCyclesG, peer_flag))
                    break;  // both epilogues drained it
                tc_fence_after();
                const uint32_t d = tmem + a * kTmemCols;
                for (uint32_t kb = 0; kb < KB; ++kb, ++q) {
                    const uint32_t s = q % kStagesP, use = q / kStagesP;
                    if (!wait_phase<true>(full0 + 8 * s, use & 1u, abort_flag, kWaitCyclesG, peer_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + size_t(s) * kStageBytesP);
#pragma unroll
                    for (uint32_t kk = 0; kk < kGemmBK / 16; ++kk)
                        tc_mma_pair(d, sw128_desc(sa + kk * 32), sw128_desc(sa + kABytes + kk * 32), (kb | kk) != 0);
                    tc_commit_pair(empty0 + 8 * s, kBoth);  // both CTAs' stages are free once read
                }
                tc_commit_pair(acc_full0 + 8 * a, kBoth);  // the tile's accumulators are complete (or abandoned)
            }
            tc_commit_pair(mma_done, kBoth);
        }
        drain_phase<true>(mma_done, 0);  // every MMA of the pair has completed
    } else if (warp >= 2) {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of the pair's tile
        const uint32_t quarter = warp & 3u;
        const uint32_t HD = p.H * kGemmHeadDim;
        uint32_t i = 0;
        for (uint32_t t = cid; t < units; t += clusters, ++i) {
            const uint32_t a = i % kAccBufs, u = i / kAccBufs;
            const bool ok = wait_phase<true>(acc_full0 + 8 * a, u & 1u, abort_flag, kWaitCyclesG, peer_flag);
            tc_fence_after();
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;  // warp-uniform: TMEM loads are collective
            const Tile tl = decode_tile<2>(p, t, rank);
            const uint32_t m = tl.m_tile * kGemmBM + quarter * 32 + lane;
            const bool valid = tl.m_tile < p.m_tiles && m < p.rows;
            const uint32_t b = valid ? m / p.Sl : 0, tt = valid ? m - b * p.Sl : 0;
            const uint32_t pos = tl.r * p.Sl + tt;
#pragma unroll 1
            for (uint32_t j = 0; j < kGemmBN / kGemmHeadDim; ++j) {
                const uint32_t f = tl.n_tile * kGemmBN + j * kGemmHeadDim;
                const uint32_t sec = f / HD;
                const uint32_t h = (f - sec * HD) / kGemmHeadDim;
                const uint32_t g = h / p.Hl, hh = h - g * p.Hl;
                uint8_t* dst_row = p.dst[sec][g] + int64_t(b) * p.d_b + int64_t(pos) * p.d_t + int64_t(hh) * p.d_h;
                const bool norm = kFusedT && sec < 2;
                const uint32_t* wp = norm ? static_cast<const uint32_t*>(p.weight[sec]) : nullptr;
                const float* tab = norm ? p.table + size_t(pos) * kGemmHeadDim : nullptr;
                epilogue_head<kFusedT, kNeox>(tmem + a * kTmemCols + ((quarter * 32u) << 16) + j * kGemmHeadDim, valid,
                                              norm, wp, tab, p.eps, dst_row);
            }
            tc_fence_before();  // this warp's TMEM reads are done before the release
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0_lead + 8 * a);
        }
    }
    // teardown: the pair's MMAs have completed and both CTAs' TMEM reads have
    // finished; the CTAs leave together and free their TMEM together
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols * kAccBufs);
    }
}

// Self-test of the bounded wait: one thread waits on a phase of an mbarrier that
// nothing ever arrives on, with a budget of `budget` clock cycles; the wait gives
// up, records the status bit and raises the abort flag, and the kernel returns.
__global__ void wait_selftest_kernel(long long budget) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
    const bool ok = wait_phase(smem_u32(&bar), 0, &abort_flag, budget);
    if (ok || !abort_flag) atomicOr(&g_gemm_status, 0x80000000u);  // would mean the wait returned wrongly
}

// The driver's tensor-map encoder, looked up once: the function-local static is
// initialised by exactly one thread (C++11 magic statics), so concurrent first
// calls all see the finished lookup.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return nullptr;
    }();
    return fn;
}

// Per-device "attributes set" flags of a kernel.  Setting an attribute twice is
// harmless, so racing first calls need only see a torn-free flag.
using AttrFlags = std::atomic<bool>[64];

template <bool kFusedT, bool kNeox>
cudaError_t launch_variant(const GemmParams& p, cudaStream_t stream) {
    static AttrFlags attr_done = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kernel = qkv_gemm_kernel<kFusedT, kNeox>;
    if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemG));
        if (e != cudaSuccess) return e;
        attr_done[dev].store(true);
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const uint64_t units = uint64_t(p.P) * p.m_tiles * p.n_tiles;
    uint64_t ctas = uint64_t(sms > 0 ? sms : 1);  // one CTA per SM
    if (ctas > units) ctas = units;
    qkv_gemm_kernel<kFusedT, kNeox><<<unsigned(ctas), kThreadsG, kSmemG, stream>>>(p);
    return cudaGetLastError();
}

// The pair form: clusters of two CTAs, as many as can be resident at once (at most
// one per unit); 0 clusters fit -> cudaErrorNotSupported (the caller falls back).
template <bool kFusedT, bool kNeox>
cudaError_t launch_pair_variant(const GemmParams& p, cudaStream_t stream) {
    static AttrFlags attr_done = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kernel = qkv_gemm_pair_kernel<kFusedT, kNeox>;
    if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemP));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return e;
        attr_done[dev].store(true);
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(sms > 1 ? sms / 2 * 2 : 2));
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = kSmemP;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int fit = 0;
    e = cudaOccupancyMaxActiveClusters(&fit, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (fit < 1) return cudaErrorNotSupported;
    const uint64_t units = (uint64_t(p.P) * p.m_tiles + 1) / 2 * p.n_tiles;
    const uint64_t clusters = uint64_t(fit) < units ? uint64_t(fit) : units;
    cfg.gridDim = dim3(unsigned(clusters * 2));
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

#ifndef TFU_GEMM_PAIR
// 1: CTA pairs with the 2-SM MMA (qkv_gemm_pair_kernel; on the video-DiT projection
// 1666-1692 TFLOP/s fused where the single-CTA kernel gives 1537-1570 on the same
// GPU, before the 32 MB raster pass and the L2 policy); 0: single CTAs (the
// fallback, built by the single-CTA parity test).
#define TFU_GEMM_PAIR 1
#endif

}  // namespace

bool encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                          uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t gdim[2] = {cols, rows};
    const cuuint64_t gstride[1] = {row_bytes};
    const cuuint32_t box[2] = {uint32_t(kGemmBK), box_rows};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_qkv_gemm(const GemmParams& p, bool fused, bool neox, cudaStream_t stream) {
    if (uint64_t(p.P) * p.m_tiles * p.n_tiles == 0) return cudaSuccess;
    if (TFU_GEMM_PAIR) {
        const cudaError_t e = !fused ? launch_pair_variant<false, false>(p, stream)
                              : neox ? launch_pair_variant<true, true>(p, stream)
                                     : launch_pair_variant<true, false>(p, stream);
        if (e != cudaErrorNotSupported) return e;
        (void)cudaGetLastError();
    }
    if (!fused) return launch_variant<false, false>(p, stream);
    return neox ? launch_variant<true, true>(p, stream) : launch_variant<true, false>(p, stream);
}

cudaError_t launch_wait_selftest(long long cycles, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(cycles);
    return cudaGetLastError();
}

cudaError_t read_gemm_status(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(unsigned));
}

}  // namespace tfu
