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
// Design (HBM-bound data movement, no tensor cores):
//  * One grouped launch per call.  Work is split into units of 32 KiB (2048
//    16-byte vectors) of one plane = (batch b, shard r, tensor slot x, head group
//    g).  Units are ordered chunk-major with g innermost, so CTAs that run at the
//    same time read whole source token rows (all head groups) and the P head
//    groups of one token block -- and, in the fused mode, reuse the same RoPE
//    table rows from L2.  V (slot 0) comes first within each token block.
//  * A persistent grid (SM count x resident CTAs) walks the units; each thread
//    issues 8 (copy) or 4 (fused) independent 16-byte loads before any store,
//    keeping ~64 KiB+ in flight per SM.  Loads bypass L1 (read-once data);
//    stores are streaming (evict-first) since targets are not re-read here.
//  * Fused rows: D/8 consecutive lanes hold one head row (8 elements each).
//    The sum of squares is accumulated as an unevaluated float pair (TwoSum,
//    Knuth, TAOCP vol. 2, 4.2.2) and reduced with xor-shuffles, so the fp32 mean
//    is the correctly rounded mean for ordinary inputs; all other steps use
//    IEEE-rounded fp32 intrinsics with no contraction, so results match a
//    step-by-step fp32 evaluation bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "relayout.h"

namespace tfu {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint8_t* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float4 ld_table(const float* p) {
    float4 v;
    asm("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

struct Plane {
    const uint8_t* src;
    uint8_t* dst;
    int64_t st, sh, dt, dh;
    uint32_t x;
    uint32_t pos0;  // global position of the plane's first token (scatter)
};

// plane index q = ((b * P + r) * nx + x) * P + g
template <Dir kDir>
__device__ __forceinline__ Plane decode_plane(const RelayoutParams& p, uint32_t q) {
    const uint32_t g = q % p.P;
    uint32_t rest = q / p.P;
    const uint32_t x = rest % p.nx;
    rest /= p.nx;
    const uint32_t r = rest % p.P;
    const uint32_t b = rest / p.P;
    Plane pl;
    pl.x = x;
    pl.st = p.s_t[x];
    pl.sh = p.s_h[x];
    pl.dt = p.d_t[x];
    pl.dh = p.d_h[x];
    if constexpr (kDir == Dir::kScatter) {
        pl.src = p.src[x][r] + int64_t(b) * p.s_b[x] + int64_t(g) * p.Hl * pl.sh;
        pl.dst = p.dst[x][g] + int64_t(b) * p.d_b[x] + int64_t(r) * p.Sl * pl.dt;
        pl.pos0 = r * p.Sl;
    } else {
        pl.src = p.src[x][g] + int64_t(b) * p.s_b[x] + int64_t(r) * p.Sl * pl.st;
        pl.dst = p.dst[x][r] + int64_t(b) * p.d_b[x] + int64_t(g) * p.Hl * pl.dh;
        pl.pos0 = 0;
    }
    return pl;
}

// vector v of a plane -> (token t, head h, vector-in-row dv) -> byte offset
__device__ __forceinline__ int64_t vec_offset(const RelayoutParams& p, uint32_t v, int64_t st, int64_t sh) {
    const uint32_t row = fastdiv(v, p.div_vpr);
    const uint32_t dv = v - row * p.vpr;
    const uint32_t t = fastdiv(row, p.div_hl);
    const uint32_t h = row - t * p.Hl;
    return int64_t(t) * st + int64_t(h) * sh + int64_t(dv) * 16;
}

// Scatter targets are contiguous [B, S, Hl, D]: vector v of a plane lands at v * 16.
template <Dir kDir>
__device__ __forceinline__ int64_t dst_offset(const RelayoutParams& p, const Plane& pl, uint32_t v) {
    if constexpr (kDir == Dir::kScatter) {
        return int64_t(v) * 16;
    } else {
        return vec_offset(p, v, pl.dt, pl.dh);
    }
}

template <Dir kDir, int VB>
__device__ __forceinline__ void copy_range(const RelayoutParams& p, const Plane& pl, uint32_t v0, uint32_t v1) {
#pragma unroll 1
    for (uint32_t base = v0; base < v1; base += kThreads * VB) {
        uint4 buf[VB];
#pragma unroll
        for (int i = 0; i < VB; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            if (v < v1) buf[i] = ld_stream(pl.src + vec_offset(p, v, pl.st, pl.sh));
        }
#pragma unroll
        for (int i = 0; i < VB; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            if (v < v1) st_stream(pl.dst + dst_offset<kDir>(p, pl, v), buf[i]);
        }
    }
}

// ---- 16-bit <-> fp32 helpers (round to nearest even) ----
template <Fused kF>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
    if constexpr (kF == Fused::kBF16) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        lo = f.x;
        hi = f.y;
    }
}

template <Fused kF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (kF == Fused::kBF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// s + e == a + b exactly, s = fl(a + b)  (TwoSum)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// One lane's 8 elements of a head row: RMSNorm (row reduced over kVpr lanes),
// weight scale, interleaved RoPE with this lane's 4 (cos, sin) pairs tab[0..8).
template <Fused kF, int kVpr>
__device__ __forceinline__ uint4 norm_rope_vec(const uint4& xin, const float (&w)[8], const float* tab, bool valid,
                                               float eps) {
    float4 c0 = make_float4(1.f, 0.f, 1.f, 0.f), c1 = c0;
    if (valid) {  // issued first: the reduction below hides its latency
        c0 = ld_table(tab);
        c1 = ld_table(tab + 4);
    }
    float x[8];
    unpack2<kF>(xin.x, x[0], x[1]);
    unpack2<kF>(xin.y, x[2], x[3]);
    unpack2<kF>(xin.z, x[4], x[5]);
    unpack2<kF>(xin.w, x[6], x[7]);
    // squares of 16-bit values are exact in fp32; accumulate them as hi + lo
    float hi = __fmul_rn(x[0], x[0]), lo = 0.f;
#pragma unroll
    for (int j = 1; j < 8; ++j) {
        float s, e;
        two_sum(hi, __fmul_rn(x[j], x[j]), s, e);
        hi = s;
        lo = __fadd_rn(lo, e);
    }
#pragma unroll
    for (int m = 1; m < kVpr; m <<= 1) {
        const float ohi = __shfl_xor_sync(0xffffffffu, hi, m);
        const float olo = __shfl_xor_sync(0xffffffffu, lo, m);
        float s, e;
        two_sum(hi, ohi, s, e);
        lo = __fadd_rn(__fadd_rn(lo, olo), e);
        hi = s;
    }
    const float ss = __fadd_rn(hi, lo);
    const float ms = __fmul_rn(ss, 1.0f / float(kVpr * 8));  // D is a power of two: exact scaling
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        float y0, y1;
        unpack2<kF>(pack2<kF>(__fmul_rn(x[j], inv), __fmul_rn(x[j + 1], inv)), y0, y1);
        unpack2<kF>(pack2<kF>(__fmul_rn(y0, w[j]), __fmul_rn(y1, w[j + 1])), z[j], z[j + 1]);
    }
    const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = z[2 * k], b = z[2 * k + 1], c = cs[2 * k], s = cs[2 * k + 1];
        o[k] = pack2<kF>(__fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)), __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c)));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <Fused kF, int kVpr>
__device__ __forceinline__ void norm_rope_range(const RelayoutParams& p, const Plane& pl, uint32_t v0, uint32_t v1) {
    constexpr int VB = 4;
    constexpr int kRowFloats = kVpr * 8;  // D floats per table row: D/2 (cos, sin) pairs
    const uint32_t dv = threadIdx.x % kVpr;  // v0 and kThreads are multiples of kVpr
    float w[8];
    {
        const uint4 wv = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.weight[pl.x]) + dv * 16);
        unpack2<kF>(wv.x, w[0], w[1]);
        unpack2<kF>(wv.y, w[2], w[3]);
        unpack2<kF>(wv.z, w[4], w[5]);
        unpack2<kF>(wv.w, w[6], w[7]);
    }
    const float* tab_lane = p.table + size_t(pl.pos0) * kRowFloats + dv * 8;
#pragma unroll 1
    for (uint32_t base = v0; base < v1; base += kThreads * VB) {
        uint4 buf[VB];
#pragma unroll
        for (int i = 0; i < VB; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            buf[i] = make_uint4(0u, 0u, 0u, 0u);
            if (v < v1) {
                const uint32_t row = v / kVpr;
                const uint32_t t = fastdiv(row, p.div_hl);
                const uint32_t h = row - t * p.Hl;
                buf[i] = ld_stream(pl.src + int64_t(t) * pl.st + int64_t(h) * pl.sh + int64_t(dv) * 16);
            }
        }
#pragma unroll
        for (int i = 0; i < VB; ++i) {
            const uint32_t v = base + i * kThreads + threadIdx.x;
            const uint32_t t = fastdiv(v / kVpr, p.div_hl);
            // every lane runs the row reduction (it shuffles); only valid lanes load and store
            const uint4 o = norm_rope_vec<kF, kVpr>(buf[i], w, tab_lane + size_t(t) * kRowFloats, v < v1, p.eps);
            if (v < v1) st_stream(pl.dst + int64_t(v) * 16, o);
        }
    }
}

// Resident CTAs per SM the register budget is sized for: 4 x 256 threads for the
// plain copy (<= 64 registers), 3 x 256 for the fused kernels (<= 85 registers).
template <Fused kF>
constexpr int min_blocks() { return kF == Fused::kNone ? 4 : 3; }

template <Dir kDir, Fused kF, int kVpr>
__global__ void __launch_bounds__(kThreads, min_blocks<kF>()) relayout_kernel(const __grid_constant__ RelayoutParams p) {
#pragma unroll 1
    for (uint32_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const uint32_t c = fastdiv(u, p.div_planes);
        const uint32_t q = u - c * p.n_planes;
        const Plane pl = decode_plane<kDir>(p, q);
        const uint32_t v0 = c * uint32_t(kChunkVecs);
        const uint32_t v1 = min(v0 + uint32_t(kChunkVecs), p.nv);
        if constexpr (kF != Fused::kNone) {
            if ((p.fused_mask >> pl.x) & 1u) {
                norm_rope_range<kF, kVpr>(p, pl, v0, v1);
                continue;
            }
        }
        copy_range<kDir, 8>(p, pl, v0, v1);
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
        const float c = __double2float_rn(cos(angle));
        const float s = __double2float_rn(sin(angle));
        reinterpret_cast<float2*>(p.out)[idx] = make_float2(c, s);
    }
}

int device_sms() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

template <Dir kDir, Fused kF, int kVpr>
cudaError_t launch_one(const RelayoutParams& p, cudaStream_t stream) {
    static int blocks_per_sm = 0;  // same for every device of one architecture
    if (blocks_per_sm == 0) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, relayout_kernel<kDir, kF, kVpr>, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm = b > 0 ? b : 1;
    }
    const int64_t want = int64_t(device_sms()) * blocks_per_sm;
    const unsigned grid = unsigned(want < int64_t(p.n_units) ? want : int64_t(p.n_units));
    relayout_kernel<kDir, kF, kVpr><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <Fused kF>
cudaError_t launch_fused(const RelayoutParams& p, cudaStream_t stream) {
    switch (p.vpr) {
        case 4: return launch_one<Dir::kScatter, kF, 4>(p, stream);
        case 8: return launch_one<Dir::kScatter, kF, 8>(p, stream);
        case 16: return launch_one<Dir::kScatter, kF, 16>(p, stream);
        case 32: return launch_one<Dir::kScatter, kF, 32>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_relayout(const RelayoutParams& p, Dir dir, Fused fused, cudaStream_t stream) {
    if (p.n_units == 0) return cudaSuccess;
    if (dir == Dir::kGather) {
        if (fused != Fused::kNone) return cudaErrorInvalidValue;
        return launch_one<Dir::kGather, Fused::kNone, 0>(p, stream);
    }
    switch (fused) {
        case Fused::kNone: return launch_one<Dir::kScatter, Fused::kNone, 0>(p, stream);
        case Fused::kBF16: return launch_fused<Fused::kBF16>(p, stream);
        case Fused::kFP16: return launch_fused<Fused::kFP16>(p, stream);
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
