// device_common.cuh -- device helpers shared by the relayout kernels: vector
// loads/stores, plane decoding, 16-bit conversions and the per-lane fused
// RMSNorm + RoPE of a head row (flashinfer PR #6332 commit message,
// "Assumptions / Operator math", interleaved pairs; the half-split pairing as a
// variant, its pairs held within a lane; formulas in tf_ulysses.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "relayout.h"

namespace tfu {
namespace dev {

// ---------------------------------------------------------------- vectors
template <int VW>
struct Vec;
template <>
struct Vec<16> {
    uint32_t w[4];
};
template <>
struct Vec<32> {
    uint32_t w[8];
};

template <int VW>
__device__ __forceinline__ Vec<VW> ld_stream(const uint8_t* p) {
    Vec<VW> v;
    if constexpr (VW == 16) {
        asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
            : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
            : "l"(p));
    } else {
        asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
              "=r"(v.w[7])
            : "l"(p));
    }
    return v;
}

template <int VW>
__device__ __forceinline__ void st_stream(uint8_t* p, const Vec<VW>& v) {
    if constexpr (VW == 16) {
        asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
                     "r"(v.w[3])
                     : "memory");
    } else {
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v.w[0]),
                     "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                     : "memory");
    }
}

__device__ __forceinline__ float4 ld_table(const float* p) {
    float4 v;
    asm("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- launch overlap
// Programmatic dependent launch (launch_overlapped in relayout.h): wait until the
// grid before this one in the stream has completed and its writes are visible
// -- called before a kernel's first global memory access -- and then let the
// grid after this one be scheduled as this one's CTAs retire.  Both are no-ops
// for a launch without the attribute.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- planes
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
        pl.src = p.src[x][r] + int64_t(b) * p.s_b[x] + int64_t(g) * p.Hg * pl.sh;
        pl.dst = p.dst[x][g] + int64_t(b) * p.d_b[x] + int64_t(r) * p.Sl * pl.dt;
        pl.pos0 = r * p.Sl;
    } else {
        pl.src = p.src[x][g] + int64_t(b) * p.s_b[x] + int64_t(r) * p.Sl * pl.st;
        pl.dst = p.dst[x][r] + int64_t(b) * p.d_b[x] + int64_t(g) * p.Hg * pl.dh;
        pl.pos0 = 0;
    }
    return pl;
}

// ---------------------------------------------------------------- 16-bit helpers (RN-even)
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

// round16(a * b) for two pairs of 16-bit values: the exact product of two 16-bit
// values fits fp32, so the packed multiply's single rounding equals rounding
// the fp32 product.
template <Fused kF>
__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
    if constexpr (kF == Fused::kBF16) {
        const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                         *reinterpret_cast<const __nv_bfloat162*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    } else {
        const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
}

// s + e == a + b exactly, s = fl(a + b)  (TwoSum, Knuth, TAOCP vol. 2, 4.2.2)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// ---- packed fp32 pairs (sm_100+ f32x2 arithmetic: each lane of the pair is an
// ordinary IEEE round-to-nearest fp32 operation; one instruction issues both) ----
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// TwoSum on both lanes of a pair
__device__ __forceinline__ void f2_two_sum(uint64_t a, uint64_t b, uint64_t& s, uint64_t& e) {
    s = f2_add(a, b);
    const uint64_t bb = f2_sub(s, a);
    e = f2_add(f2_sub(a, f2_sub(s, bb)), f2_sub(b, bb));
}

// ---- the row's mean of squares (RMSNorm), fp32 ----
// The mean is the fp32 rounding of the exact mean of the squares: squares of
// 16-bit values are exact in fp32, and their sum is carried as an unevaluated
// float pair hi + lo (TwoSum), so fl(hi + lo) is the correctly rounded sum for
// ordinary inputs and the mean follows by an exact power-of-two scaling.

// Lane-local part of row_sumsq: the float pair hi + lo of the squares of the
// lane's values (exact).
template <int NP>
__device__ __forceinline__ void lane_sumsq(const uint64_t (&x2)[NP], float& hi, float& lo) {
    uint64_t hi2 = f2_mul(x2[0], x2[0]), lo2 = 0;
#pragma unroll
    for (int j = 1; j < NP; ++j) {
        uint64_t s, e;
        f2_two_sum(hi2, f2_mul(x2[j], x2[j]), s, e);
        hi2 = s;
        lo2 = f2_add(lo2, e);
    }
    float he, ho, le, lo_, e;
    f2_unpack(hi2, he, ho);
    f2_unpack(lo2, le, lo_);
    two_sum(he, ho, hi, e);
    lo = __fadd_rn(__fadd_rn(le, lo_), e);
}

// Sum of the squares of the lane's values, reduced over the row's kLanes
// lanes; every lane of the group ends with the same pair hi + lo.
template <int kLanes, int NP>
__device__ __forceinline__ void row_sumsq(const uint64_t (&x2)[NP], float& hi, float& lo) {
    lane_sumsq<NP>(x2, hi, lo);
#pragma unroll
    for (int m = 1; m < kLanes; m <<= 1) {  // both partners compute the same pair
        const float ohi = __shfl_xor_sync(0xffffffffu, hi, m);
        const float olo = __shfl_xor_sync(0xffffffffu, lo, m);
        float s, e;
        two_sum(hi, ohi, s, e);
        lo = __fadd_rn(__fadd_rn(lo, olo), e);
        hi = s;
    }
}

constexpr float kFltMax = 3.40282347e38f;

// The fp32 mean of the squares of a head row of D = 2 * kLanes * NP values.
// A float-pair sum that is not finite means an element of magnitude >= 2^64
// (its square, or the sum, overflowed fp32), an infinite element or a NaN.
//  * kExact = false (the pipelined loops): such a row only sets the flag *redo
//    (in shared memory: nothing held in registers across the loops) -- the mean
//    returned is then not the row's, and the caller computes the row again with
//    kExact = true before it is final.
//  * kExact = true: the lanes of such a row -- the condition is uniform within
//    the row's lane group, whose lanes all hold the same pair -- sum the squares
//    of the row scaled by 2^-96 (exact), one scalar pair per lane and shuffles
//    among the group's lanes only, and scale the mean back up by 2^192 in two
//    exact steps: the correctly rounded mean, or +inf when the mean itself
//    exceeds the fp32 range.  An infinite element gives +inf, a NaN NaN.
template <int kLanes, int NP, bool kExact>
__device__ __forceinline__ float row_mean_sq(const uint64_t (&x2)[NP], volatile int* redo) {
    constexpr float kInvD = 1.0f / float(kLanes * NP * 2);  // D is a power of two: exact scaling
    float hi, lo;
    row_sumsq<kLanes, NP>(x2, hi, lo);
    if constexpr (!kExact) {
        if (!(hi <= kFltMax)) *redo = 1;
        return __fmul_rn(__fadd_rn(hi, lo), kInvD);
    } else {
        if (hi <= kFltMax) return __fmul_rn(__fadd_rn(hi, lo), kInvD);
        hi = 0.f;
        lo = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            float v[2], s, e;
            f2_unpack(x2[j], v[0], v[1]);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float a = __fmul_rn(v[k], 0x1p-96f);
                two_sum(hi, __fmul_rn(a, a), s, e);
                lo = __fadd_rn(lo, e);
                hi = s;
            }
        }
        const uint32_t lane = threadIdx.x & 31u;
        const uint32_t group =
            kLanes >= 32 ? 0xffffffffu : ((1u << (kLanes & 31)) - 1u) << (lane & ~uint32_t(kLanes - 1));
#pragma unroll
        for (int m = 1; m < kLanes; m <<= 1) {
            const float ohi = __shfl_xor_sync(group, hi, m);
            const float olo = __shfl_xor_sync(group, lo, m);
            float s, e;
            two_sum(hi, ohi, s, e);
            lo = __fadd_rn(__fadd_rn(lo, olo), e);
            hi = s;
        }
        if (!(hi <= kFltMax)) return hi;  // +inf (an infinite element) or NaN
        return __fmul_rn(__fmul_rn(__fmul_rn(__fadd_rn(hi, lo), kInvD), 0x1p96f), 0x1p96f);
    }
}

// The second half of norm_rope_core for one row: y = round(x * inv),
// z = round(y * w), interleaved RoPE, into xw.
template <Fused kF, int NP>
__device__ __forceinline__ void scale_rotate(uint32_t (&xw)[NP], const uint64_t (&x2)[NP], const uint32_t (&wpk)[NP],
                                             const float4 (&cs)[NP / 2], float inv) {
    const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float a, b;
        f2_unpack(f2_mul(x2[j], inv2), a, b);
        const uint32_t y = pack2<kF>(a, b);  // normalised value rounded before the weight scale
        unpack2<kF>(mul2<kF>(y, wpk[j]), a, b);
        const float4 c4 = cs[j / 2];
        const float c = (j & 1) ? c4.z : c4.x;
        const float s = (j & 1) ? c4.w : c4.y;
        xw[j] = pack2<kF>(__fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)), __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c)));
    }
}

// The second half of norm_rope_core_split for one row: words [0, NP/2) hold the
// lane's elements of the first half of the row, words [NP/2, NP) their partners
// D/2 further on, cs[j] the (cos, sin) entries of word j's elements.
template <Fused kF, int NP>
__device__ __forceinline__ void scale_rotate_split(uint32_t (&xw)[NP], const uint64_t (&x2)[NP],
                                                   const uint32_t (&wpk)[NP], const float4 (&cs)[NP / 2], float inv) {
    const uint64_t inv2 = f2_pack(inv, inv);
    uint32_t z[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float a, b;
        f2_unpack(f2_mul(x2[j], inv2), a, b);
        z[j] = mul2<kF>(pack2<kF>(a, b), wpk[j]);
    }
#pragma unroll
    for (int j = 0; j < NP / 2; ++j) {
        const float4 c4 = cs[j];
        float a0, a1, b0, b1;
        unpack2<kF>(z[j], a0, a1);
        unpack2<kF>(z[j + NP / 2], b0, b1);
        xw[j] = pack2<kF>(__fsub_rn(__fmul_rn(a0, c4.x), __fmul_rn(b0, c4.y)),
                          __fsub_rn(__fmul_rn(a1, c4.z), __fmul_rn(b1, c4.w)));
        xw[j + NP / 2] = pack2<kF>(__fadd_rn(__fmul_rn(a0, c4.y), __fmul_rn(b0, c4.x)),
                                   __fadd_rn(__fmul_rn(a1, c4.w), __fmul_rn(b1, c4.z)));
    }
}

// The arithmetic of one lane: xw holds NP element pairs (2*NP consecutive
// elements) of one head row spread over kLanes consecutive lanes, wpk the
// matching weight pairs, cs the (cos, sin) entries of the lane's pairs, two per
// float4.  RMSNorm, weight scale, then RoPE on interleaved pairs (2i, 2i+1).
// kExact and `redo`: as in row_mean_sq.
template <Fused kF, int kLanes, int NP, bool kExact>
__device__ __forceinline__ void norm_rope_core(uint32_t (&xw)[NP], const uint32_t (&wpk)[NP],
                                               const float4 (&cs)[NP / 2], float eps, volatile int* redo) {
    uint64_t x2[NP];  // the lane's values as fp32 pairs
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float a, b;
        unpack2<kF>(xw[j], a, b);
        x2[j] = f2_pack(a, b);
    }
    scale_rotate<kF, NP>(xw, x2, wpk, cs, __frcp_rn(__fsqrt_rn(__fadd_rn(row_mean_sq<kLanes, NP, kExact>(x2, redo), eps))));
}

// norm_rope_core (fast mean; norm_rope_core_split's rows with kSplit) for two
// rows at once -- the Q and K rows of one position, spread over the same kLanes
// lanes -- sharing the cross-lane work:
// the lower half of the row's lanes reduces the first row's float-pair sums and
// the upper half the second row's (each half receives the other half's partial
// sums of the row it keeps with one exchange, then reduces among itself), each
// half computes one 1/sqrt(mean + eps), and one more exchange gives every lane
// both.  Every lane of a half holds the same pair, so a row's mean is the same
// correctly rounded value as in row_mean_sq; a sum that is not finite sets *redo.
template <Fused kF, int kLanes, int NP, bool kSplit>
__device__ __forceinline__ void norm_rope_pair(uint32_t (&xa)[NP], uint32_t (&xb)[NP], const uint32_t (&wa)[NP],
                                               const uint32_t (&wb)[NP], const float4 (&cs)[NP / 2], float eps,
                                               volatile int* redo) {
    static_assert(kLanes >= 2, "two rows share the cross-lane work of at least two lanes");
    constexpr float kInvD = 1.0f / float(kLanes * NP * 2);
    constexpr int kHalf = kLanes / 2;
    uint64_t x2a[NP], x2b[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float a, b;
        unpack2<kF>(xa[j], a, b);
        x2a[j] = f2_pack(a, b);
        unpack2<kF>(xb[j], a, b);
        x2b[j] = f2_pack(a, b);
    }
    float ha, la, hb, lb;
    lane_sumsq<NP>(x2a, ha, la);
    lane_sumsq<NP>(x2b, hb, lb);
    const bool upper = (threadIdx.x & uint32_t(kHalf)) != 0;
    float hi = upper ? hb : ha, lo = upper ? lb : la;  // the row this lane keeps
    {
        const float ohi = __shfl_xor_sync(0xffffffffu, upper ? ha : hb, kHalf);
        const float olo = __shfl_xor_sync(0xffffffffu, upper ? la : lb, kHalf);
        float s, e;
        two_sum(hi, ohi, s, e);
        lo = __fadd_rn(__fadd_rn(lo, olo), e);
        hi = s;
    }
#pragma unroll
    for (int m = 1; m < kHalf; m <<= 1) {
        const float ohi = __shfl_xor_sync(0xffffffffu, hi, m);
        const float olo = __shfl_xor_sync(0xffffffffu, lo, m);
        float s, e;
        two_sum(hi, ohi, s, e);
        lo = __fadd_rn(__fadd_rn(lo, olo), e);
        hi = s;
    }
    if (!(hi <= kFltMax)) *redo = 1;
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(__fadd_rn(hi, lo), kInvD), eps)));
    const float oinv = __shfl_xor_sync(0xffffffffu, inv, kHalf);
    if constexpr (kSplit) {
        scale_rotate_split<kF, NP>(xa, x2a, wa, cs, upper ? oinv : inv);
        scale_rotate_split<kF, NP>(xb, x2b, wb, cs, upper ? inv : oinv);
    } else {
        scale_rotate<kF, NP>(xa, x2a, wa, cs, upper ? oinv : inv);
        scale_rotate<kF, NP>(xb, x2b, wb, cs, upper ? inv : oinv);
    }
}

// Half-split RoPE on a row whose lanes hold matching halves: words [0, NP/2) are
// the lane's elements of the first half of the row, words [NP/2, NP) their
// partners D/2 further on; cs[j] holds the (cos, sin) entries of the elements
// of word j.  RMSNorm and weight scale as in norm_rope_core; the rotation pairs
// never leave the lane.  kExact and `redo`: as in row_mean_sq.
template <Fused kF, int kLanes, int NP, bool kExact>
__device__ __forceinline__ void norm_rope_core_split(uint32_t (&xw)[NP], const uint32_t (&wpk)[NP],
                                                     const float4 (&cs)[NP / 2], float eps, volatile int* redo) {
    uint64_t x2[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float a, b;
        unpack2<kF>(xw[j], a, b);
        x2[j] = f2_pack(a, b);
    }
    scale_rotate_split<kF, NP>(xw, x2, wpk, cs,
                               __frcp_rn(__fsqrt_rn(__fadd_rn(row_mean_sq<kLanes, NP, kExact>(x2, redo), eps))));
}

// The Q and K rows of one position, spread over the same kLanes lanes, computed
// together: element j of both rows forms one fp32 pair (q_j, k_j), so that every
// packed operation serves both rows -- the sums of squares, the cross-lane
// reduction (one 64-bit pair of float pairs per level), the inverse-RMS scale and
// the rotation, whose (cos, sin) entries Q and K share.  The lane's squares are
// summed in two independent float-pair chains (first and second elements of its
// words) merged once, so every row's mean is the same correctly rounded value as
// in row_mean_sq; the lower half of the row's lanes then computes Q's
// 1/sqrt(mean + eps) and the upper half K's, and one exchange gives every lane
// both.  Each rotation product is a packed fma with the addend -0, which rounds
// exactly as the product alone and cannot be contracted into the sum that
// follows; the addend comes from eps (finite and >= 0) so that the compiler
// cannot fold it.  wqk[2j] and wqk[2j+1] hold the (Q, K) weight pairs of word j's
// first and second element.  kSplit: half-split pairs as in norm_rope_core_split.
// A sum that is not finite sets *redo (row_mean_sq).
template <Fused kF, int kLanes, int NP, bool kSplit>
__device__ __forceinline__ void norm_rope_qk(uint32_t (&xq)[NP], uint32_t (&xk)[NP], const uint32_t (&wqk)[2 * NP],
                                             const float4 (&cs)[NP / 2], float eps, volatile int* redo) {
    constexpr float kInvD = 1.0f / float(kLanes * NP * 2);  // D is a power of two: exact scaling
    uint64_t e2[NP], o2[NP];  // (q, k) of each word's first and of its second element
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float qa, qb, ka, kb;
        unpack2<kF>(xq[j], qa, qb);
        unpack2<kF>(xk[j], ka, kb);
        e2[j] = f2_pack(qa, ka);
        o2[j] = f2_pack(qb, kb);
    }
    uint64_t hi2 = f2_mul(e2[0], e2[0]), lo2 = 0, hb2 = f2_mul(o2[0], o2[0]), lb2 = 0;
#pragma unroll
    for (int j = 1; j < NP; ++j) {
        uint64_t s, e;
        f2_two_sum(hi2, f2_mul(e2[j], e2[j]), s, e);
        hi2 = s;
        lo2 = f2_add(lo2, e);
        f2_two_sum(hb2, f2_mul(o2[j], o2[j]), s, e);
        hb2 = s;
        lb2 = f2_add(lb2, e);
    }
    {
        uint64_t s, e;
        f2_two_sum(hi2, hb2, s, e);
        hi2 = s;
        lo2 = f2_add(f2_add(lo2, lb2), e);
    }
#pragma unroll
    for (int m = 1; m < kLanes; m <<= 1) {  // both partners compute the same pairs
        const uint64_t ohi = __shfl_xor_sync(0xffffffffu, hi2, m);
        const uint64_t olo = __shfl_xor_sync(0xffffffffu, lo2, m);
        uint64_t s, e;
        f2_two_sum(hi2, ohi, s, e);
        lo2 = f2_add(f2_add(lo2, olo), e);
        hi2 = s;
    }
    float hq, hk, lq, lk;
    f2_unpack(hi2, hq, hk);
    f2_unpack(lo2, lq, lk);
    if (!(hq <= kFltMax) || !(hk <= kFltMax)) *redo = 1;
    // the lower half of the row's lanes computes Q's 1/sqrt(mean + eps), the upper half K's
    static_assert(kLanes >= 2, "the two halves of a row's lanes");
    const bool upper = (threadIdx.x & uint32_t(kLanes / 2)) != 0;
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(__fadd_rn(upper ? hk : hq, upper ? lk : lq), kInvD), eps)));
    const float oinv = __shfl_xor_sync(0xffffffffu, inv, kLanes / 2);
    const uint64_t inv2 = f2_pack(upper ? oinv : inv, upper ? inv : oinv);
    // normalised values rounded to 16 bits, times the weights (rounded to 16 bits)
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float a, b;
        f2_unpack(f2_mul(e2[j], inv2), a, b);
        unpack2<kF>(mul2<kF>(pack2<kF>(a, b), wqk[2 * j]), a, b);
        e2[j] = f2_pack(a, b);
        f2_unpack(f2_mul(o2[j], inv2), a, b);
        unpack2<kF>(mul2<kF>(pack2<kF>(a, b), wqk[2 * j + 1]), a, b);
        o2[j] = f2_pack(a, b);
    }
    const float nz = __fmul_rn(-0.0f, eps);
    const uint64_t z2 = f2_pack(nz, nz);
    // (u, v) rotated by (c, s): u*c - v*s and u*s + v*c, every product rounded
    auto rot = [&](uint64_t u, uint64_t v, float c, float s, uint64_t& ou, uint64_t& ov) {
        const uint64_t c2 = f2_pack(c, c), s2 = f2_pack(s, s);
        ou = f2_sub(f2_fma(u, c2, z2), f2_fma(v, s2, z2));
        ov = f2_add(f2_fma(u, s2, z2), f2_fma(v, c2, z2));
    };
    if constexpr (!kSplit) {
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const float4 c4 = cs[j / 2];
            uint64_t ou, ov;
            rot(e2[j], o2[j], (j & 1) ? c4.z : c4.x, (j & 1) ? c4.w : c4.y, ou, ov);
            float uq, uk, vq, vk;
            f2_unpack(ou, uq, uk);
            f2_unpack(ov, vq, vk);
            xq[j] = pack2<kF>(uq, vq);
            xk[j] = pack2<kF>(uk, vk);
        }
    } else {
#pragma unroll
        for (int j = 0; j < NP / 2; ++j) {
            const float4 c4 = cs[j];
            uint64_t a0, b0, a1, b1;
            rot(e2[j], e2[j + NP / 2], c4.x, c4.y, a0, b0);
            rot(o2[j], o2[j + NP / 2], c4.z, c4.w, a1, b1);
            float a0q, a0k, a1q, a1k, b0q, b0k, b1q, b1k;
            f2_unpack(a0, a0q, a0k);
            f2_unpack(a1, a1q, a1k);
            f2_unpack(b0, b0q, b0k);
            f2_unpack(b1, b1q, b1k);
            xq[j] = pack2<kF>(a0q, a1q);
            xk[j] = pack2<kF>(a0k, a1k);
            xq[j + NP / 2] = pack2<kF>(b0q, b1q);
            xk[j + NP / 2] = pack2<kF>(b0k, b1k);
        }
    }
}

}  // namespace dev
}  // namespace tfu
