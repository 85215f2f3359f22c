// tma_plan.h -- the work decomposition of the shared-memory-staged relayout
// kernel, as plain host+device code so it can be checked on the host.
//
// A plane (batch b, shard r, slot x, head group g) holds Sl*Hl head rows of
// row_bytes = D*esize bytes; plane row R = t*Hl + h.  A unit is the row range
// [c*rpu, min((c+1)*rpu, Sl*Hl)) of one plane, staged whole in one shared-memory
// stage (rpu*row_bytes <= kStageBytes).  Each unit is loaded with one bulk copy
// per maximal run of rows that is contiguous in the source and stored with one
// bulk copy per maximal run contiguous in the destination.
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#endif

namespace tfu {

// Two stage rings, chosen per launch by the planner (units of at most the ring's
// stage size; the kernel takes the ring whose stages fit the planned unit):
//  * kStageBytes (64 KiB) x 3, one unit loaded ahead: token head bands of 3 KiB
//    or more, and launches of at most 288 MiB per direction;
//  * kStageBytesSmall (32 KiB) x 6, two units ahead: the rest.
// Measured on GB300 (fractions of the copy peak): 64 KiB units raise the 72 MB
// FLUX-like copy scatter to 0.85 (0.77) and 64 MiB single-tensor relayouts to
// 0.87 (0.80) after a read flush, and 4 KiB-band relayouts of 1-2 GiB to
// 0.95-1.00 (0.89-0.97); on large launches of 1.5-2.5 KiB bands run back to
// back, 32 KiB units keep more in flight (the video-DiT gather 0.961 against
// 0.891; 16 KiB units are far lower everywhere).
#ifndef TFU_STAGE_BYTES
#define TFU_STAGE_BYTES 65536
#endif
#ifndef TFU_STAGE_BYTES_SMALL
#define TFU_STAGE_BYTES_SMALL 32768
#endif
constexpr uint32_t kStageBytes = TFU_STAGE_BYTES;            // the large ring's stage: the largest unit
constexpr uint32_t kStageBytesSmall = TFU_STAGE_BYTES_SMALL;  // the small ring's stage
static_assert(kStageBytes >= 16 && (kStageBytes & (kStageBytes - 1)) == 0,
              "a stage is a power of two bytes (the chunk exchange halves it to a row that divides the chunk)");
static_assert(kStageBytesSmall >= 16 && kStageBytesSmall <= kStageBytes &&
                  (kStageBytesSmall & (kStageBytesSmall - 1)) == 0,
              "the small ring's stage is a power of two no larger than the large one");

// A unit's loads are dealt out to the warp's lanes from this many runs up, its
// stores from this many up (fewer go from lane 0 in order).  Measured on GB300
// with 32 KiB units (fractions of the copy peak): dealing out loads gains at
// every run size (1.5 KiB bands 0.91 against 0.63 from one lane; 2 KiB 0.94
// against 0.79); dealing out stores gains from 16 runs per unit (21 runs of
// 1.5 KiB: 0.85 against 0.67; 16 of 2 KiB: 0.84-0.96 against 0.78-0.91) and
// loses below (12 runs of 2.5 KiB: 0.91 against 0.93).  With 64 KiB units the
// same 16-run threshold measured best (a 32-run one: mean 0.944 against 0.948).
#ifndef TFU_LOAD_SPLIT_RUNS
#define TFU_LOAD_SPLIT_RUNS 1
#endif
#ifndef TFU_STORE_SPLIT_RUNS
#define TFU_STORE_SPLIT_RUNS 16
#endif
constexpr uint32_t kLoadSplitRuns = TFU_LOAD_SPLIT_RUNS;
constexpr uint32_t kStoreSplitRuns = TFU_STORE_SPLIT_RUNS;

// Rows per unit for stages of `stage` bytes: whole tokens (all Hl heads) when a
// token's head band fits a stage, else as many rows as fit.  0 if a single row
// does not fit.
__host__ __device__ inline uint32_t tma_rows_per_unit(uint32_t Hl, uint32_t row_bytes, uint32_t stage = kStageBytes) {
    if (row_bytes == 0 || row_bytes > stage || Hl == 0) return 0;
    const uint64_t token_bytes = uint64_t(Hl) * row_bytes;
    if (token_bytes <= stage) return Hl * uint32_t(stage / token_bytes);
    return uint32_t(stage / row_bytes);
}

// The stage size the planner uses for a pure relayout whose token head band is
// `band` bytes, moving `bytes_per_direction` bytes: the large ring for bands of
// 3 KiB or more, for launches of at most 288 MiB per direction, and for rows
// that do not fit the small stage; the small ring otherwise.
#ifndef TFU_LARGE_RING_BAND
#define TFU_LARGE_RING_BAND 3072  // head bands from this many bytes take the large ring
#endif
#ifndef TFU_LARGE_RING_MAX_MIB
// launches up to this many MiB per direction take the large ring: 288 measured
// gathers of 1.5-2 KiB bands at 141 MiB 0.93 / 0.97 of the copy peak against
// 0.89 / 0.93 at 128, and 2 KiB bands at 256 MiB 0.97-0.98 against 0.95-0.97;
// the video-DiT gather (2.5 KiB bands, 320 MiB) keeps the small ring
#define TFU_LARGE_RING_MAX_MIB 288
#endif
__host__ __device__ inline uint32_t staged_stage_bytes(uint64_t band, uint32_t row_bytes,
                                                       uint64_t bytes_per_direction) {
    if (band >= TFU_LARGE_RING_BAND || bytes_per_direction <= (uint64_t(TFU_LARGE_RING_MAX_MIB) << 20) ||
        row_bytes > kStageBytesSmall)
        return kStageBytes;
    return kStageBytesSmall;
}

// Calls f(first_row_in_unit, n_rows, byte_offset_in_plane) for each maximal run
// of rows [R0, R1) that is contiguous under the strides (st per token, sh per
// head row) of one side of the copy.
template <class F>
__host__ __device__ inline void for_each_run(uint32_t R0, uint32_t R1, uint32_t Hl, int64_t st, int64_t sh,
                                             uint32_t row_bytes, F&& f) {
    if (R1 <= R0) return;
    const bool heads_packed = Hl == 1 || sh == int64_t(row_bytes);  // one head per token is always packed
    if (heads_packed && st == int64_t(Hl) * row_bytes) {  // the whole plane is contiguous
        f(0u, R1 - R0, int64_t(R0) * row_bytes);
        return;
    }
    uint32_t R = R0;
    while (R < R1) {
        const uint32_t t = R / Hl;
        const uint32_t h = R - t * Hl;
        uint32_t n = 1;
        if (heads_packed) {
            n = Hl - h;
            if (n > R1 - R) n = R1 - R;
        }
        f(R - R0, n, int64_t(t) * st + int64_t(h) * sh);
        R += n;
    }
}

// The runs of for_each_run(R0, R1, ...) dealt out to `lanes` workers, for one
// worker `lane`: a range of whole tokens with packed heads is one run per token,
// token k to worker k % lanes; a range with unpacked heads is one run per row,
// row i to worker i % lanes; a range of fewer than `min_split` such runs, a
// contiguous range (one run), or any other range (a token larger than a stage,
// cut by the unit bounds) goes to worker 0 in order.  Over all workers the runs
// are exactly those of for_each_run.
template <class F>
__host__ __device__ inline void for_each_run_lane(uint32_t R0, uint32_t R1, uint32_t Hl, int64_t st, int64_t sh,
                                                  uint32_t row_bytes, uint32_t lane, uint32_t lanes,
                                                  uint32_t min_split, F&& f) {
    if (R1 <= R0) return;
    const bool heads_packed = Hl == 1 || sh == int64_t(row_bytes);
    if (heads_packed && st == int64_t(Hl) * row_bytes) {
        if (lane == 0) f(0u, R1 - R0, int64_t(R0) * row_bytes);
        return;
    }
    if (heads_packed) {
        const uint32_t nt = (R1 - R0) / Hl;
        if (R0 % Hl == 0 && R1 % Hl == 0 && nt >= min_split) {
            const uint32_t t0 = R0 / Hl;
            for (uint32_t k = lane; k < nt; k += lanes) f(k * Hl, Hl, int64_t(t0 + k) * st);
        } else if (lane == 0) {
            for_each_run(R0, R1, Hl, st, sh, row_bytes, f);
        }
        return;
    }
    if (R1 - R0 < min_split) {
        if (lane == 0) for_each_run(R0, R1, Hl, st, sh, row_bytes, f);
        return;
    }
    for (uint32_t i = lane; i < R1 - R0; i += lanes) {
        const uint32_t R = R0 + i, t = R / Hl, h = R - t * Hl;
        f(i, 1u, int64_t(t) * st + int64_t(h) * sh);
    }
}

// The number of runs that for_each_run_lane can deal out for a unit of `rows`
// rows starting at a token boundary: one per token (packed heads, whole tokens),
// one per row (unpacked heads), or 0 where every run goes to worker 0 (a
// contiguous side, or units that cut tokens).  No unit of at most `rows` rows has
// more, so a side whose full units give fewer than min_split never deals out.
__host__ __device__ inline uint32_t unit_split_runs(uint32_t rows, uint32_t Hl, int64_t st, int64_t sh,
                                                    uint32_t row_bytes) {
    const bool heads_packed = Hl == 1 || sh == int64_t(row_bytes);
    if (heads_packed && st == int64_t(Hl) * row_bytes) return 0;
    if (heads_packed) return rows % Hl == 0 ? rows / Hl : 0;
    return rows;
}

}  // namespace tfu
