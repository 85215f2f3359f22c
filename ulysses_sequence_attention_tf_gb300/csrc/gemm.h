// gemm.h -- internal interface of the fused QKV projection (tcgen05 GEMM with
// the RMSNorm + RoPE + Ulysses scatter epilogue).  Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda.h>  // CUtensorMap (the struct only; the encoder is fetched through the runtime)
#include <cuda_runtime.h>

#include "relayout.h"

namespace tfu {

constexpr int kGemmBM = 128;  // tile rows (tokens) = TMEM lanes
constexpr int kGemmBN = 256;  // tile columns (features) = two heads of D = 128
constexpr int kGemmBK = 64;   // K per stage: one 128-byte row, the 128-byte swizzle span
constexpr int kGemmHeadDim = 128;

struct GemmParams {
    CUtensorMap tmap_x[kMaxShards];  // shard r's hidden states [rows = B*Sl][K], box 64 x 128, 128B swizzle
    CUtensorMap tmap_w;              // weight [N = 3*H*D][K], box 64 x 256, 128B swizzle
    CUtensorMap tmap_w_part;         // the same weight, box 64 x 128: a CTA pair's halves of a weight tile
    uint8_t* dst[3][kMaxShards];     // tensor x (Q, K, V), head group g: target base (layout offset applied)
    int64_t d_b, d_t, d_h;           // target byte strides (batch, token, head)
    const void* weight[2];           // RMSNorm weights of Q and K ([D] bf16), fused mode
    const float* table;              // [>= P*Sl][D/2][2] (cos, sin), fused mode
    float eps;
    uint32_t P, B, Sl, H, Hl, K;     // K = hidden
    uint32_t rows;                   // B * Sl rows per shard
    uint32_t m_tiles;                // ceil(rows / 128) per shard
    uint32_t n_tiles;                // 3*H*D / 256
    uint32_t n_group;                // rasterisation: n-tiles that share a pass over the rows
};

// One output tile of the projection: shard r, row tile m_tile (128 rows of the
// shard), column tile n_tile (256 features).
struct GemmTile {
    uint32_t r, m_tile, n_tile;
};

// Tile order: passes of n_group column tiles; inside a pass, row tiles (over all
// shards) outer and column tiles inner, so the CTAs running together share the
// weight columns of the pass and the rows of a few row tiles.  With clusters of
// kCluster CTAs, unit t is a group of kCluster consecutive row tiles of one
// column tile and cluster rank `rank` takes row tile kCluster*mg + rank; a rank
// past the last row tile gets m_tile = m_tiles (rows that do not exist: loads
// fill zeros, nothing is stored), so every CTA of a cluster walks the same units.
// Units: ceil(P*m_tiles / kCluster) * n_tiles.
template <int kCluster>
__host__ __device__ inline GemmTile gemm_tile(uint32_t P, uint32_t m_tiles, uint32_t n_tiles, uint32_t n_group,
                                              uint32_t t, uint32_t rank) {
    const uint32_t MT = P * m_tiles;
    const uint32_t MG = (MT + kCluster - 1) / kCluster;  // row-tile groups
    const uint32_t pass = t / (n_group * MG);
    const uint32_t within = t - pass * n_group * MG;
    const uint32_t rest = n_tiles - pass * n_group;
    const uint32_t gw = n_group < rest ? n_group : rest;  // column tiles in this pass
    const uint32_t mg = within / gw;
    GemmTile tl;
    tl.n_tile = pass * n_group + (within - mg * gw);
    const uint32_t mt = mg * kCluster + rank;
    if (mt < MT) {
        tl.r = mt / m_tiles;
        tl.m_tile = mt - tl.r * m_tiles;
    } else {
        tl.r = 0;
        tl.m_tile = m_tiles;
    }
    return tl;
}

// Launch the projection + epilogue for every (shard, row tile, column tile).
// fused: RMSNorm + RoPE on the Q and K sections; neox: half-split pairs.
cudaError_t launch_qkv_gemm(const GemmParams& p, bool fused, bool neox, cudaStream_t stream);

// One thread waits (bounded by `cycles` clock cycles) on an mbarrier nothing
// arrives on: the projection kernel's bounded wait must give up and report.
cudaError_t launch_wait_selftest(long long cycles, cudaStream_t stream);

// Device status word of the GEMM kernel: 0, or bit 0 when a bounded wait gave up.
cudaError_t read_gemm_status(unsigned* out, bool clear);

// Encode a 2-D bf16 tensor map [rows][cols] (row stride in bytes) with a box of
// 64 columns x box_rows rows and the 128-byte swizzle; false if the driver refuses.
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                          uint32_t box_rows);

}  // namespace tfu
