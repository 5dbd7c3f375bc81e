// block_scaled.cuh -- pieces shared by the block-scaled (MXFP8 and NVFP4) forward passes: the
// padded row-tile list, the scale-chunk layout and the quantization kernels' grid size.
//
// Both passes place every expert's routed rows from a 128-row boundary ("padded rows"), so a row
// tile never straddles two experts and its scales are whole 512-byte chunks. A chunk holds the
// scales of 128 rows for four consecutive blocks along K (row r, block k at byte
// 16 (r % 32) + 4 (r / 32) + k): the layout tcgen05.cp .32x128b.warpx4 copies into TMEM (MXFP8),
// and the one the NVFP4 GEMMs' scale warps store into TMEM lane quarter by lane quarter.
#pragma once

#include "gemm_pipeline.cuh"

namespace moe {
namespace {

// Byte offset of row r (of a 128-row chunk) and block k (of 4) inside a scale chunk.
__device__ __forceinline__ int sf_in_chunk(int r, int k) { return 16 * (r & 31) + 4 * ((r & 127) >> 5) + k; }

struct MxTile {
    int32_t e, n, row0, rows, rrow0, kblocks;  // row0: first padded row; rrow0: first routed row
};

// Tile list over padded rows: expert e owns (tiles[e+1] - tiles[e]) row tiles x ntn column tiles,
// rows fastest, so CTAs running at the same time share one weight tile through L2.
__device__ __forceinline__ MxTile decode_mx_tile(int32_t tile, const GemmArgs& a) {
    MxTile t;
    t.e = owning_expert(tile, a.tiles, a.ntn, a.E);
    const int32_t first = __ldg(a.tiles + t.e);
    const int32_t mt = __ldg(a.tiles + t.e + 1) - first;
    const int32_t local = tile - a.ntn * first;
    t.n = local / mt;
    const int32_t m = local - t.n * mt;
    t.row0 = kBM * (first + m);
    t.rows = min(kBM, __ldg(a.counts + t.e) - m * kBM);
    t.rrow0 = __ldg(a.offsets + t.e) + m * kBM;
    t.kblocks = a.kblocks;
    return t;
}

// Columns per work item of the token-order gathers: whole rows (rounded up to 1024) when the batch
// alone fills the GPU, else 1024-column chunks, so a small batch still spreads over every SM
// (a chunk recomputes its token's destination rows, which costs about 10 % on large batches).
int32_t gather_chunk_cols(int64_t T, int32_t cols) {
    return T >= 2048 ? (cols + 1023) / 1024 * 1024 : 1024;
}

// Blocks of 8 warps (one work item each) for the quantization kernels, at most 8 per SM.
int quant_grid(int64_t rows, int sm_count) {
    const int64_t want = (rows + 7) / 8;  // 8 warps per block, one row each
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int64_t g = want < cap ? want : cap;
    return static_cast<int>(g > 0 ? g : 1);
}

}  // namespace
}  // namespace moe
