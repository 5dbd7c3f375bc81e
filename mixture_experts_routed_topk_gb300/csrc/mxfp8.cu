// mxfp8.cu -- the MXFP8 (E4M3 with UE8M0 block scales) forward pass of the routed-experts layer
// on sm_103a (Dist-MoE 0.1.0, "Choose a precision and pipeline / MXFP8": activations quantized
// after routing, weights prepared once and reused, tensor-core products accumulated in FP32).
//
// Format (the OCP Microscaling v1.0 reading of MXFP8_E4M3): a block is 32 consecutive elements
// along a GEMM's contraction axis; it shares the scale 2^e, e = floor(log2 max|v|) - 8 clamped to
// [-127, 127] (-127 for an all-zero block), stored as the UE8M0 byte e + 127; each element is
// v * 2^-e rounded to E4M3, nearest even, saturating at 448 (the hardware's cvt .satfinite).
//
// Kernels, in stream order (weights prepared beforehand by k_mx_prepare_weight):
//   routing (shared with the bf16 path; row-tile prefix tiles[e] = sum ceil(n_e' / 128))
//   -> k_mx_gather_quant: x rows, quantized once per token -> XQ codes + scales, every expert's rows
//      starting on a 128-row boundary ("padded rows"), so a row tile's scales are one chunk
//   -> gate/up GEMM (block-scaled tcgen05): H = SiLU(g) * u from the fp32 accumulators,
//      quantized per 32 f in the epilogue -> HQ codes + scales
//   -> down GEMM (block-scaled tcgen05): Y[perm[r]] = score * (H W2^T), bf16
//   -> the deterministic combine of the bf16 path.
//
// Scale layout: a chunk is 512 bytes holding the scales of 128 rows for 4 consecutive blocks
// (row r, block k at 16 (r % 32) + 4 (r / 32) + k), the layout tcgen05.cp .32x128b.warpx4
// copies into TMEM. Activation scales: chunk (row / 128, block / 4) of a [rows/128, cols/128]
// grid. Weight scales are grouped per GEMM tile: 1024 bytes (two chunks, 256 tile rows) per
// (expert, column tile, 128-wide K group); a gate/up tile's rows are 96 gate rows then the same
// 96 up rows, a down tile's rows 192 consecutive output rows.
#include <cuda_fp8.h>

#include "block_scaled.cuh"

namespace moe {

namespace {

// ------------------------------------------------------------------------------ quantization

// e of a block whose largest magnitude is amax: floor(log2 amax) - 8, clamped to [-127, 127];
// zero and subnormal maxima (floor(log2) <= -127) give -127.
__device__ __forceinline__ int mx_exponent(float amax) {
    const int field = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
    if (field == 0) return -127;
    const int e = field - 127 - 8;
    return e < -127 ? -127 : e;
}

// 2^-e as a float (exact: -e is in [-119, 127]).
__device__ __forceinline__ float mx_inv_scale(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

// Four values times m, rounded to E4M3 (nearest even, saturating), packed low byte first.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float m) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a * m, b * m), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c * m, d * m), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

// One 256-column step of a warp's row quantization: lane l takes the 8 values at c = c0 + 8 l
// (zeros past cols), lanes 4j .. 4j+3 share one 32-value block. Returns the lane's 8 E4M3 codes;
// word = the four UE8M0 codes of the 128-column group starting at c0 + 8 (l & 16), valid in lanes
// with (l & 15) == 0.
__device__ __forceinline__ uint2 mx_quantize_step(const uint4* src, int cols, int c0, uint32_t& word) {
    const int lane = threadIdx.x & 31;
    const int c = c0 + lane * 8;
    float v[8];
    if (c < cols) {
        const uint4 q = __ldg(src + c / 8);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int e = mx_exponent(amax);
    const float m = mx_inv_scale(e);
    const uint32_t code = static_cast<uint32_t>(e + 127);
    const int base = lane & 16;
    word = __shfl_sync(0xffffffffu, code, base) | (__shfl_sync(0xffffffffu, code, base + 4) << 8) |
           (__shfl_sync(0xffffffffu, code, base + 8) << 16) | (__shfl_sync(0xffffffffu, code, base + 12) << 24);
    return make_uint2(e4m3x4(v[0], v[1], v[2], v[3], m), e4m3x4(v[4], v[5], v[6], v[7], m));
}

// One warp quantizes one row of `cols` bf16 values (cols % 128 == 0; src null = a zero row: zero
// codes and the all-zero block's scale code 0, written directly) into
// E4M3 codes at dst and UE8M0 scales: the four scales of 128-column group g go, as one 32-bit
// word, to sf_row + g * sf_group_stride.
__device__ __forceinline__ void warp_quantize_row(const uint4* src, uint8_t* dst, int cols, uint8_t* sf_row,
                                                  int64_t sf_group_stride) {
    const int lane = threadIdx.x & 31;
    if (src == nullptr) {  // a zero row: codes 0 and scale codes 0 (e = -127), no arithmetic
        for (int c = lane * 16; c < cols; c += 512) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
        for (int g = lane; g < cols / 128; g += 32)
            *reinterpret_cast<uint32_t*>(sf_row + static_cast<int64_t>(g) * sf_group_stride) = 0u;
        return;
    }
    for (int c0 = 0; c0 < cols; c0 += 256) {
        uint32_t word;
        const uint2 codes = mx_quantize_step(src, cols, c0, word);
        const int c = c0 + lane * 8;
        if (c < cols) *reinterpret_cast<uint2*>(dst + c) = codes;
        if ((lane & 15) == 0 && c < cols) *reinterpret_cast<uint32_t*>(sf_row + static_cast<int64_t>(c / 128) * sf_group_stride) = word;
    }
}

// Columns [c_begin, c_end) of a token's row (c_begin a multiple of 256), quantized once and written
// to up to 32 padded rows of XQ / XS: lane k < nk holds the k-th destination row (-1: none).
// Scales of padded row r, group g: chunk (r / 128, g) of a [rows / 128, groups] grid of 512-byte
// chunks, byte sf_in_chunk(r, 0) of it.
__device__ __forceinline__ void warp_quantize_row_to_rows(const uint4* src, int cols, int c_begin, int c_end,
                                                          int64_t dst_row, int nk, uint8_t* xq, uint8_t* xs) {
    const int lane = threadIdx.x & 31;
    const int groups = cols / 128;
    for (int c0 = c_begin; c0 < c_end && c0 < cols; c0 += 256) {
        uint32_t word;
        const uint2 codes = mx_quantize_step(src, cols, c0, word);
        const int c = c0 + lane * 8;
        for (int k = 0; k < nk; ++k) {
            const int64_t prow = __shfl_sync(0xffffffffu, dst_row, k);
            if (prow < 0) continue;  // warp-uniform
            if (c < cols) *reinterpret_cast<uint2*>(xq + prow * cols + c) = codes;
            if ((lane & 15) == 0 && c < cols)
                *reinterpret_cast<uint32_t*>(xs + ((prow >> 7) * groups + c / 128) * 512 +
                                             sf_in_chunk(static_cast<int>(prow & 127), 0)) = word;
        }
    }
}

// Weight preparation. which = 0: w13 viewed as [E*2F, D] rows (gate rows of expert e at e*2F,
// up rows at e*2F + F); which = 1: w2 viewed as [E*D, F]. Codes keep the row order; scales go
// to the tile-grouped layout. One warp per row. The scale buffer is cleared beforehand.
__global__ void __launch_bounds__(256) k_mx_prepare_weight(const uint4* __restrict__ w, int which, int32_t D,
                                                           int32_t F, int32_t E, uint8_t* __restrict__ data,
                                                           uint8_t* __restrict__ scales) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t rows = which == 0 ? static_cast<int64_t>(E) * 2 * F : static_cast<int64_t>(E) * D;
    const int cols = which == 0 ? D : F;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += warps_total) {
        int64_t e, j, ntn;
        int n;
        if (which == 0) {
            e = row / (2 * F);
            const int rem = static_cast<int>(row - e * 2 * F);
            const int half = rem / F, f = rem - half * F;
            j = f / kMxGateUpF;
            n = half * kMxGateUpF + (f - static_cast<int>(j) * kMxGateUpF);
            ntn = (F + kMxGateUpF - 1) / kMxGateUpF;
        } else {
            e = row / D;
            const int d = static_cast<int>(row - e * D);
            j = d / kMxDownN;
            n = d - static_cast<int>(j) * kMxDownN;
            ntn = (D + kMxDownN - 1) / kMxDownN;
        }
        uint8_t* sf_row = scales + ((e * ntn + j) * (cols / 128)) * 1024 + 512 * (n >> 7) + sf_in_chunk(n, 0);
        warp_quantize_row(w + row * (cols / 8), data + row * cols, cols, sf_row, 1024);
    }
}

// XQ in token order. Work item i < T * chunks: chunk i % chunks (chunk_cols columns, a multiple of
// 1024: whole rows for large batches, 1024 columns for small ones) of x[t], t = i / chunks,
// is quantized once and written to the padded row of each of the token's valid pairs (pair
// p = t K + k of expert e = ids[p] sits at padded row 128 tiles[e] + inv[p] - offsets[e]), so x is
// read once per token, not once per pair. The next 128 E items fill padded row
// 128 tiles[e] + counts[e] + j when it lies in expert e's last row tile: zero codes and scale
// 2^-127. One warp per item.
__global__ void __launch_bounds__(256) k_mx_gather_quant(const uint4* __restrict__ x, const int32_t* __restrict__ ids,
                                                         const int32_t* __restrict__ inv,
                                                         const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets,
                                                         const int32_t* __restrict__ tiles, int32_t E, int32_t K,
                                                         int64_t T, int32_t D, int32_t chunk_cols,
                                                         uint8_t* __restrict__ xq, uint8_t* __restrict__ xs) {
    extern __shared__ int32_t s_tiles[];  // tiles[0 .. E], the padded-row base of every expert
    griddep_wait();
    griddep_launch_dependents();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_tiles[i] = __ldg(tiles + i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int chunks = (D + chunk_cols - 1) / chunk_cols;
    const int64_t token_items = T * chunks;
    const int64_t items = token_items + 128 * static_cast<int64_t>(E);
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
         item += warps_total) {
        if (item < token_items) {
            const int64_t t = item / chunks;
            const int c_begin = static_cast<int>(item - t * chunks) * chunk_cols;
            for (int k0 = 0; k0 < K; k0 += 32) {
                const int nk = min(32, K - k0);
                int64_t dst_row = -1;
                if (lane < nk) {
                    const int64_t p = t * K + k0 + lane;
                    const int32_t e = __ldg(ids + p);
                    if (e >= 0 && e < E)
                        dst_row = 128 * static_cast<int64_t>(s_tiles[e]) + __ldg(inv + p) - __ldg(offsets + e);
                }
                warp_quantize_row_to_rows(x + t * (D / 8), D, c_begin, c_begin + chunk_cols, dst_row, nk, xq, xs);
            }
        } else {
            const int32_t e = static_cast<int32_t>((item - token_items) >> 7);
            const int32_t j = static_cast<int32_t>((item - token_items) & 127);
            const int32_t n = __ldg(counts + e);
            if (n + j < 128 * (s_tiles[e + 1] - s_tiles[e])) {
                const int64_t prow = 128 * static_cast<int64_t>(s_tiles[e]) + n + j;
                warp_quantize_row(nullptr, xq + prow * D, D,
                                  xs + (prow >> 7) * (D / 128) * 512 + sf_in_chunk(static_cast<int>(prow & 127), 0),
                                  512);
            }
        }
    }
}

// ------------------------------------------------------------------------------ tile policies

// Gate/up GEMM with SwiGLU and MX quantization of H: A = XQ rows (K = D), B = 96 gate rows and
// the same 96 up rows of w13; the epilogue writes HQ codes and scales for all 128 rows of the tile
// (padding rows come from zero XQ rows and give zero H rows).
struct MxGateUp {
    using Shape = Mxf8Shape;
    using Tile = MxTile;
    static constexpr uint32_t kIdesc = idesc_mxf8_e4m3(kBM, kMxBN);

    __device__ static int32_t num_tiles(const GemmArgs& a) { return a.ntn * __ldg(a.tiles + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_mx_tile(tile, a); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * kMxBK, t.row0);
        // the tile's 96 gate rows, then its 96 up rows (halves 2e and 2e + 1), in one copy
        tma_load_3d(sb, tb, bar, kb * kMxBK, t.n * kMxGateUpF, 2 * t.e);
    }
    // The stage's scale chunks (A's, then B's), on their own barrier so that they land, and are
    // written to TMEM, while the operand boxes are still in flight.
    __device__ static void load_scales(const Tile& t, int32_t kb, uint8_t* sf, uint64_t* bar, const GemmArgs& a) {
        const int64_t groups = a.D / 128;
        bulk_load(sf, a.sf_a + ((t.row0 >> 7) * groups + kb) * 512, 512, bar);
        bulk_load(sf + 512, a.sf_b + ((static_cast<int64_t>(t.e) * a.ntn + t.n) * groups + kb) * 1024, 1024, bar);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4*, const GemmArgs& a) {
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
        const int64_t fgroups = a.F / 128;
#pragma unroll 1
        for (int c = 0; c < kMxGateUpF / 32; ++c) {
            __syncwarp();  // tcgen05.ld is .sync.aligned
            uint32_t g[32], u[32];
            tmem_ld_32cols(taddr + c * 32, g);
            tmem_ld_32cols(taddr + kMxGateUpF + c * 32, u);
            tmem_ld_wait(g);
            tmem_ld_tie(u);
            const int32_t f0 = t.n * kMxGateUpF + c * 32;
            if (f0 < a.F) {  // F % 32 == 0: a 32-wide block is all in or all out
                float h[32];
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                    h[j] = silu_fast(gv) * uv;
                    amax = fmaxf(amax, fabsf(h[j]));
                }
                const int e = mx_exponent(amax);
                const float m = mx_inv_scale(e);
                uint32_t w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) w[q] = e4m3x4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3], m);
                uint4* dst = reinterpret_cast<uint4*>(a.q_out + row * a.F + f0);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                a.sf_out[((row >> 7) * fgroups + (f0 >> 7)) * 512 + sf_in_chunk(row_in_tile, (f0 >> 5) & 3)] =
                    static_cast<uint8_t>(e + 127);
            }
        }
    }
};

// Down GEMM with the score: A = HQ rows (K = F), B = 192 rows of W2; Y[perm[r]] = score * acc for
// the tile's routed rows, through the per-warp staging buffer (whole 128-byte row segments).
struct MxDown {
    using Shape = Mxf8Shape;
    using Tile = MxTile;
    static constexpr uint32_t kIdesc = idesc_mxf8_e4m3(kBM, kMxBN);

    __device__ static int32_t num_tiles(const GemmArgs& a) { return a.ntn * __ldg(a.tiles + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_mx_tile(tile, a); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * kMxBK, t.row0);
        tma_load_2d(sb, tb, bar, kb * kMxBK, t.e * a.D + t.n * kMxDownN);
    }
    // The stage's scale chunks (A's, then B's), on their own barrier so that they land, and are
    // written to TMEM, while the operand boxes are still in flight.
    __device__ static void load_scales(const Tile& t, int32_t kb, uint8_t* sf, uint64_t* bar, const GemmArgs& a) {
        const int64_t groups = a.F / 128;
        bulk_load(sf, a.sf_a + ((t.row0 >> 7) * groups + kb) * 512, 512, bar);
        bulk_load(sf + 512, a.sf_b + ((static_cast<int64_t>(t.e) * a.ntn + t.n) * groups + kb) * 1024, 1024, bar);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        const bool valid = row_in_tile < t.rows;
        int32_t pair = 0;
        float score = 0.0f;
        if (valid) {
            pair = __ldg(a.perm + t.rrow0 + row_in_tile);
            score = pair_score(a, pair);
        }
        uint32_t words[32];  // 64 bf16 of this thread's row
#pragma unroll 1
        for (int cp = 0; cp < kMxDownN / 64; ++cp) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                __syncwarp();
                uint32_t v[32];
                tmem_ld_32cols(taddr + (2 * cp + half) * 32, v);
                tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    words[half * 16 + j] =
                        pack_bf16x2(__uint_as_float(v[2 * j]) * score, __uint_as_float(v[2 * j + 1]) * score);
            }
            const int32_t d0 = t.n * kMxDownN + cp * 64;  // D % 64 == 0: all 64 columns in or out
            warp_store_row_segments(stage, words,
                                    reinterpret_cast<char*>(a.out0 + static_cast<int64_t>(pair) * a.D + d0),
                                    valid && d0 < a.D);
        }
    }
};

}  // namespace

moe_status_t launch_mx_prepare_weight(int which, const void* w, int32_t D, int32_t F, int32_t E, void* data,
                                      void* scales, size_t scale_bytes, int sm_count, cudaStream_t stream) {
    const int64_t rows = which == 0 ? static_cast<int64_t>(E) * 2 * F : static_cast<int64_t>(E) * D;
    if (cudaMemsetAsync(scales, 0, scale_bytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_pdl(k_mx_prepare_weight, dim3(quant_grid(rows, sm_count)), dim3(256), 0, stream,
                      static_cast<const uint4*>(w), which, D, F, E, static_cast<uint8_t*>(data),
                      static_cast<uint8_t*>(scales)) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

namespace {

// Stage 0: status word, routing (the row-tile prefix, with one column tile) and the gather-quantize.
moe_status_t mx_dispatch(const MxProblem& p, cudaStream_t stream) {
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    RoutingBuffers b{};
    b.ids = p.ids;
    b.R = p.T * p.K;
    b.E = p.E;
    b.nblk = p.nblk;
    b.block_counts = p.block_counts;
    b.block_bases = p.block_bases;
    b.counts = p.counts;
    b.offsets = p.offsets;
    b.perm = p.perm;
    b.inv = p.inv;
    b.tiles1 = p.tiles1;
    b.tiles2 = p.tiles2;
    b.ntiles_n1 = 1;
    b.ntiles_n2 = 1;
    b.status = p.status;
    moe_status_t st = launch_routing(b, stream);
    if (st != MOE_OK) return st;
    const int32_t chunk = gather_chunk_cols(p.T, p.D);
    return launch_pdl(k_mx_gather_quant,
                      dim3(quant_grid(p.T * ((p.D + chunk - 1) / chunk) + 128 * static_cast<int64_t>(p.E), p.sm_count)),
                      dim3(256), sizeof(int32_t) * (p.E + 1), stream, static_cast<const uint4*>(p.x), p.ids,
                      static_cast<const int32_t*>(p.inv), static_cast<const int32_t*>(p.counts),
                      static_cast<const int32_t*>(p.offsets), static_cast<const int32_t*>(p.tiles1), p.E, p.K, p.T,
                      p.D, chunk, p.xq, p.xs) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

GemmArgs mx_args(const MxProblem& p) {
    GemmArgs a{};
    a.counts = p.counts;
    a.offsets = p.offsets;
    a.tiles = p.tiles1;
    a.E = p.E;
    a.D = p.D;
    a.F = p.F;
    a.status = p.status;
    return a;
}

// Upper bound of the row tiles: ceil(R/128) + (experts that can be non-empty).
int64_t mx_max_row_tiles(const MxProblem& p) {
    const int64_t R = p.T * p.K;
    return ceil_div(R, kBM) + (R < p.E ? R : p.E);
}

// Stage 1: gate/up + SwiGLU + MX quantization of H.
moe_status_t mx_gate_up(const MxProblem& p, cudaStream_t stream) {
    GemmArgs a = mx_args(p);
    CUtensorMap ta, tb;
    if (!make_tmap_u8(&ta, p.xq, p.D, p.padded_rows, kMxBK, kBM) ||
        !make_tmap_u8_pairs(&tb, p.w13q, p.D, p.F, static_cast<uint64_t>(p.E) * 2, kMxBK, kMxGateUpF))
        return MOE_ERR_CUDA;
    a.kblocks = p.D / kMxBK;
    a.ntn = static_cast<int32_t>(ceil_div(p.F, kMxGateUpF));
    a.sf_a = p.xs;
    a.sf_b = static_cast<const uint8_t*>(p.w13s);
    a.q_out = p.hq;
    a.sf_out = p.hs;
    return launch_gemm<MxGateUp>(ta, tb, a, sm_count_grid(mx_max_row_tiles(p) * a.ntn, p.sm_count), stream);
}

// Stage 2: down projection + score, rows scattered to pair order.
moe_status_t mx_down(const MxProblem& p, cudaStream_t stream) {
    GemmArgs a = mx_args(p);
    CUtensorMap ta, tb;
    if (!make_tmap_u8(&ta, p.hq, p.F, p.padded_rows, kMxBK, kBM) ||
        !make_tmap_u8(&tb, p.w2q, p.F, static_cast<uint64_t>(p.E) * p.D, kMxBK, kMxDownN))
        return MOE_ERR_CUDA;
    a.kblocks = p.F / kMxBK;
    a.ntn = static_cast<int32_t>(ceil_div(p.D, kMxDownN));
    a.sf_a = p.hs;
    a.sf_b = static_cast<const uint8_t*>(p.w2s);
    a.perm = p.perm;
    a.scores = p.scores;
    a.scores_bf16 = p.scores_dtype == MOE_SCORES_BF16 ? 1 : 0;
    a.out0 = static_cast<__nv_bfloat16*>(p.y);
    return launch_gemm<MxDown>(ta, tb, a, sm_count_grid(mx_max_row_tiles(p) * a.ntn, p.sm_count), stream);
}

}  // namespace

moe_status_t launch_mx_forward(const MxProblem& p, int stage_begin, int stage_end, cudaStream_t stream) {
    const auto run = [&](int stage) { return stage_begin <= stage && stage < stage_end; };
    moe_status_t st = MOE_OK;
    if (run(0) && (st = mx_dispatch(p, stream)) != MOE_OK) return st;
    if (run(1) && (st = mx_gate_up(p, stream)) != MOE_OK) return st;
    if (run(2) && (st = mx_down(p, stream)) != MOE_OK) return st;
    if (run(3)) st = launch_combine(p.y, p.ids, p.T, p.D, p.E, p.K, p.out, p.sm_count, stream);
    return st;
}

}  // namespace moe
