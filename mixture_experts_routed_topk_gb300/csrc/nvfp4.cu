// nvfp4.cu -- the NVFP4 inference forward pass of the routed-experts layer on sm_103a (Dist-MoE
// 0.1.0, "Choose a precision and pipeline / NVFP4": inference only, prepared weights).
//
// Format (the reading of NVIDIA's published two-level NVFP4): E2M1 elements in blocks of 16 along
// a GEMM's contraction axis; a block scale S = E4M3(amax / (6 G)) (nearest even, saturating at
// 448), stored as a UE4M3 byte; a per-tensor fp32 scale G; elements E2M1(v / (S G)) (nearest even,
// saturating at 6), +0 when S = 0. The fp32 steps are fixed so that the codes are reproducible:
// t = 6 G, b = amax / t (IEEE quotient), r = 1 / (S G) (IEEE reciprocal of the fp32 product), v * r.
// A weight's G is amax(tensor) / 2688, found when it is prepared; the activations' G (x and the
// SwiGLU output h) are calibration constants given by the caller.
//
// Kernels, in stream order (weights prepared beforehand: k_nv_amax, k_nv_prepare_weight):
//   routing -> k_nv_gather_quant (x rows, quantized once per token, at padded rows: packed E2M1 +
//   UE4M3 chunks)
//   (both GEMMs: the scale chunks of a stage reach TMEM through four scale warps, tcgen05.st)
//   -> gate/up GEMM (kind::mxf4nvf4, 128 x 128 tiles of 64 gate + 64 up columns): g and u scaled
//      by G_x G_w13 in fp32, h = SiLU(g) u quantized per 16 f with G_h -> HQ, HS
//   -> down GEMM (128 x 128 tiles of D): Y[perm[r]] = score G_h G_w2 acc, bf16
//   -> the deterministic combine of the bf16 path.
//
// Packed E2M1: two codes per byte, the lower K index in the low nibble. Scales: chunks of 128 rows
// x 4 blocks (64 K values); a stage (256 K values = one 128-byte swizzled row of codes) takes four
// consecutive chunks, so the K groups of every scale grid are padded to a multiple of 4 with zero
// chunks (zero scales and zero codes contribute 0). A prepared weight's scale buffer starts with a
// 256-byte header holding G (fp32, at byte 0) and its amax (at byte 4, as fp32 bits).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "block_scaled.cuh"

namespace moe {
namespace {

constexpr int kNvHeader = 256;    // bytes before the first scale chunk of a prepared weight
constexpr int kNvGateUpF = 64;    // f values per gate/up tile (64 gate + 64 up accumulator columns)
constexpr int kNvDownN = kNvBN;   // 128 output columns per down tile

// Groups of 64 K values per row, padded to whole 256-wide stages.
__host__ __device__ __forceinline__ int nv_groups(int cols) { return (cols + 255) / 256 * 4; }

// The value of a UE4M3 scale code (exact in fp32).
__device__ __forceinline__ float ue4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// One block of 16 values: returns its UE4M3 scale code and writes the 16 packed E2M1 codes.
// G: the tensor scale; t6g = fp32(6 G).
__device__ __forceinline__ uint32_t nv_block(const float (&v)[16], float G, float t6g, uint2& packed) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float b = __fdiv_rn(amax, t6g);
    const uint32_t s = __nv_cvt_float2_to_fp8x2(make_float2(b, 0.0f), __NV_SATFINITE, __NV_E4M3) & 0xffu;
    const float S = ue4m3_value(s);
    uint32_t w[2] = {0u, 0u};
    if (S != 0.0f) {
        const float r = __frcp_rn(__fmul_rn(S, G));
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float y0 = __fmul_rn(v[8 * q + 2 * p], r), y1 = __fmul_rn(v[8 * q + 2 * p + 1], r);
                const uint32_t byte = __nv_cvt_float2_to_fp4x2(make_float2(y0, y1), __NV_E2M1, cudaRoundNearest);
                w[q] |= (byte & 0xffu) << (8 * p);
            }
    }
    packed = make_uint2(w[0], w[1]);
    return s;
}

// One 512-column step of a warp's row quantization: lane l takes the 16 values at c = c0 + 16 l
// (zeros past cols) as one block and returns its packed codes; word = the four UE4M3 codes of
// lanes 4j .. 4j+3 (valid in lanes with (l & 3) == 0).
__device__ __forceinline__ uint2 nv_quantize_step(const uint4* src, int cols, int c0, float G, float t6g, uint32_t& word) {
    const int lane = threadIdx.x & 31;
    const int c = c0 + lane * 16;
    float v[16];
    if (c < cols) {
        const uint4 q0 = __ldg(src + c / 8), q1 = __ldg(src + c / 8 + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    }
    uint2 packed;
    const uint32_t s = nv_block(v, G, t6g, packed);
    const int base = lane & ~3;
    word = __shfl_sync(0xffffffffu, s, base) | (__shfl_sync(0xffffffffu, s, base + 1) << 8) |
           (__shfl_sync(0xffffffffu, s, base + 2) << 16) | (__shfl_sync(0xffffffffu, s, base + 3) << 24);
    return packed;
}

// One warp quantizes one row of `cols` bf16 values (cols % 128 == 0) into packed E2M1 codes at dst
// (cols / 2 bytes) and UE4M3 scales: the four scales of 64-column group g go, as one 32-bit word,
// to sf_row + g * sf_group_stride, for g < nv_groups(cols) (zero words for the padding groups).
// src null marks a padding row: its scales are written as zero and its codes are left as they are
// (a zero block scale makes every product of the row exactly 0, and E2M1 has no NaN). Lane l
// handles 16 consecutive values per 512-column step.
__device__ __forceinline__ void warp_quantize_row_nv(const uint4* src, uint8_t* dst, int cols, float G, float t6g,
                                                     uint8_t* sf_row, int64_t sf_group_stride) {
    const int lane = threadIdx.x & 31;
    if (src == nullptr) {  // a padding row: zero scale words only
        for (int g = lane; g < nv_groups(cols); g += 32)
            *reinterpret_cast<uint32_t*>(sf_row + static_cast<int64_t>(g) * sf_group_stride) = 0u;
        return;
    }
    const int cols_pad = nv_groups(cols) * 64;
    for (int c0 = 0; c0 < cols_pad; c0 += 512) {
        uint32_t word;
        const uint2 packed = nv_quantize_step(src, cols, c0, G, t6g, word);
        const int c = c0 + lane * 16;
        if (c < cols) *reinterpret_cast<uint2*>(dst + c / 2) = packed;
        if ((lane & 3) == 0 && c < cols_pad)
            *reinterpret_cast<uint32_t*>(sf_row + static_cast<int64_t>(c / 64) * sf_group_stride) = word;
    }
}

// Columns [c_begin, c_end) of a token's row, padded to whole 256-wide groups (c_begin a multiple of
// 512), quantized once and written to up to 32 padded rows of XQ / XS: lane k < nk holds the k-th
// destination row (-1: none). Scales of padded row r, group g: chunk (r / 128, g) of a
// [rows / 128, nv_groups(cols)] grid of 512-byte chunks, byte sf_in_chunk(r, 0) of it.
__device__ __forceinline__ void warp_quantize_row_nv_to_rows(const uint4* src, int cols, int c_begin, int c_end,
                                                             float G, float t6g, int64_t dst_row, int nk, uint8_t* xq,
                                                             uint8_t* xs) {
    const int lane = threadIdx.x & 31;
    const int groups = nv_groups(cols);
    const int cols_pad = groups * 64;
    for (int c0 = c_begin; c0 < c_end && c0 < cols_pad; c0 += 512) {
        uint32_t word;
        const uint2 packed = nv_quantize_step(src, cols, c0, G, t6g, word);
        const int c = c0 + lane * 16;
        for (int k = 0; k < nk; ++k) {
            const int64_t prow = __shfl_sync(0xffffffffu, dst_row, k);
            if (prow < 0) continue;  // warp-uniform
            if (c < cols) *reinterpret_cast<uint2*>(xq + prow * (cols / 2) + c / 2) = packed;
            if ((lane & 3) == 0 && c < cols_pad)
                *reinterpret_cast<uint32_t*>(xs + ((prow >> 7) * groups + c / 64) * 512 +
                                             sf_in_chunk(static_cast<int>(prow & 127), 0)) = word;
        }
    }
}

// The tensor scale of a weight: amax / 2688 (IEEE quotient), 1 for an all-zero tensor.
__device__ __forceinline__ float nv_weight_scale(uint32_t amax_bits) {
    const float amax = __uint_as_float(amax_bits);
    return amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// amax of a bf16 tensor of n8 * 8 elements into *amax_bits (fp32 bits; non-negative floats order
// as unsigned integers), which the caller cleared.
__global__ void __launch_bounds__(256) k_nv_amax(const uint4* __restrict__ w, int64_t n8,
                                                 uint32_t* __restrict__ amax_bits) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float warp_max[8];
    float m = 0.0f;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 q = __ldg(w + i);
        const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(ws[j] << 16)), fabsf(__uint_as_float(ws[j] & 0xffff0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, warp_max[i]);
        atomicMax(amax_bits, __float_as_uint(m));
    }
}

// Weight preparation. which = 0: w13 as [E*2F, D] rows; which = 1: w2 as [E*D, F]. Codes keep the
// row order (two per byte); scales go to the tile-grouped layout after the header: per (expert,
// column tile, 64-wide K group) one 512-byte chunk of the tile's 128 rows (gate/up tile j: gate
// rows f = 64 j .. 64 j + 63 then the same up rows; down tile j: rows d = 128 j .. 128 j + 127).
__global__ void __launch_bounds__(256) k_nv_prepare_weight(const uint4* __restrict__ w, int which, int32_t D,
                                                           int32_t F, int32_t E, uint8_t* __restrict__ data,
                                                           uint8_t* __restrict__ scales) {
    griddep_wait();
    griddep_launch_dependents();
    const float G = nv_weight_scale(reinterpret_cast<const uint32_t*>(scales)[1]);
    if (blockIdx.x == 0 && threadIdx.x == 0) reinterpret_cast<float*>(scales)[0] = G;
    const float t6g = __fmul_rn(6.0f, G);
    const int64_t rows = which == 0 ? static_cast<int64_t>(E) * 2 * F : static_cast<int64_t>(E) * D;
    const int cols = which == 0 ? D : F;
    const int groups = nv_groups(cols);
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += warps_total) {
        int64_t e, j, ntn;
        int n;
        if (which == 0) {
            e = row / (2 * F);
            const int rem = static_cast<int>(row - e * 2 * F);
            const int half = rem / F, f = rem - half * F;
            j = f / kNvGateUpF;
            n = half * kNvGateUpF + (f - static_cast<int>(j) * kNvGateUpF);
            ntn = (F + kNvGateUpF - 1) / kNvGateUpF;
        } else {
            e = row / D;
            const int d = static_cast<int>(row - e * D);
            j = d / kNvDownN;
            n = d - static_cast<int>(j) * kNvDownN;
            ntn = (D + kNvDownN - 1) / kNvDownN;
        }
        uint8_t* sf_row = scales + kNvHeader + ((e * ntn + j) * groups) * 512 + sf_in_chunk(n, 0);
        warp_quantize_row_nv(w + row * (cols / 8), data + row * (cols / 2), cols, G, t6g, sf_row, 512);
    }
}

// XQ in token order, as the MXFP8 gather: item i < T * chunks quantizes chunk i % chunks
// (chunk_cols columns of the row padded to whole 256-wide groups) of x[i / chunks] once (tensor scale gx)
// and writes it to the padded row of each of the token's valid pairs; the next 128 E items clear
// the scale words of padded row 128 tiles[e] + counts[e] + j when it lies in expert e's last row
// tile (a zero scale makes every product 0, whatever the codes). One warp per item.
__global__ void __launch_bounds__(256) k_nv_gather_quant(const uint4* __restrict__ x, const int32_t* __restrict__ ids,
                                                         const int32_t* __restrict__ inv,
                                                         const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets,
                                                         const int32_t* __restrict__ tiles, int32_t E, int32_t K,
                                                         int64_t T, int32_t D, int32_t chunk_cols, float gx,
                                                         uint8_t* __restrict__ xq, uint8_t* __restrict__ xs) {
    extern __shared__ int32_t s_tiles[];  // tiles[0 .. E], the padded-row base of every expert
    griddep_wait();
    griddep_launch_dependents();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_tiles[i] = __ldg(tiles + i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int groups = nv_groups(D);
    const float t6g = __fmul_rn(6.0f, gx);
    const int chunks = (groups * 64 + chunk_cols - 1) / chunk_cols;
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
                warp_quantize_row_nv_to_rows(x + t * (D / 8), D, c_begin, c_begin + chunk_cols, gx, t6g, dst_row, nk,
                                             xq, xs);
            }
        } else {
            const int32_t e = static_cast<int32_t>((item - token_items) >> 7);
            const int32_t j = static_cast<int32_t>((item - token_items) & 127);
            const int32_t n = __ldg(counts + e);
            if (n + j < 128 * (s_tiles[e + 1] - s_tiles[e])) {
                const int64_t prow = 128 * static_cast<int64_t>(s_tiles[e]) + n + j;
                warp_quantize_row_nv(nullptr, xq + prow * (D / 2), D, gx, t6g,
                                     xs + (prow >> 7) * groups * 512 + sf_in_chunk(static_cast<int>(prow & 127), 0),
                                     512);
            }
        }
    }
}

// ------------------------------------------------------------------------------ tile policies

// Gate/up GEMM: A = XQ rows (K = D), B = 64 gate rows and the same 64 up rows of w13. The
// epilogue scales the accumulators by G_x G_w13, computes h = SiLU(g) u and writes its NVFP4 codes
// (G_h = act_scale_out) and scales for all 128 rows of the tile.
struct NvGateUp {
    using Shape = Nvf4Shape;
    using Tile = MxTile;
    static constexpr uint32_t kIdesc = idesc_nvf4(kBM, kNvBN);

    __device__ static int32_t num_tiles(const GemmArgs& a) { return a.ntn * __ldg(a.tiles + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_mx_tile(tile, a); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * 128, t.row0);
        // the tile's 64 gate rows, then its 64 up rows (halves 2e and 2e + 1), in one copy
        tma_load_3d(sb, tb, bar, kb * 128, t.n * kNvGateUpF, 2 * t.e);
    }
    // The stage's scale chunks (A's, then B's), on their own barrier so that they land, and are
    // written to TMEM, while the operand boxes are still in flight.
    __device__ static void load_scales(const Tile& t, int32_t kb, uint8_t* sf, uint64_t* bar, const GemmArgs& a) {
        const int64_t groups = nv_groups(a.D);
        bulk_load(sf, a.sf_a + ((t.row0 >> 7) * groups + 4 * kb) * 512, 2048, bar);
        bulk_load(sf + 2048, a.sf_b + kNvHeader + ((static_cast<int64_t>(t.e) * a.ntn + t.n) * groups + 4 * kb) * 512,
                  2048, bar);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4*, const GemmArgs& a) {
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
        const float scale = __fmul_rn(a.act_scale_a, __ldg(reinterpret_cast<const float*>(a.sf_b)));
        const float gh = a.act_scale_out;
        const float t6g = __fmul_rn(6.0f, gh);
        const int64_t fgroups = nv_groups(a.F);
#pragma unroll 1
        for (int c = 0; c < kNvGateUpF / 32; ++c) {
            __syncwarp();  // tcgen05.ld is .sync.aligned
            uint32_t g[32], u[32];
            tmem_ld_32cols(taddr + c * 32, g);
            tmem_ld_32cols(taddr + kNvGateUpF + c * 32, u);
            tmem_ld_wait(g);
            tmem_ld_tie(u);
            const int32_t f0 = t.n * kNvGateUpF + c * 32;
            if (f0 < a.F) {  // F % 32 == 0: both 16-blocks are in or out
                float h0[16], h1[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    h0[j] = silu_fast(__uint_as_float(g[j]) * scale) * (__uint_as_float(u[j]) * scale);
                    h1[j] = silu_fast(__uint_as_float(g[16 + j]) * scale) * (__uint_as_float(u[16 + j]) * scale);
                }
                uint2 p0, p1;
                const uint32_t s0 = nv_block(h0, gh, t6g, p0);
                const uint32_t s1 = nv_block(h1, gh, t6g, p1);
                *reinterpret_cast<uint4*>(a.q_out + row * (a.F / 2) + f0 / 2) = make_uint4(p0.x, p0.y, p1.x, p1.y);
                *reinterpret_cast<uint16_t*>(a.sf_out + ((row >> 7) * fgroups + (f0 >> 6)) * 512 +
                                             sf_in_chunk(row_in_tile, (f0 >> 4) & 3)) =
                    static_cast<uint16_t>(s0 | (s1 << 8));
            }
        }
    }
};

// Down GEMM: A = HQ rows (K = F), B = 128 rows of W2; Y[perm[r]] = score G_h G_w2 acc for the
// tile's routed rows (G_h = act_scale_a), through the per-warp staging buffer.
struct NvDown {
    using Shape = Nvf4Shape;
    using Tile = MxTile;
    static constexpr uint32_t kIdesc = idesc_nvf4(kBM, kNvBN);

    __device__ static int32_t num_tiles(const GemmArgs& a) { return a.ntn * __ldg(a.tiles + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_mx_tile(tile, a); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * 128, t.row0);
        tma_load_2d(sb, tb, bar, kb * 128, t.e * a.D + t.n * kNvDownN);
    }
    // The stage's scale chunks (A's, then B's), on their own barrier so that they land, and are
    // written to TMEM, while the operand boxes are still in flight.
    __device__ static void load_scales(const Tile& t, int32_t kb, uint8_t* sf, uint64_t* bar, const GemmArgs& a) {
        const int64_t groups = nv_groups(a.F);
        bulk_load(sf, a.sf_a + ((t.row0 >> 7) * groups + 4 * kb) * 512, 2048, bar);
        bulk_load(sf + 2048, a.sf_b + kNvHeader + ((static_cast<int64_t>(t.e) * a.ntn + t.n) * groups + 4 * kb) * 512,
                  2048, bar);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        const bool valid = row_in_tile < t.rows;
        int32_t pair = 0;
        float scale = 0.0f;
        if (valid) {
            pair = __ldg(a.perm + t.rrow0 + row_in_tile);
            scale = __fmul_rn(__fmul_rn(a.act_scale_a, __ldg(reinterpret_cast<const float*>(a.sf_b))),
                              pair_score(a, pair));
        }
        uint32_t words[32];  // 64 bf16 of this thread's row
#pragma unroll 1
        for (int cp = 0; cp < kNvDownN / 64; ++cp) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                __syncwarp();
                uint32_t v[32];
                tmem_ld_32cols(taddr + (2 * cp + half) * 32, v);
                tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    words[half * 16 + j] =
                        pack_bf16x2(__uint_as_float(v[2 * j]) * scale, __uint_as_float(v[2 * j + 1]) * scale);
            }
            const int32_t d0 = t.n * kNvDownN + cp * 64;  // D % 64 == 0: all 64 columns in or out
            warp_store_row_segments(stage, words,
                                    reinterpret_cast<char*>(a.out0 + static_cast<int64_t>(pair) * a.D + d0),
                                    valid && d0 < a.D);
        }
    }
};

// Stage 0: status word, routing, scale chunks of HQ cleared when F leaves padding groups, and the
// gather-quantize of x.
moe_status_t nv_dispatch(const MxProblem& p, cudaStream_t stream) {
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (p.F % 256 != 0 &&
        cudaMemsetAsync(p.hs, 0, static_cast<size_t>(p.padded_rows / 128) * nv_groups(p.F) * 512, stream) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
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
    const int32_t chunk = gather_chunk_cols(p.T, nv_groups(p.D) * 64);
    return launch_pdl(k_nv_gather_quant,
                      dim3(quant_grid(p.T * ((nv_groups(p.D) * 64 + chunk - 1) / chunk) + 128 * static_cast<int64_t>(p.E),
                                      p.sm_count)),
                      dim3(256), sizeof(int32_t) * (p.E + 1), stream, static_cast<const uint4*>(p.x), p.ids,
                      static_cast<const int32_t*>(p.inv), static_cast<const int32_t*>(p.counts),
                      static_cast<const int32_t*>(p.offsets), static_cast<const int32_t*>(p.tiles1), p.E, p.K, p.T,
                      p.D, chunk, p.act_scale_x, p.xq, p.xs) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

GemmArgs nv_args(const MxProblem& p) {
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

int64_t nv_max_row_tiles(const MxProblem& p) {
    const int64_t R = p.T * p.K;
    return ceil_div(R, kBM) + (R < p.E ? R : p.E);
}

// Stage 1: gate/up + SwiGLU + NVFP4 quantization of H.
moe_status_t nv_gate_up(const MxProblem& p, cudaStream_t stream) {
    GemmArgs a = nv_args(p);
    CUtensorMap ta, tb;
    if (!make_tmap_u8(&ta, p.xq, p.D / 2, p.padded_rows, 128, kBM) ||
        !make_tmap_u8_pairs(&tb, p.w13q, p.D / 2, p.F, static_cast<uint64_t>(p.E) * 2, 128, kNvGateUpF))
        return MOE_ERR_CUDA;
    a.kblocks = nv_groups(p.D) / 4;
    a.ntn = static_cast<int32_t>(ceil_div(p.F, kNvGateUpF));
    a.sf_a = p.xs;
    a.sf_b = static_cast<const uint8_t*>(p.w13s);
    a.q_out = p.hq;
    a.sf_out = p.hs;
    a.act_scale_a = p.act_scale_x;
    a.act_scale_out = p.act_scale_h;
    return launch_gemm<NvGateUp>(ta, tb, a, sm_count_grid(nv_max_row_tiles(p) * a.ntn, p.sm_count), stream);
}

// Stage 2: down projection + score, rows scattered to pair order.
moe_status_t nv_down(const MxProblem& p, cudaStream_t stream) {
    GemmArgs a = nv_args(p);
    CUtensorMap ta, tb;
    if (!make_tmap_u8(&ta, p.hq, p.F / 2, p.padded_rows, 128, kBM) ||
        !make_tmap_u8(&tb, p.w2q, p.F / 2, static_cast<uint64_t>(p.E) * p.D, 128, kNvDownN))
        return MOE_ERR_CUDA;
    a.kblocks = nv_groups(p.F) / 4;
    a.ntn = static_cast<int32_t>(ceil_div(p.D, kNvDownN));
    a.sf_a = p.hs;
    a.sf_b = static_cast<const uint8_t*>(p.w2s);
    a.perm = p.perm;
    a.scores = p.scores;
    a.scores_bf16 = p.scores_dtype == MOE_SCORES_BF16 ? 1 : 0;
    a.out0 = static_cast<__nv_bfloat16*>(p.y);
    a.act_scale_a = p.act_scale_h;
    return launch_gemm<NvDown>(ta, tb, a, sm_count_grid(nv_max_row_tiles(p) * a.ntn, p.sm_count), stream);
}

}  // namespace

size_t nv_weight_scale_bytes(int which, int32_t D, int32_t F, int32_t E) {
    const int64_t ntn = which == 0 ? ceil_div(F, kNvGateUpF) : ceil_div(D, kNvDownN);
    const int groups = nv_groups(which == 0 ? D : F);
    return kNvHeader + static_cast<size_t>(E) * ntn * groups * 512;
}

size_t nv_act_scale_bytes(int64_t padded_rows, int32_t cols) {
    return static_cast<size_t>(padded_rows / 128) * nv_groups(cols) * 512;
}

moe_status_t launch_nv_prepare_weight(int which, const void* w, int32_t D, int32_t F, int32_t E, void* data,
                                      void* scales, size_t scale_bytes, int sm_count, cudaStream_t stream) {
    const int64_t rows = which == 0 ? static_cast<int64_t>(E) * 2 * F : static_cast<int64_t>(E) * D;
    const int cols = which == 0 ? D : F;
    if (cudaMemsetAsync(scales, 0, scale_bytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t n8 = rows * cols / 8;
    const int amax_grid = static_cast<int>(ceil_div(n8, 256) < sm_count * 4 ? ceil_div(n8, 256) : sm_count * 4);
    if (launch_pdl(k_nv_amax, dim3(amax_grid > 0 ? amax_grid : 1), dim3(256), 0, stream, static_cast<const uint4*>(w),
                   n8, reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + 4)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_pdl(k_nv_prepare_weight, dim3(quant_grid(rows, sm_count)), dim3(256), 0, stream,
                      static_cast<const uint4*>(w), which, D, F, E, static_cast<uint8_t*>(data),
                      static_cast<uint8_t*>(scales)) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

moe_status_t launch_nv_forward(const MxProblem& p, int stage_begin, int stage_end, cudaStream_t stream) {
    const auto run = [&](int stage) { return stage_begin <= stage && stage < stage_end; };
    moe_status_t st = MOE_OK;
    if (run(0) && (st = nv_dispatch(p, stream)) != MOE_OK) return st;
    if (run(1) && (st = nv_gate_up(p, stream)) != MOE_OK) return st;
    if (run(2) && (st = nv_down(p, stream)) != MOE_OK) return st;
    if (run(3)) st = launch_combine(p.y, p.ids, p.T, p.D, p.E, p.K, p.out, p.sm_count, stream);
    return st;
}

}  // namespace moe
