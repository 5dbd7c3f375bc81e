// grouped_gemm.cu -- the two grouped expert GEMMs of the routed-experts forward pass on sm_103a,
// as tile policies of the shared tcgen05 pipeline (gemm_pipeline.cuh).
//
//   gate/up GEMM + SwiGLU (TeraMoE README, compute worker: "gate/up projection, activation"; the
//   Dist-MoE execution model's W13 then SwiGLU):
//       H[r, f] = SiLU( XP[r,:] . Wg[e,f,:] ) * ( XP[r,:] . Wu[e,f,:] )      rows r of expert e
//   down GEMM + score (the compute worker's down projection; the combine worker's weighting):
//       Y[p, d] = score[p] * ( H[r,:] . W2[e,d,:] ),   p = perm[r]
//
//  * Tile list: expert e owns ceil(n_e/128) row tiles x the column tiles, rows fastest, so CTAs
//    running at the same time share one weight tile through L2. It is built on the device by the
//    routing scan; the host never reads it, so the call never synchronises.
//  * A gate/up accumulator tile holds 128 gate columns and the same 128 up columns of one f range
//    (two TMA boxes of w13), so SwiGLU is local to the tile and H is written once, in bf16.
//  * Ragged expert segments need no padding: a tile's 128-row TMA box may run into the next
//    expert's rows (computed, not stored) or past the end (zero-filled by TMA).
//  * Expert weights are addressed by row offset in one tensor per projection: expert e's gate rows
//    start at row e*2F of w13 viewed as [E*2F, D], its up rows at e*2F + F, its W2 rows at e*D of
//    w2 viewed as [E*D, F] (the MoonEP FAQ's single contiguous weight tensor per projection).
//  * The down GEMM's output rows (scattered to pair positions) leave through the per-warp
//    shared-memory staging buffer, so each store instruction writes whole 128-byte row segments
//    (measured 5-9 % faster than scattered 16-byte stores). H rows of a tile are consecutive in
//    memory and are written directly (staging them measured slower).
#include "gemm_pipeline.cuh"

namespace moe {
namespace {

struct RowTile {
    int32_t e, n, row0, rows, kblocks;
    int32_t f0, nf;  // gate/up tiles: the first f value and the f values (128, or 64 / 32 in the tail)
};

// Tile index -> (expert, column tile, first routed row, valid rows) for the forward tile list:
// prefix tiles[e], expert e owning ceil(counts[e]/128) row tiles times the column tiles.
__device__ __forceinline__ RowTile decode_row_tile(int32_t tile, const GemmArgs& a) {
    RowTile t;
    t.e = owning_expert(tile, a.tiles, 1, a.E);
    const int32_t local = tile - __ldg(a.tiles + t.e);
    const int32_t ne = __ldg(a.counts + t.e);
    const int32_t mt = (ne + kBM - 1) / kBM;
    t.n = local / mt;
    const int32_t m = local - t.n * mt;
    t.row0 = __ldg(a.offsets + t.e) + m * kBM;
    t.rows = min(kBM, ne - m * kBM);
    t.kblocks = a.kblocks;
    return t;
}

// Gate/up GEMM with SwiGLU: A = XP rows (K-major, K = D), B = w13 gate and up rows (K-major).
//
// Tail split: the tiles past the last whole wave of the grid are cut along f into halves (64 gate +
// 64 up columns, N = 128) or quarters (N = 64) when that many pieces still fit in one wave, so the
// last wave takes a half or a quarter of a tile's time instead of a whole one on a few SMs. The B
// boxes of the pieces come from tensor maps with 64- and 32-row boxes (maps 2 and 3). Every output
// element is still one K-ordered sum of the same products.
struct FwdGateUp {
    using Tile = RowTile;
    static constexpr bool kAMnMajor = false, kBMnMajor = false;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows);

    // tiles in whole waves, and how many pieces each tile of the partial last wave becomes
    __device__ static void tail(int32_t total, int32_t& full, int32_t& split) {
        const int32_t grid = static_cast<int32_t>(gridDim.x);
        const int32_t rem = total % grid;
        full = total - rem;
        split = 4 * rem <= grid ? 4 : (2 * rem <= grid ? 2 : 1);
    }

    __device__ static int32_t num_tiles(const GemmArgs& a) {
        const int32_t total = __ldg(a.tiles + a.E);
        int32_t full, split;
        tail(total, full, split);
        return full + (total - full) * split;
    }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) {
        int32_t full, split;
        tail(__ldg(a.tiles + a.E), full, split);
        if (tile < full) {
            Tile t = decode_row_tile(tile, a);
            t.f0 = t.n * kBN1;
            t.nf = kBN1;
            return t;
        }
        const int32_t j = tile - full;
        Tile t = decode_row_tile(full + j / split, a);
        t.nf = kBN1 / split;
        t.f0 = t.n * kBN1 + (j % split) * t.nf;
        return t;
    }
    __device__ static uint32_t idesc(const Tile& t) {
        return t.nf == kBN1 ? kIdesc : (t.nf == kBN1 / 2 ? idesc_bf16_f32(kBM, kBN1) : idesc_bf16_f32(kBM, kBN1 / 2));
    }
    __device__ static uint32_t tx_bytes(const Tile& t) {
        return static_cast<uint32_t>(kABytes + 2 * t.nf * kBK * 2);
    }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        const CUtensorMap* mb = t.nf == kBN1 ? tb : (t.nf == kBN1 / 2 ? ta + 2 : ta + 3);
        const int32_t gate = t.e * 2 * a.F + t.f0;
        tma_load_2d(sa, ta, bar, kb * kBK, t.row0);
        tma_load_2d(sb, mb, bar, kb * kBK, gate);
        tma_load_2d(sb + t.nf * kBK * 2, mb, bar, kb * kBK, gate + a.F);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4*, const GemmArgs& a) {
        const bool valid = row_in_tile < t.rows;
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
#pragma unroll 1
        for (int c = 0; c < t.nf / 32; ++c) {
            __syncwarp();  // tcgen05.ld is .sync.aligned: reconverge after the masked store
            uint32_t g[32], u[32];
            tmem_ld_32cols(taddr + c * 32, g);
            tmem_ld_32cols(taddr + t.nf + c * 32, u);
            tmem_ld_wait(g);
            tmem_ld_tie(u);
            const int32_t f0 = t.f0 + c * 32;
            if (valid && f0 < a.F) {
                uint32_t packed[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                    const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
                    packed[j] = pack_bf16x2(silu_fast(g0) * u0, silu_fast(g1) * u1);
                }
                store_64B(a.out0 + row * a.F + f0, packed);
            }
        }
    }
};

// Down GEMM with the score: A = H rows (K-major, K = F), B = W2 rows (K-major); Y[perm[r]] rows.
// With kRms (route-wise RMSNorm post-processing) it writes the unweighted expert output instead,
// plus each row's fp32 sum of squares over the tile's columns to fout[pair * column tiles + n].
template <bool kRms>
struct FwdDownT {
    using Tile = RowTile;
    static constexpr bool kAMnMajor = false, kBMnMajor = false;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows);

    __device__ static int32_t num_tiles(const GemmArgs& a) { return __ldg(a.tiles + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_row_tile(tile, a); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * kBK, t.row0);
        tma_load_2d(sb, tb, bar, kb * kBK, t.e * a.D + t.n * kBN2);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        epilogue_to(t, taddr, row_in_tile, stage, a, a.out0);
    }

    // The epilogue with an explicit destination for the Y rows.
    __device__ static void epilogue_to(const RowTile& t, uint32_t taddr, int row_in_tile, uint4* stage,
                                       const GemmArgs& a, __nv_bfloat16* y) {
        const bool valid = row_in_tile < t.rows;
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
        int32_t pair = 0;
        float score = 0.0f;
        if (valid) {
            pair = __ldg(a.perm + row);
            score = kRms ? 1.0f : pair_score(a, pair);
        }
        float sumsq = 0.0f;
        uint32_t words[32];  // 64 bf16 of this thread's row: two 32-column chunks
#pragma unroll 1
        for (int cp = 0; cp < kBN2 / 64; ++cp) {
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
                if (kRms && t.n * kBN2 + cp * 64 < a.D) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) sumsq += __uint_as_float(v[j]) * __uint_as_float(v[j]);
                }
            }
            const int32_t d0 = t.n * kBN2 + cp * 64;  // D % 64 == 0: the 64 columns are all in or all out
            warp_store_row_segments(stage, words,
                                    reinterpret_cast<char*>(y + static_cast<int64_t>(pair) * a.D + d0),
                                    valid && d0 < a.D);
        }
        if (kRms && valid) a.fout[static_cast<int64_t>(pair) * ((a.D + kBN2 - 1) / kBN2) + t.n] = sumsq;
    }
};

// ------------------------------------------------------------------ the fused (Mega) forward
//
// Both GEMMs in one grid (Dist-MoE 0.1.0, "Block-scaled execution": the Mega pipeline
// runs the two projections as one chunked pipeline instead of separate W13 and SwiGLU/W2 kernels).
// The grid walks one interleaved list of slots: a slot is one expert's gate/up tiles (phase 0) or
// its down tiles (phase 1); expert e's down slot comes after the gate/up slot of expert e + L, so
// its H rows are written about L experts earlier and are read back while still in L2:
//     G1(0) .. G1(L-1), G1(L) G2(0), G1(L+1) G2(1), .., G1(E-1) G2(E-L-1), G2(E-L) .. G2(E-1)
// Inside a slot the order is the staged kernels' (rows fastest). CTAs claim tiles in list order
// from a global counter (the tiles differ in length, so a fixed assignment would let CTAs drift
// apart along the list). A down tile's producer waits (bounded) until the four epilogue warps of
// every gate/up tile of its row tile have released the row tile's counter; those tiles come
// earlier in the list and only running CTAs claim tiles, so the lowest unfinished tile can always
// proceed, whether or not every CTA of the grid is resident (another stream may hold SMs). The tiles, their arithmetic and their roundings are
// the staged kernels', so the result is bit-identical to the staged forward's.

struct MegaTile : RowTile {
    int32_t phase;  // 0: gate/up + SwiGLU, 1: down + score
    int32_t rt;     // row tile index over all experts (the readiness counter)
};

// Gate/up slots (a) and down slots (b) among the first k slots of the interleaved list, lag L.
__device__ __forceinline__ void mega_slots_before(int32_t k, int32_t E, int32_t L, int32_t& a, int32_t& b) {
    if (k <= L) {
        a = k;
        b = 0;
    } else if (k <= 2 * E - L) {
        const int32_t j = k - L;
        a = L + (j + 1) / 2;
        b = j / 2;
    } else {
        a = E;
        b = k - E;
    }
}

// Lag in experts: the gate/up tiles of about two waves of the grid between an expert's gate/up
// slot and its down slot.
__device__ __forceinline__ int32_t mega_lag(const GemmArgs& a) {
    // 2 * grid * E < 2^31 (grid <= SM count, E <= 4096)
    const uint32_t g1 = max(__ldg(a.tiles + a.E), 1);
    const uint32_t want = (2u * gridDim.x * static_cast<uint32_t>(a.E) + g1 - 1) / g1;
    return static_cast<int32_t>(min(max(want, 1u), static_cast<uint32_t>(a.E)));
}

struct FwdMega {
    using Tile = MegaTile;
    static constexpr bool kAMnMajor = false, kBMnMajor = false;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows);
    static constexpr bool kDynamicSchedule = true;  // gate/up and down tiles differ in length
    static_assert(FwdGateUp::kIdesc == kIdesc && FwdDownT<false>::kIdesc == kIdesc, "one accumulator shape");

    __device__ static int32_t num_tiles(const GemmArgs& a) { return __ldg(a.tiles + a.E) + __ldg(a.tiles_b + a.E); }

    __device__ static Tile decode(int32_t tile, const GemmArgs& a) {
        const int32_t L = mega_lag(a);
        // the last slot k whose first tile is <= tile
        int32_t lo = 0, hi = 2 * a.E - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            int32_t na, nb;
            mega_slots_before(mid, a.E, L, na, nb);
            if (__ldg(a.tiles + na) + __ldg(a.tiles_b + nb) <= tile) lo = mid;
            else hi = mid - 1;
        }
        int32_t na, nb;
        mega_slots_before(lo, a.E, L, na, nb);
        Tile t;
        if (lo < L) {
            t.phase = 0;
            t.e = lo;
        } else if (lo < 2 * a.E - L) {
            const int32_t j = lo - L;
            t.phase = j & 1;
            t.e = (j & 1) ? (j - 1) / 2 : L + j / 2;
        } else {
            t.phase = 1;
            t.e = lo - a.E;
        }
        const int32_t local = tile - __ldg(a.tiles + na) - __ldg(a.tiles_b + nb);
        const int32_t ne = __ldg(a.counts + t.e);
        const int32_t mt = (ne + kBM - 1) / kBM;
        t.n = local / mt;
        const int32_t m = local - t.n * mt;
        t.row0 = __ldg(a.offsets + t.e) + m * kBM;
        t.rows = min(kBM, ne - m * kBM);
        t.kblocks = t.phase ? a.kblocks_b : a.kblocks;
        t.rt = __ldg(a.tiles + t.e) / a.ntn + m;
        t.f0 = t.n * kBN1;  // gate/up tiles are never split here
        t.nf = kBN1;
        return t;
    }

    // Down tiles: wait until every gate/up epilogue warp of the row tile has released its H rows.
    __device__ static bool acquire(const Tile& t, const GemmArgs& a, volatile int* abort) {
        if (t.phase == 0) return true;
        const uint32_t target = 4u * static_cast<uint32_t>(a.ntn);
        const uint32_t* flag = a.ready + t.rt;
        if (ld_acquire_gpu(flag) < target) {
            const unsigned long long t0 = global_timer_ns();
            while (ld_acquire_gpu(flag) < target) {
                if (*abort) return false;
                if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                    atomicOr(a.status, MOE_DEV_TIMEOUT);
                    *abort = 1;
                    return false;
                }
                __nanosleep(64);
            }
        }
        fence_proxy_async_global();  // the H rows are read next by TMA
        return true;
    }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        if (t.phase == 0) FwdGateUp::load(t, kb, sa, sb, bar, ta, tb, a);
        else FwdDownT<false>::load(t, kb, sa, sb, bar, ta + 2, ta + 3, a);
    }

    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        if (t.phase == 1) {
            FwdDownT<false>::epilogue_to(t, taddr, row_in_tile, stage, a, a.out1);
            return;
        }
        FwdGateUp::epilogue(t, taddr, row_in_tile, stage, a);
        // release this warp's 32 rows of H to the down tiles of the row tile: every lane orders its
        // stores for the async proxy and at GPU scope, then one lane counts the warp
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) red_release_gpu_add(a.ready + t.rt, 1u);
    }
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (f) return f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f, std::memory_order_release);
    return f;
}

GemmArgs row_args(const GemmProblem& p, int32_t kblocks) {
    GemmArgs a{};
    a.counts = p.counts;
    a.offsets = p.offsets;
    a.tiles = p.tiles;
    a.E = p.E;
    a.kblocks = kblocks;
    a.D = p.D;
    a.F = p.F;
    a.status = p.status;
    return a;
}

int row_grid(const GemmProblem& p, int32_t ntn) {
    // upper bound of the tile count: ceil(R/128) + (experts that can be non-empty), per column tile
    const int64_t nonempty = p.R < p.E ? p.R : p.E;
    return sm_count_grid((ceil_div(p.R, kBM) + nonempty) * ntn, p.sm_count);
}

}  // namespace

bool make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8_pairs(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t halves,
                        uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {inner, rows, halves};
    const cuuint64_t strides[2] = {inner, inner * rows};
    const cuuint32_t box[3] = {box_inner, box_rows, 2};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count_grid(int64_t max_tiles, int sm_count) {
    const int64_t g = max_tiles < sm_count ? max_tiles : sm_count;
    return static_cast<int>(g > 0 ? g : 1);
}

moe_status_t launch_gemm1_swiglu(const GemmProblem& p, const void* xp, const void* w13, void* h,
                                 cudaStream_t stream) {
    GemmMaps maps{};
    const uint64_t w13_rows = static_cast<uint64_t>(p.E) * 2 * p.F;
    if (!make_tmap(&maps.m[0], xp, static_cast<uint64_t>(p.D), static_cast<uint64_t>(p.R), kBK, kBM) ||
        !make_tmap(&maps.m[1], w13, static_cast<uint64_t>(p.D), w13_rows, kBK, kBN1) ||
        !make_tmap(&maps.m[2], w13, static_cast<uint64_t>(p.D), w13_rows, kBK, kBN1 / 2) ||  // tail halves
        !make_tmap(&maps.m[3], w13, static_cast<uint64_t>(p.D), w13_rows, kBK, kBN1 / 4))    // tail quarters
        return MOE_ERR_CUDA;
    GemmArgs a = row_args(p, p.D / kBK);
    a.out0 = static_cast<__nv_bfloat16*>(h);
    return launch_gemm<FwdGateUp>(maps, a, row_grid(p, static_cast<int32_t>(ceil_div(p.F, kBN1))), stream);
}

moe_status_t launch_gemm2_score(const GemmProblem& p, const void* h, const void* w2, const int32_t* perm,
                                const void* scores, int32_t scores_dtype, void* y, float* rms_sumsq,
                                cudaStream_t stream) {
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, h, static_cast<uint64_t>(p.F), static_cast<uint64_t>(p.R), kBK, kBM) ||
        !make_tmap(&tb, w2, static_cast<uint64_t>(p.F), static_cast<uint64_t>(p.E) * p.D, kBK, kBN2))
        return MOE_ERR_CUDA;
    GemmArgs a = row_args(p, p.F / kBK);
    a.perm = perm;
    a.scores = scores;
    a.scores_bf16 = scores_dtype == MOE_SCORES_BF16 ? 1 : 0;
    a.out0 = static_cast<__nv_bfloat16*>(y);
    a.fout = rms_sumsq;
    const int grid = row_grid(p, static_cast<int32_t>(ceil_div(p.D, kBN2)));
    return rms_sumsq ? launch_gemm<FwdDownT<true>>(ta, tb, a, grid, stream)
                     : launch_gemm<FwdDownT<false>>(ta, tb, a, grid, stream);
}

moe_status_t launch_fused_gemms(const GemmProblem& p, const int32_t* tiles2, const void* xp, const void* w13, void* h,
                                const void* w2, const int32_t* perm, const void* scores, int32_t scores_dtype, void* y,
                                uint32_t* ready, cudaStream_t stream) {
    GemmMaps maps{};
    if (!make_tmap(&maps.m[0], xp, static_cast<uint64_t>(p.D), static_cast<uint64_t>(p.R), kBK, kBM) ||
        !make_tmap(&maps.m[1], w13, static_cast<uint64_t>(p.D), static_cast<uint64_t>(p.E) * 2 * p.F, kBK, kBN1) ||
        !make_tmap(&maps.m[2], h, static_cast<uint64_t>(p.F), static_cast<uint64_t>(p.R), kBK, kBM) ||
        !make_tmap(&maps.m[3], w2, static_cast<uint64_t>(p.F), static_cast<uint64_t>(p.E) * p.D, kBK, kBN2))
        return MOE_ERR_CUDA;
    GemmArgs a = row_args(p, p.D / kBK);
    a.out0 = static_cast<__nv_bfloat16*>(h);  // phase 0 writes H ...
    a.tiles_b = tiles2;
    a.kblocks_b = p.F / kBK;
    a.ntn = static_cast<int32_t>(ceil_div(p.F, kBN1));
    a.ntn_b = static_cast<int32_t>(ceil_div(p.D, kBN2));
    a.ticket = ready;       // the grid's tile counter, then (128 bytes on) one counter per row tile
    a.ready = ready + 32;
    a.perm = perm;
    a.scores = scores;
    a.scores_bf16 = scores_dtype == MOE_SCORES_BF16 ? 1 : 0;
    a.out1 = static_cast<__nv_bfloat16*>(y);
    return launch_gemm<FwdMega>(maps, a, row_grid(p, a.ntn + a.ntn_b), stream);
}

}  // namespace moe
