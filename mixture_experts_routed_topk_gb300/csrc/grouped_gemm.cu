// grouped_gemm.cu -- the two grouped expert GEMMs of the routed-experts forward pass on sm_103a.
//
//   gate/up GEMM + SwiGLU (TeraMoE README, compute worker: "gate/up projection, activation"; the
//   Dist-MoE execution model's W13 then SwiGLU):
//       H[r, f] = SiLU( XP[r,:] . Wg[e,f,:] ) * ( XP[r,:] . Wu[e,f,:] )      rows r of expert e
//   down GEMM + score (the compute worker's down projection; the combine worker's weighting):
//       Y[p, d] = score[p] * ( H[r,:] . W2[e,d,:] ),   p = perm[r]
//
// Design (one kernel template, two epilogues):
//  * Persistent: grid = number of SMs; CTA c takes tiles c, c + grid, ... of a device-built tile
//    list (expert e owns ceil(n_e/128) row tiles x the column tiles, rows fastest, so concurrent
//    CTAs share the same weight tile through L2). No host synchronisation: the list's length is
//    read on the device.
//  * Warp-specialised, 6 warps: warp 0 issues TMA loads, warp 1 owns TMEM and issues tcgen05.mma
//    from one thread, warps 2-5 are the epilogue (one TMEM lane = one output row per thread).
//  * Operands: TMA 2-D tiles with 128-byte swizzle into a 4-stage shared-memory ring (16 KB of A +
//    32 KB of B per stage), full/empty mbarriers between producer and MMA.
//  * Accumulators: 2 x 256 fp32 TMEM columns (all 512), so the epilogue of tile i overlaps the
//    mainloop of tile i+1; tcgen05.commit signals "accumulator full", the epilogue warps signal
//    "accumulator empty".
//  * Ragged expert segments need no padding: a tile's 128-row TMA box may run into the next
//    expert's rows (computed, not stored) or past the end (zero-filled by TMA).
//  * Expert weights are addressed by row offset in one tensor per projection: expert e's gate rows
//    start at row e*2F of w13 viewed as [E*2F, D], its up rows at e*2F + F, its W2 rows at e*D of
//    w2 viewed as [E*D, F] (the MoonEP FAQ's single contiguous weight tensor per projection).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "moe_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB: 128 rows x 64 bf16
constexpr int kBRows = 256;              // accumulator columns per tile
constexpr int kBBytes = kBRows * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kGemmThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows);

struct alignas(8) PipeState {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kGemmSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(PipeState);

struct GemmArgs {
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* tiles;
    int32_t E;
    int32_t kblocks;  // K extent / 64
    int32_t D, F;
    __nv_bfloat16* H;      // gate/up output [R, F]
    const int32_t* perm;   // down: row -> pair
    const void* scores;    // down: [T*K] fp32 or bf16
    int32_t scores_bf16;
    __nv_bfloat16* Y;      // down output [T*K, D]
    uint32_t* status;
};

struct Tile {
    int32_t e, n, row0, rows;
};

// Tile index -> (expert, column tile, first row, valid rows). tiles[] is non-decreasing with
// tiles[E] = total; the owning expert is the last e with tiles[e] <= tile.
__device__ __forceinline__ Tile decode_tile(int32_t tile, const GemmArgs& a) {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.tiles + mid) <= tile) lo = mid;
        else hi = mid - 1;
    }
    const int32_t local = tile - __ldg(a.tiles + lo);
    const int32_t ne = __ldg(a.counts + lo);
    const int32_t mt = (ne + kBM - 1) / kBM;
    Tile t;
    t.e = lo;
    t.n = local / mt;
    const int32_t m = local - t.n * mt;
    t.row0 = __ldg(a.offsets + lo) + m * kBM;
    t.rows = min(kBM, ne - m * kBM);
    return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast, so tcgen05.ld (which needs
// the whole warp) is executed by all lanes or none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status, MOE_DEV_TIMEOUT) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The producer's walk over (tile, K step) pairs: tiles blockIdx.x, +gridDim.x, ...; K steps in order.
struct StepCursor {
    int32_t tile, kb;
    Tile t;
    int32_t brow0, brow1;
};

template <int kMode>
__device__ __forceinline__ void cursor_enter_tile(StepCursor& c, const GemmArgs& a) {
    c.t = decode_tile(c.tile, a);
    if (kMode == 1) {
        c.brow0 = c.t.e * 2 * a.F + c.t.n * kBN1;
        c.brow1 = c.brow0 + a.F;
    } else {
        c.brow0 = c.t.e * a.D + c.t.n * kBN2;
        c.brow1 = 0;
    }
}

// Advances by one K step; returns false past the last tile.
template <int kMode>
__device__ __forceinline__ bool cursor_next(StepCursor& c, const GemmArgs& a, int32_t total) {
    if (++c.kb < a.kblocks) return true;
    c.kb = 0;
    c.tile += gridDim.x;
    if (c.tile >= total) return false;
    cursor_enter_tile<kMode>(c, a);
    return true;
}

template <int kMode>  // 1: gate/up + SwiGLU, 2: down + score
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must start on 1024-byte boundaries of the shared address space
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    PipeState* ps = reinterpret_cast<PipeState*>(smem + kStages * kStageBytes);
    volatile int* abort_flag = &ps->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ps->full[s], 1);
            mbar_init(&ps->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ps->acc_full[b], 1);
            mbar_init(&ps->acc_empty[b], kEpilogueThreads);
        }
        mbar_init(&ps->drain, 1);
        ps->abort = 0;
        mbar_init_fence();
        tma_prefetch_descriptor(&tmap_a);
        tma_prefetch_descriptor(&tmap_b);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(&ps->tmem_base, kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    tcgen05_fence_after_sync();
    // everything above overlaps the previous kernel's tail; its outputs are read from here on
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = ps->tmem_base;
    const int32_t total = __ldg(args.tiles + args.E);

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0 && static_cast<int32_t>(blockIdx.x) < total) {
            StepCursor ld{static_cast<int32_t>(blockIdx.x), 0, {}, 0, 0};
            cursor_enter_tile<kMode>(ld, args);
            uint32_t it = 0;
            bool ok = true, more = true;
            while (more) {
                const uint32_t s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                if (!mbar_wait(&ps->empty[s], ph ^ 1u, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                uint8_t* sa = smem + s * kStageBytes;
                uint8_t* sb = sa + kABytes;
                mbar_arrive_expect_tx(&ps->full[s], kStageBytes);
                tma_load_2d(sa, &tmap_a, &ps->full[s], ld.kb * kBK, ld.t.row0);
                if (kMode == 1) {
                    tma_load_2d(sb, &tmap_b, &ps->full[s], ld.kb * kBK, ld.brow0);
                    tma_load_2d(sb + kBBytes / 2, &tmap_b, &ps->full[s], ld.kb * kBK, ld.brow1);
                } else {
                    tma_load_2d(sb, &tmap_b, &ps->full[s], ld.kb * kBK, ld.brow0);
                }
                ++it;
                more = cursor_next<kMode>(ld, args, total);
            }
            if (!ok) {
                // aborting: give the copies already issued time to land before the CTA exits
                const unsigned long long t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++tcount) {
                const uint32_t acc = tcount & 1u;
                const uint32_t aph = (tcount >> 1) & 1u;
                if (!mbar_wait(&ps->acc_empty[acc], aph ^ 1u, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tcgen05_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kAccCols;
                for (int32_t kb = 0; kb < args.kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(&ps->full[s], ph, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after_sync();
                    const uint32_t a0 = smem_addr(smem + s * kStageBytes);
                    const uint32_t b0 = a0 + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // each 16-element K step is 32 bytes further along the swizzled rows
                        mma_bf16_ss(d_tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32),
                                    kIdesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&ps->empty[s]);  // frees the stage once these MMAs have read it
                }
                if (!ok) break;
                mma_commit(&ps->acc_full[acc]);
            }
            if (!ok) {
                // aborting: wait (bounded) until every MMA issued so far has finished with TMEM
                mma_commit(&ps->drain);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&ps->drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue (warps 2-5)
        const int quarter = warp & 3;  // TMEM lanes this warp may access: 32*quarter .. +31
        const int row_in_tile = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t tcount = 0;
        for (int32_t tile = blockIdx.x; tile < total; tile += gridDim.x, ++tcount) {
            const Tile t = decode_tile(tile, args);
            const uint32_t acc = tcount & 1u;
            const uint32_t aph = (tcount >> 1) & 1u;
            if (!warp_wait(&ps->acc_full[acc], aph, abort_flag, args.status)) break;
            tcgen05_fence_after_sync();
            const uint32_t taddr = tmem_base + lane_base + acc * kAccCols;
            const bool valid = row_in_tile < t.rows;
            const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
            if (kMode == 1) {
#pragma unroll 1
                for (int c = 0; c < kBN1 / 32; ++c) {
                    __syncwarp();  // tcgen05.ld is .sync.aligned: reconverge after the masked store
                    uint32_t g[32], u[32];
                    tmem_ld_32cols(taddr + c * 32, g);
                    tmem_ld_32cols(taddr + kBN1 + c * 32, u);
                    tmem_ld_wait(g);
                    tmem_ld_tie(u);
                    const int32_t f0 = t.n * kBN1 + c * 32;
                    if (valid && f0 < args.F) {
                        uint32_t packed[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                            const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
                            const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
                            const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
                            packed[j] = pack_bf16x2(h0, h1);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(args.H + row * args.F + f0);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    }
                }
            } else {
                int32_t pair = 0;
                float score = 0.0f;
                if (valid) {
                    pair = __ldg(args.perm + row);
                    score = args.scores_bf16
                                ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(args.scores)[pair])
                                : __ldg(reinterpret_cast<const float*>(args.scores) + pair);
                }
#pragma unroll 1
                for (int c = 0; c < kBN2 / 32; ++c) {
                    __syncwarp();
                    uint32_t v[32];
                    tmem_ld_32cols(taddr + c * 32, v);
                    tmem_ld_wait(v);
                    const int32_t d0 = t.n * kBN2 + c * 32;
                    if (valid && d0 < args.D) {
                        uint32_t packed[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            packed[j] = pack_bf16x2(__uint_as_float(v[2 * j]) * score,
                                                    __uint_as_float(v[2 * j + 1]) * score);
                        uint4* dst = reinterpret_cast<uint4*>(args.Y + static_cast<int64_t>(pair) * args.D + d0);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    }
                }
            }
            tcgen05_fence_before_sync();
            mbar_arrive(&ps->acc_empty[acc]);
        }
    }

    tcgen05_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();  // lane 0 ran the MMA loop alone; .sync.aligned needs the whole warp
        tcgen05_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------------------------- host

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

// A 2-D bf16 tensor [rows, inner] (inner contiguous) read in boxes of 64 x box_rows with 128-byte
// swizzle; reads outside the tensor return zeros.
bool make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_smem_attr[2][kMaxDevices];

template <int kMode>
moe_status_t ensure_smem_attr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    if (!g_smem_attr[kMode - 1][dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(k_grouped_gemm<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmemBytes)) != cudaSuccess)
            return MOE_ERR_CUDA;
        g_smem_attr[kMode - 1][dev].store(true, std::memory_order_release);
    }
    return MOE_OK;
}

int gemm_grid(const GemmProblem& p, int32_t ntn) {
    // upper bound of the tile count: ceil(R/128) + (experts that can be non-empty), per column tile
    const int64_t nonempty = p.R < p.E ? p.R : p.E;
    const int64_t max_tiles = (ceil_div(p.R, kBM) + nonempty) * ntn;
    const int64_t g = max_tiles < p.sm_count ? max_tiles : p.sm_count;
    return static_cast<int>(g > 0 ? g : 1);
}

}  // namespace

moe_status_t launch_gemm1_swiglu(const GemmProblem& p, const void* xp, const void* w13, void* h,
                                 cudaStream_t stream) {
    moe_status_t st = ensure_smem_attr<1>();
    if (st != MOE_OK) return st;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, xp, static_cast<uint64_t>(p.D), static_cast<uint64_t>(p.R), kBM) ||
        !make_tmap(&tb, w13, static_cast<uint64_t>(p.D), static_cast<uint64_t>(p.E) * 2 * p.F, kBN1))
        return MOE_ERR_CUDA;
    GemmArgs a{};
    a.counts = p.counts;
    a.offsets = p.offsets;
    a.tiles = p.tiles;
    a.E = p.E;
    a.kblocks = p.D / kBK;
    a.D = p.D;
    a.F = p.F;
    a.H = static_cast<__nv_bfloat16*>(h);
    a.status = p.status;
    const int32_t ntn = static_cast<int32_t>(ceil_div(p.F, kBN1));
    return launch_pdl(k_grouped_gemm<1>, dim3(gemm_grid(p, ntn)), dim3(kGemmThreads), kGemmSmemBytes, stream, ta, tb,
                      a) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

moe_status_t launch_gemm2_score(const GemmProblem& p, const void* h, const void* w2, const int32_t* perm,
                                const void* scores, int32_t scores_dtype, void* y, cudaStream_t stream) {
    moe_status_t st = ensure_smem_attr<2>();
    if (st != MOE_OK) return st;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, h, static_cast<uint64_t>(p.F), static_cast<uint64_t>(p.R), kBM) ||
        !make_tmap(&tb, w2, static_cast<uint64_t>(p.F), static_cast<uint64_t>(p.E) * p.D, kBN2))
        return MOE_ERR_CUDA;
    GemmArgs a{};
    a.counts = p.counts;
    a.offsets = p.offsets;
    a.tiles = p.tiles;
    a.E = p.E;
    a.kblocks = p.F / kBK;
    a.D = p.D;
    a.F = p.F;
    a.perm = perm;
    a.scores = scores;
    a.scores_bf16 = scores_dtype == MOE_SCORES_BF16 ? 1 : 0;
    a.Y = static_cast<__nv_bfloat16*>(y);
    a.status = p.status;
    const int32_t ntn = static_cast<int32_t>(ceil_div(p.D, kBN2));
    return launch_pdl(k_grouped_gemm<2>, dim3(gemm_grid(p, ntn)), dim3(kGemmThreads), kGemmSmemBytes, stream, ta, tb,
                      a) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

}  // namespace moe
