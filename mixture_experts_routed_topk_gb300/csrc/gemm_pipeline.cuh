// gemm_pipeline.cuh -- the persistent, warp-specialised tcgen05 GEMM pipeline shared by every
// grouped GEMM of the library (forward and backward), generic over a tile policy.
//
// One CTA per SM walks tiles c, c + grid, ... of a tile list the policy defines (or claims them in
// list order from a global counter, see kDynamicSchedule). Warp 0 issues TMA loads into a
// shared-memory ring of stages, warp 1 owns all 512 TMEM columns and issues tcgen05.mma from one
// thread into one of two fp32 accumulators, warps 2-5 run the policy's epilogue from TMEM (one
// TMEM lane = one output row per thread). full/empty mbarriers link producer and MMA;
// acc_full/acc_empty link MMA and epilogue, so a tile's epilogue overlaps the next tile's
// mainloop. The producer and the MMA thread decode the next tile while the current one's first
// stage is in flight, so no decode sits between two tiles' MMAs. Every wait is bounded.
//
// The policy's Shape fixes the ring and the MMA kind (Bf16Shape unless the policy names another):
//   Bf16Shape: 4 stages of 16 KB A + 32 KB B (64 bf16 of K), 128 x 256 accumulators, kind::f16.
//   Nvf4Shape: 5 stages of 16 KB A + 16 KB B (256 packed E2M1 of K) + 4 KB of UE4M3 scale chunks,
//              128 x 128 accumulators, kind::mxf4nvf4 block-scaled (four scale chunks per operand
//              per stage, one per K=64 MMA). The scale chunks are loaded on their own barrier and
//              written into the stage's TMEM slot by four more warps (6-9, one per TMEM lane
//              quarter) with tcgen05.st, so the MMA thread issues only MMAs.
//   Mxf8Shape: 4 stages of 16 KB A + 24 KB B (128 E4M3 of K) + their UE8M0 scale chunks (512 B
//              for A's 128 rows, 1 KB for B's 192 rows), 128 x 192 accumulators (TMEM columns
//              0..191 and 256..447), kind::mxf8f6f4 block-scaled; the MMA thread copies a stage's
//              scales into that stage's 32-column TMEM slot (192, 224, 448, 480) with tcgen05.cp
//              right before the stage's MMAs.
//
// A policy P provides
//   struct P::Tile { int32_t kblocks; ... }              one tile's coordinates and K steps
//   static constexpr uint32_t kIdesc                     tcgen05 instruction descriptor
//   static constexpr bool kAMnMajor, kBMnMajor           operand layouts in shared memory
//   __device__ static int32_t num_tiles(const GemmArgs&)
//   __device__ static Tile decode(int32_t tile, const GemmArgs&)
//   __device__ static void load(const Tile&, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
//                               const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs&)
//   block-scaled shapes also:
//   __device__ static void load_scales(const Tile&, int32_t kb, uint8_t* sf, uint64_t* bar,
//                                      const GemmArgs&)    the stage's A then B scale chunks
//   __device__ static void epilogue(const Tile&, uint32_t taddr, int row, uint4* stage,
//                                   const GemmArgs&)          (taddr = this warp's TMEM lanes)
// Every load() must deliver exactly the shape's kTxBytes (or tx_bytes(t)) into the stage (with
// load_scales() when the MMA thread copies the scales; kSfaBytes + kSfbBytes on their own barrier
// when warps write them). ta and tb point into the
// kernel's array of four tensor maps (tb == ta + 1); a policy with more operands reads ta[2], ta[3].
// Optional:
//   __device__ static bool acquire(const Tile&, const GemmArgs&, volatile int* abort)
//        run by the producer before a tile's first load: waits (bounded) until data that other
//        CTAs of the same grid produce for this tile is visible to TMA; false aborts the CTA.
//        Requires kDynamicSchedule and a list whose tiles depend only on earlier tiles: then only
//        running CTAs hold tiles, so the wait never depends on a CTA that has not started.
//   __device__ static uint32_t idesc(const Tile&), tx_bytes(const Tile&)
//        per-tile instruction descriptor and stage transaction bytes, for policies whose tiles
//        differ in N (default: kIdesc and the shape's kTxBytes)
//   static constexpr bool kDynamicSchedule = true
//        CTAs take tiles in list order from the global counter args.ticket (zero on entry)
//        instead of the fixed c, c + grid, ...: the producer takes a tile, decodes it and hands it
//        to the MMA and epilogue warps through a small ring of shared-memory slots. For tile lists
//        of unequal tiles, where a fixed assignment lets CTAs drift apart along the list.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>
#include <utility>

#include "moe_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe {

constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;      // 16 KB: 128 rows x 64 bf16
constexpr int kBRows = 256;                 // accumulator columns per tile
constexpr int kBBytes = kBRows * kBK * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kMaxStages = 8;

struct Bf16Shape {
    static constexpr int kStages = moe::kStages;
    static constexpr int kABytes = moe::kABytes, kBBytes = moe::kBBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;  // a multiple of 1024
    static constexpr int kTxBytes = kABytes + kBBytes;
    static constexpr int kAccCols = moe::kAccCols;
    static constexpr bool kBlockScaled = false;
    static constexpr bool kScalesByWarps = false;
};

// E4M3 operands with UE8M0 block scales: kMxBK = 128 K elements (128 bytes, one swizzled row) per
// stage, kMxBN = 192 accumulator columns per tile.
struct Mxf8Shape {
    static constexpr int kStages = 4;
    static constexpr int kABytes = kBM * kMxBK;         // 16 KB
    static constexpr int kBBytes = kMxBN * kMxBK;       // 24 KB
    static constexpr int kSfaBytes = 512, kSfbBytes = 1024;
    static constexpr int kStageBytes = 43008;           // 16 + 24 + 1.5 KB, rounded up to 1024
    static constexpr int kTxBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kAccCols = 256;  // accumulators at TMEM columns 0 and 256, 192 wide each
    static constexpr bool kBlockScaled = true;
    // the MMA thread copies each stage's scales into the stage's slot (tcgen05.cp)
    static constexpr bool kScalesByWarps = false;
    // Scale slot of stage s (32 columns: A's scales at +0, B's at +16): in the two gaps after the
    // accumulators, columns 192..255 and 448..511.
    __device__ static constexpr uint32_t sf_slot_col(uint32_t s) { return (s & 2u) * 128u + 192u + 32u * (s & 1u); }
    // One A chunk (128 rows x 4 blocks of 32 = the stage's K) read by all four MMAs through the
    // scale-factor id; two B chunks (192 rows).
    static constexpr int kSfaChunks = 1, kSfbChunks = 2;
    __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t slot, int kk,
                               uint32_t acc) {
        mma_mxf8_ss(d, a, b, idesc | mxf8_ids(kk), slot, slot + 16u, acc);
    }
};

// Packed E2M1 operands with UE4M3 scales per 16: 256 K elements (128 bytes) per stage, four K=64
// MMAs, each with its own A and B scale chunk. 128 x 128 accumulators at TMEM columns 0 and 256;
// 32-column scale slots at 128, 160, 192, 224 and 384, one per stage (A's four chunks at +0..+15,
// B's at +16..+31).
//
// The scales reach TMEM through four scale warps (tcgen05.st), not through tcgen05.cp from the MMA
// thread: after a tcgen05.cp the MMA thread's next shared-memory access (its wait on the next
// stage's barrier) stalls until the copies have executed, which left the tensor pipe idle between
// stages (eight copies per stage here). A stage's scale chunks are loaded on their own barrier.
constexpr int kNvBN = 128;
struct Nvf4Shape {
    static constexpr int kStages = 5;
    static constexpr int kABytes = kBM * 128;           // 16 KB
    static constexpr int kBBytes = kNvBN * 128;         // 16 KB
    static constexpr int kSfaBytes = 2048, kSfbBytes = 2048;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;  // 36 KB
    static constexpr int kTxBytes = kABytes + kBBytes;  // the operand boxes (scales: their own barrier)
    static constexpr int kAccCols = 256;
    static constexpr bool kBlockScaled = true;
    static constexpr bool kScalesByWarps = true;
    __device__ static constexpr uint32_t sf_slot_col(uint32_t s) { return s < 4u ? 128u + 32u * s : 384u; }
    static constexpr int kSfaChunks = 4, kSfbChunks = 4;
    __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t slot, int kk,
                               uint32_t acc) {
        mma_nvf4_ss(d, a, b, idesc, slot + 4u * kk, slot + 16u + 4u * kk, acc);
    }
};
static_assert(Nvf4Shape::kStageBytes % 1024 == 0 && Nvf4Shape::kStages == 5, "stage ring / scale slots");
static_assert(Mxf8Shape::kStageBytes % 1024 == 0 && Mxf8Shape::kTxBytes <= Mxf8Shape::kStageBytes, "stage");
static_assert(Mxf8Shape::kSfaChunks <= 4 && Mxf8Shape::kSfbChunks <= 4 && Nvf4Shape::kSfaChunks <= 4 &&
                  Nvf4Shape::kSfbChunks <= 4,
              "a scale slot holds four chunks of A at columns 0..15 and four of B at 16..31");
static_assert(Mxf8Shape::kStages == 4 && kMxBN + 64 == Mxf8Shape::kAccCols, "four 32-column scale slots in the gaps");

// The kernel's tensor maps: A and B of the policy's GEMM, then two more for policies that run
// two GEMMs in one grid. Passed as one __grid_constant__ parameter, so TMA reads them from the
// parameter space.
struct GemmMaps {
    CUtensorMap m[4];
};

template <class P, class = void>
struct ShapeOf {
    using type = Bf16Shape;
};
template <class P>
struct ShapeOf<P, std::void_t<typename P::Shape>> {
    using type = typename P::Shape;
};
constexpr int kGemmThreads = 192;
constexpr int kEpilogueThreads = 128;
// Shapes whose scales are written by warps add four warps (one per TMEM lane quarter) that write
// each K step's scale factors into TMEM.
constexpr int kScaleWarps = 4;
template <class S>
constexpr int gemm_threads() {
    return kGemmThreads + (S::kScalesByWarps ? 32 * kScaleWarps : 0);
}
constexpr int kMnBoxBytes = 64 * kBK * 2;   // one 64 (M or N) x 64 (K) MN-major box: 8 KB

// Epilogue staging: each epilogue warp owns 32 rows x 128 bytes (+16 bytes of padding per row, so
// that both the per-thread row writes and the per-row reads are free of bank conflicts).
constexpr int kStageRowU4 = 9;  // 144-byte row stride in 16-byte units
constexpr int kEpilogueStagingBytes = (kEpilogueThreads / 32) * 32 * kStageRowU4 * 16;

constexpr int kTileRing = 4;  // tiles in flight between producer and consumers (dynamic schedule)
constexpr int kTileStoreBytes = 48;

struct alignas(16) PipeState {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t sf_loaded[kMaxStages];  // scales by warps: the stage's scale chunks are in shared memory
    uint64_t sf_full[kMaxStages];    // scales by warps: the stage's scales are in its TMEM slot
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t tile_full[kTileRing];   // producer -> MMA + epilogue: a tile is in the slot
    uint64_t tile_empty[kTileRing];  // MMA + 4 epilogue warps -> producer: the slot was read
    uint32_t tile_ring[kTileRing];   // the tile's index in the list (>= the tile count: no more tiles)
    alignas(16) uint8_t tile_store[kTileRing][kTileStoreBytes];  // the producer's decode of it
    uint32_t tmem_base;
    int abort;
};

template <class S>
constexpr size_t gemm_smem_bytes() {
    return 1024 + static_cast<size_t>(S::kStages) * S::kStageBytes + kEpilogueStagingBytes + sizeof(PipeState);
}
static_assert(gemm_smem_bytes<Mxf8Shape>() <= 232448 && gemm_smem_bytes<Bf16Shape>() <= 232448 &&
                  gemm_smem_bytes<Nvf4Shape>() <= 232448,
              "smem");

// Everything any policy needs (each policy reads its own fields).
struct GemmArgs {
    const int32_t* counts;   // [E] routed rows per expert
    const int32_t* offsets;  // [E+1] first routed row per expert
    const int32_t* tiles;    // [E+1] forward tile prefix
    const int32_t* pmt;      // [E+1] padded 128-row tile prefix (backward)
    const int32_t* perm;     // routed row -> pair
    const int32_t* pperm;    // padded row -> pair, or -1 (backward)
    int32_t E;
    int32_t kblocks;         // K extent / 64 for fixed-K policies
    int32_t D, F;
    int32_t mdim, ndim;      // weight-gradient output rows / columns
    int32_t mtiles, ntiles;  // weight-gradient tile grid per expert
    const void* scores;      // [T*K] fp32 or bf16
    int32_t scores_bf16;
    __nv_bfloat16* out0;     // policy output 1
    __nv_bfloat16* out1;     // policy output 2
    const __nv_bfloat16* in0;  // extra epilogue input
    float* fout;             // fp32 policy output
    uint32_t* status;
    // block-scaled (MXFP8) policies
    const uint8_t* sf_a;     // A's UE8M0 scale chunks
    const uint8_t* sf_b;     // B's UE8M0 scale chunks
    uint8_t* q_out;          // E4M3 output codes
    uint8_t* sf_out;         // the output's scale chunks
    int32_t ntn;             // column tiles per row tile
    // two-GEMM grids (the fused forward): the second GEMM's tile prefix, K steps and column tiles,
    // and one readiness counter per row tile, counting first-GEMM epilogue warps that finished
    const int32_t* tiles_b;
    int32_t kblocks_b;
    int32_t ntn_b;
    uint32_t* ready;
    uint32_t* ticket;        // dynamic schedule: the next unclaimed tile of the list
    float act_scale_a;       // NVFP4: tensor scale of the A operand's activations
    float act_scale_out;     // NVFP4: tensor scale used to quantize the epilogue's output
};

template <class P, class = void>
struct HasAcquire : std::false_type {};
template <class P>
struct HasAcquire<P, std::void_t<decltype(P::acquire(std::declval<const typename P::Tile&>(),
                                                       std::declval<const GemmArgs&>(),
                                                       std::declval<volatile int*>()))>> : std::true_type {};

template <class P, class = void>
struct HasTileShape : std::false_type {};
template <class P>
struct HasTileShape<P, std::void_t<decltype(P::idesc(std::declval<const typename P::Tile&>())),
                                   decltype(P::tx_bytes(std::declval<const typename P::Tile&>()))>>
    : std::true_type {};

template <class P, class = void>
struct IsDynamic : std::false_type {};
template <class P>
struct IsDynamic<P, std::void_t<decltype(P::kDynamicSchedule)>> : std::integral_constant<bool, P::kDynamicSchedule> {};


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Logistic sigmoid and SiLU for the SwiGLU epilogues: exp through the hardware exp2 and the
// quotient through the reciprocal approximation (__fdividef, 2 ulp). An IEEE-rounded division
// here made the gate/up epilogue slower than the block-scaled mainloop it overlaps. For g below
// about -87 the denominator exceeds 2^126 and the result is 0 (the exact value is below 2^-120).
__device__ __forceinline__ float sigmoid_fast(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ float pair_score(const GemmArgs& a, int32_t pair) {
    return a.scores_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.scores)[pair])
                         : __ldg(reinterpret_cast<const float*>(a.scores) + pair);
}

// The expert owning `tile` in a tile list whose prefix is ntn * prefix[e]: the last e with
// ntn * prefix[e] <= tile.
__device__ __forceinline__ int32_t owning_expert(int32_t tile, const int32_t* prefix, int32_t ntn, int32_t E) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ntn * __ldg(prefix + mid) <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast, so tcgen05.ld (which needs
// the whole warp) is executed by all lanes or none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status, MOE_DEV_TIMEOUT) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Writes, for every lane of the warp, 64 bf16 (128 bytes, packed two per 32-bit word) to that
// lane's own row. Lane i's words go to its staging row first; then lane l copies 16-byte piece
// (l & 7) of row (4 j + l / 8) for j = 0..7, so one store instruction covers four complete
// 128-byte row segments. dst: this lane's destination (16-byte aligned); ok: whether this lane's
// row is stored at all.
__device__ __forceinline__ void warp_store_row_segments(uint4* stage, const uint32_t (&words)[32], char* dst,
                                                        bool ok) {
    const int lane = threadIdx.x & 31;
    uint4* mine = stage + lane * kStageRowU4;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        mine[c] = make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
    __syncwarp();
    const unsigned long long my_dst = reinterpret_cast<unsigned long long>(dst);
    const int my_ok = ok ? 1 : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = 4 * j + (lane >> 3);
        const int piece = lane & 7;
        const unsigned long long rd = __shfl_sync(0xffffffffu, my_dst, r);
        const int rok = __shfl_sync(0xffffffffu, my_ok, r);
        if (rok) reinterpret_cast<uint4*>(rd)[piece] = stage[r * kStageRowU4 + piece];
    }
    __syncwarp();
}

// The inverse: reads, for every lane of the warp, 64 bf16 (128 bytes) of that lane's own row, where
// row i of the warp starts at base + i * row_stride bytes (16-byte aligned). Lane l loads 16-byte
// piece (l & 7) of rows 4 j + l / 8 (j = 0..7), so each load instruction covers four whole 128-byte
// row segments; the pieces meet in the staging rows and each lane takes its own row back as 32
// packed words.
__device__ __forceinline__ void warp_load_row_segments(uint4* stage, const char* base, int64_t row_stride,
                                                       uint32_t (&words)[32]) {
    const int lane = threadIdx.x & 31;
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        v[j] = __ldg(reinterpret_cast<const uint4*>(base + (4 * j + (lane >> 3)) * row_stride) + (lane & 7));
#pragma unroll
    for (int j = 0; j < 8; ++j) stage[(4 * j + (lane >> 3)) * kStageRowU4 + (lane & 7)] = v[j];
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 x = stage[lane * kStageRowU4 + c];
        words[4 * c] = x.x;
        words[4 * c + 1] = x.y;
        words[4 * c + 2] = x.z;
        words[4 * c + 3] = x.w;
    }
    __syncwarp();
}

// 16 packed words (32 bf16 = 64 bytes) to a 16-byte-aligned address.
__device__ __forceinline__ void store_64B(void* dst, const uint32_t (&w)[16]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// Shared-memory operand descriptor of the 16-wide K step kk of a stage operand at `base`.
template <bool kMnMajor>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
    // K-major: each K step is 32 bytes further along the swizzled 128-byte rows.
    // MN-major: each K step is 16 rows of 128 bytes further down the 64-wide MN blocks.
    return kMnMajor ? sw128_mnmajor_desc(base + kk * 2048, kMnBoxBytes) : sw128_kmajor_desc(base + kk * 32);
}

template <class P>
__global__ void __launch_bounds__(gemm_threads<typename ShapeOf<P>::type>(), 1)
    k_grouped_gemm(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
    using S = typename ShapeOf<P>::type;
    const CUtensorMap* tmap_a = &maps.m[0];
    const CUtensorMap* tmap_b = &maps.m[1];
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must start on 1024-byte boundaries of the shared address space
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    uint4* staging = reinterpret_cast<uint4*>(smem + S::kStages * S::kStageBytes);
    PipeState* ps = reinterpret_cast<PipeState*>(smem + S::kStages * S::kStageBytes + kEpilogueStagingBytes);
    volatile int* abort_flag = &ps->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(&ps->full[s], 1);
            mbar_init(&ps->empty[s], 1);
            mbar_init(&ps->sf_loaded[s], 1);
            mbar_init(&ps->sf_full[s], kScaleWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ps->acc_full[b], 1);
            mbar_init(&ps->acc_empty[b], kEpilogueThreads);
        }
        mbar_init(&ps->drain, 1);
        for (int r = 0; r < kTileRing; ++r) {
            mbar_init(&ps->tile_full[r], 1);
            mbar_init(&ps->tile_empty[r], 1 + kEpilogueThreads / 32);
        }
        ps->abort = 0;
        mbar_init_fence();
        tma_prefetch_descriptor(tmap_a);
        tma_prefetch_descriptor(tmap_b);
        if constexpr (HasAcquire<P>::value) {
            tma_prefetch_descriptor(&maps.m[2]);
            tma_prefetch_descriptor(&maps.m[3]);
        }
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
    const int32_t total = P::num_tiles(args);
    constexpr bool kDynamic = IsDynamic<P>::value;
    static_assert(!HasAcquire<P>::value || kDynamic, "a tile that waits for other tiles needs the dynamic schedule");
    static_assert(!(kDynamic && S::kScalesByWarps), "the scale warps follow the static schedule");
    static_assert(!kDynamic || (sizeof(typename P::Tile) <= kTileStoreBytes &&
                                std::is_trivially_copyable<typename P::Tile>::value),
                  "a dynamically scheduled policy's tiles travel through the shared-memory ring");

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            // tile indices are compared unsigned: the list has fewer than 2^31 tiles, and the end
            // marks and the last claimed tickets lie at most a few grids past its end
            const uint32_t utotal = static_cast<uint32_t>(total);
            // The next tile is claimed and decoded one tile ahead, right after the current tile's
            // first stage is issued, so neither the claim nor the decode delays the first loads of
            // a tile (the stage ring covers them).
            uint32_t tile = kDynamic ? atomicAdd(args.ticket, 1u) : blockIdx.x;
            typename P::Tile t{};
            if (tile < utotal) t = P::decode(static_cast<int32_t>(tile), args);
            for (uint32_t i = 0; ok; ++i) {
                uint32_t next;
                if constexpr (kDynamic) {
                    // hand the tile, decoded (or the end mark, any index >= total), to the MMA and
                    // epilogue warps
                    const uint32_t r = i % kTileRing, rph = (i / kTileRing) & 1u;
                    if (!mbar_wait(&ps->tile_empty[r], rph ^ 1u, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    ps->tile_ring[r] = tile;
                    *reinterpret_cast<typename P::Tile*>(ps->tile_store[r]) = t;
                    mbar_arrive(&ps->tile_full[r]);
                    if (tile >= utotal) break;
                    next = atomicAdd(args.ticket, 1u);  // its value is first needed after stage 0
                } else {
                    if (tile >= utotal) break;
                    next = tile + gridDim.x;
                }
                if constexpr (HasAcquire<P>::value) {
                    if (!P::acquire(t, args, abort_flag)) {
                        ok = false;
                        break;
                    }
                }
                typename P::Tile nt{};
                bool decoded = false;
                for (int32_t kb = 0; kb < t.kblocks; ++kb, ++it) {
                    const uint32_t s = it % S::kStages;
                    const uint32_t ph = (it / S::kStages) & 1u;
                    if (!mbar_wait(&ps->empty[s], ph ^ 1u, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + s * S::kStageBytes;
                    if constexpr (S::kScalesByWarps) {  // the small scale chunks first, on their own barrier
                        mbar_arrive_expect_tx(&ps->sf_loaded[s], S::kSfaBytes + S::kSfbBytes);
                        P::load_scales(t, kb, sa + S::kABytes + S::kBBytes, &ps->sf_loaded[s], args);
                    }
                    if constexpr (HasTileShape<P>::value) mbar_arrive_expect_tx(&ps->full[s], P::tx_bytes(t));
                    else mbar_arrive_expect_tx(&ps->full[s], S::kTxBytes);
                    P::load(t, kb, sa, sa + S::kABytes, &ps->full[s], tmap_a, tmap_b, args);
                    if constexpr (S::kBlockScaled && !S::kScalesByWarps)  // with the operands
                        P::load_scales(t, kb, sa + S::kABytes + S::kBBytes, &ps->full[s], args);
                    if (!decoded) {
                        if (next < utotal) nt = P::decode(static_cast<int32_t>(next), args);
                        decoded = true;
                    }
                }
                if (!ok) break;
                if (!decoded && next < utotal) nt = P::decode(static_cast<int32_t>(next), args);
                tile = next;
                t = nt;
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
            uint32_t it = 0;
            bool ok = true;
            // static schedule: each tile is decoded during the previous one (after its first MMAs
            // are issued), so the decode never leaves the tensor pipe idle between tiles
            typename P::Tile t{}, nt{};
            if (!kDynamic && blockIdx.x < static_cast<uint32_t>(total)) nt = P::decode(static_cast<int32_t>(blockIdx.x), args);
            for (uint32_t tcount = 0; ok; ++tcount) {
                uint32_t tile;
                if constexpr (kDynamic) {
                    const uint32_t r = tcount % kTileRing, rph = (tcount / kTileRing) & 1u;
                    if (!mbar_wait(&ps->tile_full[r], rph, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tile = ps->tile_ring[r];
                    t = *reinterpret_cast<const typename P::Tile*>(ps->tile_store[r]);
                    mbar_arrive(&ps->tile_empty[r]);
                } else {
                    tile = blockIdx.x + tcount * gridDim.x;
                    t = nt;  // decoded during the previous tile
                }
                if (tile >= static_cast<uint32_t>(total)) break;
                const uint32_t next = tile + gridDim.x;  // static schedule only
                bool decoded = kDynamic;
                const uint32_t acc = tcount & 1u;
                const uint32_t aph = (tcount >> 1) & 1u;
                if (!mbar_wait(&ps->acc_empty[acc], aph ^ 1u, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tcgen05_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * S::kAccCols;
                uint32_t idesc = P::kIdesc;
                if constexpr (HasTileShape<P>::value) idesc = P::idesc(t);
                for (int32_t kb = 0; kb < t.kblocks; ++kb, ++it) {
                    const uint32_t s = it % S::kStages;
                    const uint32_t ph = (it / S::kStages) & 1u;
                    if (!mbar_wait(&ps->full[s], ph, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after_sync();
                    const uint32_t a0 = smem_addr(smem + s * S::kStageBytes);
                    const uint32_t b0 = a0 + S::kABytes;
                    if constexpr (S::kScalesByWarps) {
                        // the scale warps have written this stage's scales into its TMEM slot
                        if (!mbar_wait(&ps->sf_full[s], ph, abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                        tcgen05_fence_after_sync();
                        const uint32_t slot = tmem_base + S::sf_slot_col(s);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // 128-byte stage rows, 32 bytes of K per MMA
                            S::mma(d_tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32),
                                   idesc, slot, kk, (kb | kk) != 0 ? 1u : 0u);
                    } else if constexpr (S::kBlockScaled) {
                        // this stage's scales into its TMEM slot; the slot's previous reader (the MMAs
                        // of stage use it - kStages) completed before the stage was refilled
                        const uint32_t sf0 = b0 + S::kBBytes;  // A's chunks, then B's, 512 bytes each
                        const uint32_t slot = tmem_base + S::sf_slot_col(s);
#pragma unroll
                        for (int c = 0; c < S::kSfaChunks; ++c)
                            tmem_cp_scale_chunk(slot + 4u * c, sf_chunk_desc(sf0 + 512 * c));
#pragma unroll
                        for (int c = 0; c < S::kSfbChunks; ++c)
                            tmem_cp_scale_chunk(slot + 16u + 4u * c, sf_chunk_desc(sf0 + S::kSfaBytes + 512 * c));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // 128-byte stage rows, 32 bytes of K per MMA
                            S::mma(d_tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32),
                                   idesc, slot, kk, (kb | kk) != 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16_ss(d_tmem, operand_desc<P::kAMnMajor>(a0, kk),
                                        operand_desc<P::kBMnMajor>(b0, kk), idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&ps->empty[s]);  // frees the stage once these MMAs have read it
                    if (!decoded) {
                        if (next < static_cast<uint32_t>(total)) nt = P::decode(static_cast<int32_t>(next), args);
                        decoded = true;
                    }
                }
                if (!ok) break;
                if (!decoded && next < static_cast<uint32_t>(total)) nt = P::decode(static_cast<int32_t>(next), args);
                mma_commit(&ps->acc_full[acc]);  // a tile without K steps signals at once
            }
            if (!ok) {
                // aborting: wait (bounded) until every MMA issued so far has finished with TMEM
                mma_commit(&ps->drain);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&ps->drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else if (warp >= 2 + kEpilogueThreads / 32) {
        // ------------------------------------------------------------------ scale warps (6-9)
        // Scales by warps only. For every stage, each warp writes the stage's scale chunks into
        // the stage's TMEM slot for its own 32-lane quarter: chunk c of A at slot columns
        // 4c .. 4c+3, chunk c of B at 16 + 4c .. 16 + 4c + 3, lane l of the quarter taking the
        // chunk's 16 bytes at 16 l (rows l, 32 + l, 64 + l, 96 + l of the chunk's 128 rows, one per
        // column): the layout the block-scaled MMAs read. The slot's previous reader (the MMAs of
        // the stage's previous use) completed before the stage was refilled.
        if constexpr (S::kScalesByWarps) {
            const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const uint32_t tile = blockIdx.x + tcount * gridDim.x;
                if (tile >= static_cast<uint32_t>(total)) break;
                const int32_t kblocks = P::decode(static_cast<int32_t>(tile), args).kblocks;
                for (int32_t kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % S::kStages;
                    const uint32_t ph = (it / S::kStages) & 1u;
                    if (!warp_wait(&ps->sf_loaded[s], ph, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after_sync();
                    const uint8_t* sf = smem + s * S::kStageBytes + S::kABytes + S::kBBytes;
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
#pragma unroll
                    for (int c = 0; c < S::kSfaChunks; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4*>(sf + 512 * c + 16 * lane);
                        r[4 * c] = v.x, r[4 * c + 1] = v.y, r[4 * c + 2] = v.z, r[4 * c + 3] = v.w;
                    }
#pragma unroll
                    for (int c = 0; c < S::kSfbChunks; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4*>(sf + S::kSfaBytes + 512 * c + 16 * lane);
                        r[16 + 4 * c] = v.x, r[17 + 4 * c] = v.y, r[18 + 4 * c] = v.z, r[19 + 4 * c] = v.w;
                    }
                    tmem_st_32cols(tmem_base + lane_base + S::sf_slot_col(s), r);
                    tmem_st_wait();
                    tcgen05_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ps->sf_full[s]);
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue (warps 2-5)
        const int quarter = warp & 3;  // TMEM lanes this warp may access: 32*quarter .. +31
        const int row_in_tile = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint4* wstage = staging + (warp - 2) * 32 * kStageRowU4;
        for (uint32_t tcount = 0;; ++tcount) {
            uint32_t tile;
            typename P::Tile t;
            if constexpr (kDynamic) {
                const uint32_t r = tcount % kTileRing, rph = (tcount / kTileRing) & 1u;
                if (!warp_wait(&ps->tile_full[r], rph, abort_flag, args.status)) break;
                __syncwarp();  // orders every lane's reads of the slot after lane 0's wait
                tile = ps->tile_ring[r];
                t = *reinterpret_cast<const typename P::Tile*>(ps->tile_store[r]);
                __syncwarp();  // every lane has read the slot
                if (lane == 0) mbar_arrive(&ps->tile_empty[r]);
                if (tile >= static_cast<uint32_t>(total)) break;
            } else {
                tile = blockIdx.x + tcount * gridDim.x;
                if (tile >= static_cast<uint32_t>(total)) break;
                t = P::decode(static_cast<int32_t>(tile), args);
            }
            const uint32_t acc = tcount & 1u;
            const uint32_t aph = (tcount >> 1) & 1u;
            if (!warp_wait(&ps->acc_full[acc], aph, abort_flag, args.status)) break;
            tcgen05_fence_after_sync();
            P::epilogue(t, tmem_base + lane_base + acc * S::kAccCols, row_in_tile, wstage, args);
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

// A 2-D bf16 tensor [rows, inner] (inner contiguous) read in boxes of box_inner x box_rows with
// 128-byte swizzle; reads outside the tensor return zeros.
bool make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows);

// The same for a byte tensor (E4M3 codes): inner and box_inner count bytes.
// A byte tensor [halves, rows, inner] read in boxes of box_inner x box_rows x 2: two consecutive
// halves (the gate and the up rows of one expert's w13, halves = 2 E) in one copy, written to
// shared memory as the first half's box_rows rows, then the second's.
bool make_tmap_u8_pairs(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t halves,
                        uint32_t box_inner, uint32_t box_rows);

bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows);

int sm_count_grid(int64_t max_tiles, int sm_count);

template <class P>
moe_status_t launch_gemm(const GemmMaps& maps, const GemmArgs& a, int grid, cudaStream_t stream) {
    constexpr size_t kGemmSmemBytes = gemm_smem_bytes<typename ShapeOf<P>::type>();
    constexpr int kMaxDevices = 64;
    static std::atomic<bool> attr_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(k_grouped_gemm<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmemBytes)) != cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_grouped_gemm<P>, dim3(grid), dim3(gemm_threads<typename ShapeOf<P>::type>()),
                      kGemmSmemBytes, stream, maps, a) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

template <class P>
moe_status_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int grid,
                         cudaStream_t stream) {
    GemmMaps maps{};
    maps.m[0] = ta;
    maps.m[1] = tb;
    return launch_gemm<P>(maps, a, grid, stream);
}

}  // namespace moe
