// routing.cu -- the local "dispatch" of the routed-experts layer on one GPU: expert histogram,
// exclusive scan to expert offsets, stable permutation of the (token, k) pairs into
// expert-contiguous rows, and the gather of token rows into that order.
//
// Dist-MoE 0.1.0, "Understand the execution model": rows are routed on the GPU before W13. The
// MoonEP FAQ on zero-copy: tokens are written straight to their expert-grouped positions, so the
// gate/up GEMM reads them with plain tiled loads and no further copy.
//
// Every result here is an integer with a unique answer (the order inside an expert segment is
// ascending pair index t*K+k), so the kernels are deterministic and bit-exact: counts come from
// shared-memory integer histograms, and ranks from warp match masks plus per-warp prefix counts,
// never from the order in which atomics land.
#include <cuda_runtime.h>

#include <atomic>

#include "moe_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe {
namespace {

__device__ __forceinline__ int route_key(int32_t id, int32_t E) { return (id >= 0 && id < E) ? id : E; }

// a1: per-block counts of the E+1 keys (key E collects ids outside [0, E)).
// block_counts is key-major: block_counts[key * nblk + block].
__global__ void __launch_bounds__(256) k_route_hist(const int32_t* __restrict__ ids, int64_t R, int32_t E, int nblk,
                                                    int32_t* __restrict__ block_counts, uint32_t* status) {
    extern __shared__ int32_t hist[];  // [E+1]
    for (int i = threadIdx.x; i <= E; i += blockDim.x) hist[i] = 0;
    griddep_wait();
    griddep_launch_dependents();
    __syncthreads();
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
    const int64_t c1 = min(c0 + kRouteChunk, R);
    int bad = 0;
    for (int64_t i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
        const int key = route_key(__ldg(ids + i), E);
        bad |= (key == E);
        atomicAdd(&hist[key], 1);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, static_cast<uint32_t>(MOE_DEV_BAD_EXPERT_ID));
    for (int k = threadIdx.x; k <= E; k += blockDim.x)
        block_counts[static_cast<int64_t>(k) * nblk + blockIdx.x] = hist[k];
}

// Exclusive prefix sum of one value per thread across the block (blockDim.x a multiple of 32).
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_sums, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < nwarps) warp_sums[lane] = w;  // inclusive over warps
        if (lane == 31 && total) *total = w;
    }
    __syncthreads();
    const int32_t before = warp == 0 ? 0 : warp_sums[warp - 1];
    const int32_t out = before + inc - v;
    __syncthreads();  // warp_sums may be reused by the caller
    return out;
}

// a2: one block. Exclusive scan of block_counts in (key, block) order gives every block the first
// row of its pairs of each key; from it come counts, offsets and the GEMM tile prefix lists
// tiles[e] = ntiles_n * sum_{e' < e} ceil(counts[e'] / kBM).
__global__ void __launch_bounds__(1024) k_route_scan(const int32_t* __restrict__ block_counts,
                                                     int32_t* __restrict__ block_bases, int nblk, int32_t E,
                                                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ tiles1, int32_t ntn1,
                                                     int32_t* __restrict__ tiles2, int32_t ntn2) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t total_mtiles;
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t N = static_cast<int64_t>(E + 1) * nblk;
    const int64_t b0 = N * tid / nt, b1 = N * (tid + 1) / nt;
    int32_t s = 0;
    for (int64_t i = b0; i < b1; ++i) s += block_counts[i];
    int32_t run = block_exclusive_scan(s, warp_sums, nullptr);
    for (int64_t i = b0; i < b1; ++i) {
        const int32_t c = block_counts[i];
        block_bases[i] = run;
        run += c;
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) {
        const int32_t o = block_bases[static_cast<int64_t>(e) * nblk];
        offsets[e] = o;
        counts[e] = block_bases[static_cast<int64_t>(e + 1) * nblk] - o;
    }
    if (tid == 0) offsets[E] = block_bases[static_cast<int64_t>(E) * nblk];
    if (tiles1 == nullptr) return;
    __syncthreads();
    const int e0 = static_cast<int>(static_cast<int64_t>(E) * tid / nt);
    const int e1 = static_cast<int>(static_cast<int64_t>(E) * (tid + 1) / nt);
    int32_t m = 0;
    for (int e = e0; e < e1; ++e) m += (counts[e] + kBM - 1) / kBM;
    int32_t mrun = block_exclusive_scan(m, warp_sums, &total_mtiles);
    for (int e = e0; e < e1; ++e) {
        tiles1[e] = mrun * ntn1;
        tiles2[e] = mrun * ntn2;
        mrun += (counts[e] + kBM - 1) / kBM;
    }
    __syncthreads();
    if (tid == 0) {
        tiles1[E] = total_mtiles * ntn1;
        tiles2[E] = total_mtiles * ntn2;
    }
}

// a3: stable permutation. Warp w of block b owns pairs [b*chunk + w*256, +256). Phase 1 counts each
// key in the warp's slice; phase 2 turns the counts into each warp's first row per key (starting
// from the block's base row from the scan); phase 3 walks the slice again in 32-pair rounds and
// ranks each pair among the earlier pairs with the same key (match mask + population count).
__global__ void __launch_bounds__(kRouteWarps * 32) k_route_permute(const int32_t* __restrict__ ids, int64_t R,
                                                                    int32_t E, int nblk,
                                                                    const int32_t* __restrict__ block_bases,
                                                                    int32_t* __restrict__ perm,
                                                                    int32_t* __restrict__ inv) {
    extern __shared__ int32_t cnt[];  // [kRouteWarps][E+1]
    constexpr int kRounds = kRoutePairsPerWarp / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stride = E + 1;
    for (int i = threadIdx.x; i < kRouteWarps * stride; i += blockDim.x) cnt[i] = 0;
    griddep_wait();
    griddep_launch_dependents();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk + static_cast<int64_t>(warp) * kRoutePairsPerWarp;
    // the warp's 256 keys, loaded once (all loads in flight together) and kept for both passes
    int key[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int64_t i = base + r * 32 + lane;
        key[r] = (i < R) ? route_key(__ldg(ids + i), E) : -1;
    }
    __syncthreads();
    int32_t* mine = cnt + warp * stride;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const unsigned peers = __match_any_sync(0xffffffffu, key[r]);
        if (key[r] >= 0 && lane == __ffs(peers) - 1) mine[key[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int k = threadIdx.x; k <= E; k += blockDim.x) {
        int32_t run = block_bases[static_cast<int64_t>(k) * nblk + blockIdx.x];
        for (int w = 0; w < kRouteWarps; ++w) {
            const int32_t c = cnt[w * stride + k];
            cnt[w * stride + k] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lower = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const int64_t i = base + r * 32 + lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key[r]);
        if (key[r] >= 0) {
            const int32_t row = mine[key[r]] + __popc(peers & lower);
            perm[row] = static_cast<int32_t>(i);
            inv[i] = row;
        }
        __syncwarp();
        if (key[r] >= 0 && lane == __ffs(peers) - 1) mine[key[r]] += __popc(peers);
        __syncwarp();
    }
}

// Gather: XP[inv[t*K+k], :] = x[t, :] for every pair whose row is valid (< offsets[E]). A work item
// is one 1024-column chunk of one token (one warp, 16-byte vectors, four per lane): it reads the
// chunk of x[t] once and writes it to each of the token's K rows, so x is read once instead of
// once per pair (K times the bytes when x does not fit in L2), and a small batch still has
// tokens x chunks items to spread over the GPU.
constexpr int kGatherChunkVec = 128;  // 16-byte vectors per chunk (1024 bf16)

__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ x, const int32_t* __restrict__ inv,
                                                     const int32_t* __restrict__ offsets, int32_t E, int32_t K,
                                                     int64_t T, int vec_per_row, uint4* __restrict__ xp) {
    griddep_wait();
    griddep_launch_dependents();
    const int32_t nvalid = __ldg(offsets + E);
    const int lane = threadIdx.x & 31;
    const int chunks = (vec_per_row + kGatherChunkVec - 1) / kGatherChunkVec;
    const int64_t items = T * chunks;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
         item += warps_total) {
        const int64_t t = item / chunks;
        const int j = static_cast<int>(item - t * chunks) * kGatherChunkVec + lane;
        const uint4* src = x + t * vec_per_row;
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (j + u * 32 < vec_per_row) v[u] = __ldg(src + j + u * 32);
        const int32_t* rows = inv + t * K;
        for (int k = 0; k < K; ++k) {
            const int32_t row = __ldg(rows + k);
            if (row >= nvalid) continue;  // a pair with an invalid id (warp-uniform)
            uint4* dst = xp + static_cast<int64_t>(row) * vec_per_row;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j + u * 32 < vec_per_row) dst[j + u * 32] = v[u];
        }
    }
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_permute_attr[kMaxDevices];

}  // namespace

moe_status_t launch_routing(const RoutingBuffers& b, cudaStream_t stream) {
    const size_t hist_smem = sizeof(int32_t) * (b.E + 1);
    const size_t perm_smem = sizeof(int32_t) * kRouteWarps * (b.E + 1);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    if (!g_permute_attr[dev].load(std::memory_order_acquire)) {
        // the permute kernel needs more than the default 48 KB of shared memory for large E
        if (cudaFuncSetAttribute(k_route_permute, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(int32_t) * kRouteWarps * (kMaxExperts + 1))) != cudaSuccess)
            return MOE_ERR_CUDA;
        g_permute_attr[dev].store(true, std::memory_order_release);
    }
    if (launch_pdl(k_route_hist, dim3(b.nblk), dim3(256), hist_smem, stream, b.ids, b.R, b.E, b.nblk, b.block_counts,
                   b.status) != cudaSuccess ||
        launch_pdl(k_route_scan, dim3(1), dim3(1024), 0, stream, b.block_counts, b.block_bases, b.nblk, b.E, b.counts,
                   b.offsets, b.tiles1, b.ntiles_n1, b.tiles2, b.ntiles_n2) != cudaSuccess ||
        launch_pdl(k_route_permute, dim3(b.nblk), dim3(kRouteWarps * 32), perm_smem, stream, b.ids, b.R, b.E, b.nblk,
                   b.block_bases, b.perm, b.inv) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status_t launch_gather(const void* x, const int32_t* inv, const int32_t* offsets, int32_t E, int32_t K,
                           int64_t R, int32_t D, void* xp, int sm_count, cudaStream_t stream) {
    const int vec_per_row = D / 8;
    const int64_t T = R / K;
    const int64_t want = ceil_div(T * ceil_div(vec_per_row, kGatherChunkVec), 8);  // one warp per item, 8 per block
    const int grid = static_cast<int>(want < static_cast<int64_t>(sm_count) * 8 ? want : static_cast<int64_t>(sm_count) * 8);
    return launch_pdl(k_gather_rows, dim3(grid > 0 ? grid : 1), dim3(256), 0, stream, static_cast<const uint4*>(x), inv,
                      offsets, E, K, T, vec_per_row, static_cast<uint4*>(xp)) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

}  // namespace moe
