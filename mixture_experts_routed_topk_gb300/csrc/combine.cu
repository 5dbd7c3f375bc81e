// combine.cu -- the deterministic combine of the routed-experts forward pass: each token's K
// score-weighted expert outputs are summed in fixed k order (TeraMoE README, combine worker: the
// final weighted accumulation; gather worker: reducing a token's several local expert results).
//
//   out[t, :] = bf16( sum_{k=0..K-1, ids[t,k] in [0,E)} float(Y[t, k, :]) )
//
// One thread owns 8 consecutive columns (one 16-byte vector) of one token, loads up to 8 of the
// token's pair rows before adding them (in k order), and stores one 16-byte vector. HBM-bound:
// reads T*K*D*2 bytes, writes T*D*2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_internal.cuh"
#include "ptx_sm103.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename Index>
__global__ void __launch_bounds__(256) k_combine(const uint4* __restrict__ y, const int32_t* __restrict__ ids,
                                                 Index T, int32_t E, int32_t K, int32_t vec_per_row,
                                                 uint4* __restrict__ out) {
    griddep_wait();
    griddep_launch_dependents();
    const Index total = T * vec_per_row;
    const Index step = static_cast<Index>(gridDim.x) * blockDim.x;
    for (Index v = static_cast<Index>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += step) {
        const Index t = v / vec_per_row;
        const Index j = v - t * vec_per_row;
        const Index pair0 = t * K;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < K; k0 += 8) {
            int32_t e[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) e[u] = (k0 + u < K) ? __ldg(ids + pair0 + k0 + u) : -1;
            uint4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (e[u] >= 0 && e[u] < E) q[u] = __ldg(y + (pair0 + k0 + u) * vec_per_row + j);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (e[u] >= 0 && e[u] < E) add_bf16x8(acc, q[u]);
        }
        out[v] = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]), pack2(acc[4], acc[5]),
                            pack2(acc[6], acc[7]));
    }
}

// rstd[p] = 1 / sqrt(sum of the pair's per-tile sums of squares / D + eps), written over the first
// entry of the pair's row of sumsq (each pair owns its row).
__global__ void __launch_bounds__(256) k_rms_rstd(float* __restrict__ sumsq, int64_t R, int32_t ntd, int32_t D,
                                                  float eps) {
    griddep_wait();
    griddep_launch_dependents();
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < R;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float ss = 0.0f;
        for (int j = 0; j < ntd; ++j) ss += sumsq[p * ntd + j];
        sumsq[p * ntd] = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);
    }
}

// out[t] = bf16( sum_k score * rstd * Y[t,k] ) in k order, skipping invalid ids.
__global__ void __launch_bounds__(256) k_combine_rmsnorm(const uint4* __restrict__ y, const int32_t* __restrict__ ids,
                                                         const void* __restrict__ scores, int32_t scores_bf16,
                                                         const float* __restrict__ rstd, int32_t ntd, int64_t T,
                                                         int32_t E, int32_t K, int32_t vec_per_row,
                                                         uint4* __restrict__ out) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t total = T * vec_per_row;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = v / vec_per_row;
        const int64_t j = v - t * vec_per_row;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < K; ++k) {
            const int64_t p = t * K + k;
            const int32_t e = __ldg(ids + p);
            if (e < 0 || e >= E) continue;
            const float s = scores_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(scores)[p])
                                        : __ldg(reinterpret_cast<const float*>(scores) + p);
            const float w = s * __ldg(rstd + p * ntd);
            const uint4 q = __ldg(y + p * vec_per_row + j);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += w * __uint_as_float(wd[i] << 16);
                acc[2 * i + 1] += w * __uint_as_float(wd[i] & 0xffff0000u);
            }
        }
        out[v] = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]), pack2(acc[4], acc[5]),
                            pack2(acc[6], acc[7]));
    }
}

}  // namespace

moe_status_t launch_combine_rmsnorm(const void* y, const int32_t* ids, const void* scores, int32_t scores_dtype,
                                    float* sumsq, int64_t T, int32_t D, int32_t E, int32_t K, float eps, void* out,
                                    int sm_count, cudaStream_t stream) {
    const int32_t ntd = static_cast<int32_t>(ceil_div(D, kBN2));
    const int64_t R = T * K;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int64_t g1 = ceil_div(R, 256) < cap ? ceil_div(R, 256) : cap;
    const int vec_per_row = D / 8;
    const int64_t g2 = ceil_div(T * vec_per_row, 256) < cap ? ceil_div(T * vec_per_row, 256) : cap;
    if (launch_pdl(k_rms_rstd, dim3(static_cast<unsigned>(g1 > 0 ? g1 : 1)), dim3(256), 0, stream, sumsq, R, ntd, D,
                   eps) != cudaSuccess ||
        launch_pdl(k_combine_rmsnorm, dim3(static_cast<unsigned>(g2 > 0 ? g2 : 1)), dim3(256), 0, stream,
                   static_cast<const uint4*>(y), ids, scores, scores_dtype == MOE_SCORES_BF16 ? 1 : 0,
                   static_cast<const float*>(sumsq), ntd, T, E, K, vec_per_row, static_cast<uint4*>(out)) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status_t launch_combine(const void* y, const int32_t* ids, int64_t T, int32_t D, int32_t E, int32_t K,
                            void* out, int sm_count, cudaStream_t stream) {
    const int vec_per_row = D / 8;
    const int64_t total = T * vec_per_row;
    const int64_t want = ceil_div(total, 256);
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    const dim3 g(grid > 0 ? grid : 1), b(256);
    const uint4* yv = static_cast<const uint4*>(y);
    uint4* ov = static_cast<uint4*>(out);
    cudaError_t err;
    // 32-bit indexing when every index (and the grid-stride loop's overshoot) fits
    if (T * K * static_cast<int64_t>(vec_per_row) + static_cast<int64_t>(grid) * 256 < (int64_t{1} << 31))
        err = launch_pdl(k_combine<int32_t>, g, b, 0, stream, yv, ids, static_cast<int32_t>(T), E, K, vec_per_row, ov);
    else
        err = launch_pdl(k_combine<int64_t>, g, b, 0, stream, yv, ids, T, E, K, vec_per_row, ov);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
