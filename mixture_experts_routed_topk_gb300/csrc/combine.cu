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

__global__ void __launch_bounds__(256) k_combine(const uint4* __restrict__ y, const int32_t* __restrict__ ids,
                                                 int64_t T, int32_t E, int32_t K, int vec_per_row,
                                                 uint4* __restrict__ out) {
    const int64_t total = T * vec_per_row;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += step) {
        const int64_t t = v / vec_per_row;
        const int64_t j = v - t * vec_per_row;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < K; k0 += 8) {
            uint4 q[8];
            bool use[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int k = k0 + u;
                use[u] = false;
                if (k < K) {
                    const int32_t e = __ldg(ids + t * K + k);
                    use[u] = (e >= 0 && e < E);
                    if (use[u]) q[u] = __ldg(y + (t * K + k) * vec_per_row + j);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (use[u]) add_bf16x8(acc, q[u]);
        }
        out[v] = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]), pack2(acc[4], acc[5]),
                            pack2(acc[6], acc[7]));
    }
}

}  // namespace

moe_status_t launch_combine(const void* y, const int32_t* ids, int64_t T, int32_t D, int32_t E, int32_t K,
                            void* out, int sm_count, cudaStream_t stream) {
    const int vec_per_row = D / 8;
    const int64_t total = T * vec_per_row;
    const int64_t want = ceil_div(total, 256);
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    k_combine<<<grid > 0 ? grid : 1, 256, 0, stream>>>(static_cast<const uint4*>(y), ids, T, E, K, vec_per_row,
                                                       static_cast<uint4*>(out));
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
