// moe_internal.cuh -- constants, workspace layout and kernel launchers shared by the translation
// units of the GB300 routed-experts library. Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "moe_routed_experts.h"

namespace moe {

// Routing: each routing block owns a contiguous chunk of (token, k) pairs; each of its warps owns
// a contiguous 256-pair slice of that chunk, so ranks inside a block follow the pair order.
constexpr int kRouteWarps = 8;
constexpr int kRoutePairsPerWarp = 256;
constexpr int kRouteChunk = kRouteWarps * kRoutePairsPerWarp;  // pairs per routing block
constexpr int kMaxExperts = 4096;

// Grouped GEMM tiles. Both GEMMs use a 128-row x 256-column fp32 accumulator in TMEM and walk K
// in 64-element (128-byte) steps. The gate/up GEMM's 256 columns are 128 gate columns and the
// same 128 up columns of one f range, so SwiGLU is local to one accumulator tile.
constexpr int kBM = 128;
constexpr int kBN1 = 128;  // f values per gate/up tile
constexpr int kBN2 = 256;  // output columns per down tile
constexpr int kBK = 64;

// MXFP8 grouped GEMM tiles: 128 rows x 192 accumulator columns, K in 128-element (128-byte)
// steps. A gate/up tile holds 96 gate and the same 96 up columns of one f range.
constexpr int kMxBK = 128;
constexpr int kMxBN = 192;
constexpr int kMxGateUpF = kMxBN / 2;  // 96 f values per gate/up tile
constexpr int kMxDownN = kMxBN;        // 192 output columns per down tile

// Host: launches `kernel` with programmatic stream serialization, so its launch and prologue may
// overlap the tail of the previous kernel on the stream. Every kernel launched this way calls
// griddep_wait() before its first global memory access, so the stream order of memory effects is
// unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct Layout {
    size_t off[MOE_WS_REGIONS];
    int nblk;  // routing blocks
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Host: workspace layout for the forward pass (with_activations = true) or for moe_routing alone
// (counts/offsets/perm/inv/XP/H regions empty; those arrays are the caller's).
// fused: also the READY counters and the separate Y region of the fused forward.
bool make_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, bool with_activations, Layout* L,
                 bool fused = false);

// Host: per-device facts, queried once per device.
struct DeviceInfo {
    int sm_count;
    bool supported;  // compute capability 10.3
};
moe_status_t device_info(DeviceInfo* info);

// Kernel launchers (host). They enqueue on `stream` and return MOE_ERR_CUDA if a launch fails.
struct RoutingBuffers {
    const int32_t* ids;
    int64_t R;
    int32_t E;
    int nblk;
    int32_t* block_counts;
    int32_t* block_bases;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* inv;
    int32_t* tiles1;  // may be null (moe_routing)
    int32_t* tiles2;  // may be null
    int32_t ntiles_n1;
    int32_t ntiles_n2;
    uint32_t* status;
};
moe_status_t launch_routing(const RoutingBuffers& b, cudaStream_t stream);

// XP[inv[t*K+k]] = x[t] for the valid pairs (token order: each x row is read once).
moe_status_t launch_gather(const void* x, const int32_t* inv, const int32_t* offsets, int32_t E, int32_t K,
                           int64_t R, int32_t D, void* xp, int sm_count, cudaStream_t stream);

struct GemmProblem {
    int64_t R;
    int32_t D, F, E;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* tiles;
    uint32_t* status;
    int sm_count;
};
moe_status_t launch_gemm1_swiglu(const GemmProblem& p, const void* xp, const void* w13, void* h,
                                 cudaStream_t stream);
// rms_sumsq: null for the plain layer; otherwise the route-wise RMSNorm variant (unweighted Y
// plus per-tile sums of squares, [T*K, ceil(D/256)] fp32).
moe_status_t launch_gemm2_score(const GemmProblem& p, const void* h, const void* w2, const int32_t* perm,
                                const void* scores, int32_t scores_dtype, void* y, float* rms_sumsq,
                                cudaStream_t stream);

// The fused forward: both grouped GEMMs in one grid, the down tiles of a row tile
// starting once its gate/up tiles have written their H rows. ready: the grid's tile counter, then
// from word 32 on one uint32 per row tile (ceil(R/128) + min(R, E) of them), all zero on entry. y must not overlap xp (Y rows are written while
// later experts' XP rows are still being read).
moe_status_t launch_fused_gemms(const GemmProblem& p, const int32_t* tiles2, const void* xp, const void* w13, void* h,
                                const void* w2, const int32_t* perm, const void* scores, int32_t scores_dtype, void* y,
                                uint32_t* ready, cudaStream_t stream);

// Backward pass (backward.cu): every pointer is device memory; padded_rows is the capacity of the
// padded-row buffers (R + 127 * min(E, R), a multiple of 128).
struct BwdProblem {
    int64_t T;
    int32_t D, F, E, K;
    const void* x;
    const int32_t* ids;
    const void* scores;
    int32_t scores_dtype;
    const void* w13;
    const void* w2;
    const void* dout;
    void* dx;
    float* dscores;
    void* dw13;
    void* dw2;
    // workspace
    uint32_t* status;
    int32_t *counts, *offsets, *block_counts, *block_bases, *perm, *inv;
    int32_t *pmt, *pperm, *pinv;
    void *xpp, *dop, *gu, *hs, *dgu, *dxp;
    float* partial;
    int nblk;
    int64_t padded_rows;
    int sm_count;
};
// Stages [stage_begin, stage_end) of the backward (MOE_BWD_STAGE_*).
moe_status_t launch_backward(const BwdProblem& p, int stage_begin, int stage_end, cudaStream_t stream);

moe_status_t launch_combine(const void* y, const int32_t* ids, int64_t T, int32_t D, int32_t E, int32_t K,
                            void* out, int sm_count, cudaStream_t stream);

// MXFP8 forward (mxfp8.cu). Weights are prepared once (E4M3 codes in the weight's own row order,
// UE8M0 scales grouped per GEMM tile); every pointer below is device memory.
// which = 0: w13 [E, 2F, D]; which = 1: w2 [E, D, F]. scales is cleared, then filled.
moe_status_t launch_mx_prepare_weight(int which, const void* w, int32_t D, int32_t F, int32_t E, void* data,
                                      void* scales, size_t scale_bytes, int sm_count, cudaStream_t stream);

struct MxProblem {
    int64_t T;
    int32_t D, F, E, K;
    const void* x;
    const int32_t* ids;
    const void* scores;
    int32_t scores_dtype;
    const void *w13q, *w13s, *w2q, *w2s;
    void* out;
    // workspace
    uint32_t* status;
    int32_t *counts, *offsets, *tiles1, *tiles2, *block_counts, *block_bases, *perm, *inv;
    uint8_t *xq, *xs, *hq, *hs;
    void* y;
    int nblk;
    int64_t padded_rows;  // capacity of XQ / HQ: 128 * (ceil(R / 128) + min(E, R))
    int sm_count;
    float act_scale_x, act_scale_h;  // NVFP4 only: the activations' tensor scales
};
// Stages [stage_begin, stage_end) of: 0 status + routing + gather-quantize, 1 gate/up GEMM,
// 2 down GEMM, 3 combine.
moe_status_t launch_mx_forward(const MxProblem& p, int stage_begin, int stage_end, cudaStream_t stream);

// NVFP4 forward (nvfp4.cu): the same problem and stages, with packed E2M1 operands (cols / 2 bytes
// per row) and UE4M3 scales per 16; a prepared weight's scale buffer starts with a 256-byte header
// holding its fp32 tensor scale.
size_t nv_weight_scale_bytes(int which, int32_t D, int32_t F, int32_t E);
size_t nv_act_scale_bytes(int64_t padded_rows, int32_t cols);
moe_status_t launch_nv_prepare_weight(int which, const void* w, int32_t D, int32_t F, int32_t E, void* data,
                                      void* scales, size_t scale_bytes, int sm_count, cudaStream_t stream);
moe_status_t launch_nv_forward(const MxProblem& p, int stage_begin, int stage_end, cudaStream_t stream);

// The combine of the route-wise RMSNorm variant: out[t] = sum_k s * y / sqrt(mean(y^2) + eps).
moe_status_t launch_combine_rmsnorm(const void* y, const int32_t* ids, const void* scores, int32_t scores_dtype,
                                    float* sumsq, int64_t T, int32_t D, int32_t E, int32_t K, float eps, void* out,
                                    int sm_count, cudaStream_t stream);

}  // namespace moe
