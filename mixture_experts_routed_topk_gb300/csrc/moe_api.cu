// moe_api.cu -- the C ABI (include/moe_routed_experts.h): argument checks, the workspace layout
// and the launch sequence of the routed-experts forward pass.
//
// Every check that needs no GPU runs first, so a bad call returns before touching CUDA. After
// that, the entry points only enqueue work on the caller's stream: no allocation, no host
// synchronisation, no device-to-host copy (moe_get_status is the one synchronising call).
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape limits shared by every entry point (D/F ignored when with_activations is false).
moe_status_t check_shape(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, bool with_activations) {
    if (T < 0 || E <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
    if (with_activations && (D <= 0 || F <= 0)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t R = T * static_cast<int64_t>(K);
    if (T > 0 && R / K != T) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (R >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (with_activations) {
        if (D % 64 != 0 || F % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
        // TMA row coordinates and tile indices are 32-bit
        if (static_cast<int64_t>(E) * 2 * F >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (static_cast<int64_t>(E) * D >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
        const int64_t ntn = ceil_div(F, kBN1) > ceil_div(D, kBN2) ? ceil_div(F, kBN1) : ceil_div(D, kBN2);
        if ((ceil_div(R, kBM) + E) * ntn >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    }
    return MOE_OK;
}

}  // namespace

bool make_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, bool with_activations, Layout* L,
                 bool fused) {
    if (check_shape(T, D, F, E, K, with_activations) != MOE_OK) return false;
    const int64_t R = T * static_cast<int64_t>(K);
    L->nblk = static_cast<int>(ceil_div(R, kRouteChunk));
    if (L->nblk < 1) L->nblk = 1;
    const size_t e1 = static_cast<size_t>(E) + 1;
    size_t sizes[MOE_WS_TOTAL] = {};
    sizes[MOE_WS_STATUS] = sizeof(uint32_t);
    sizes[MOE_WS_TILES1] = sizeof(int32_t) * e1;
    sizes[MOE_WS_TILES2] = sizeof(int32_t) * e1;
    sizes[MOE_WS_BLOCK_COUNTS] = sizeof(int32_t) * e1 * L->nblk;
    sizes[MOE_WS_BLOCK_BASES] = sizeof(int32_t) * e1 * L->nblk;
    if (with_activations) {
        sizes[MOE_WS_COUNTS] = sizeof(int32_t) * E;
        sizes[MOE_WS_OFFSETS] = sizeof(int32_t) * e1;
        sizes[MOE_WS_PERM] = sizeof(int32_t) * R;
        sizes[MOE_WS_INV] = sizeof(int32_t) * R;
        sizes[MOE_WS_XP] = 2 * static_cast<size_t>(R) * D;
        sizes[MOE_WS_H] = 2 * static_cast<size_t>(R) * F;
        sizes[MOE_WS_RMS] = sizeof(float) * static_cast<size_t>(R) * ceil_div(D, kBN2);
        if (fused) {
            const int64_t nonempty = R < E ? R : E;
            sizes[MOE_WS_READY] = sizeof(uint32_t) * static_cast<size_t>(32 + ceil_div(R, kBM) + nonempty);
            sizes[MOE_WS_Y] = 2 * static_cast<size_t>(R) * D;
        }
    }
    size_t off = 0;
    for (int r = 0; r < MOE_WS_TOTAL; ++r) {
        L->off[r] = off;
        off += align_up(sizes[r]);
    }
    L->off[MOE_WS_TOTAL] = off;
    return true;
}

moe_status_t device_info(DeviceInfo* info) {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cached_sm[kMaxDevices];      // 0 = not queried yet
    static std::atomic<int> cached_ok[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    int sm = cached_sm[dev].load(std::memory_order_acquire);
    if (sm == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sm <= 0)
            return MOE_ERR_CUDA;
        cached_ok[dev].store(major == 10 && minor == 3 ? 1 : 0, std::memory_order_relaxed);
        cached_sm[dev].store(sm, std::memory_order_release);
    }
    info->sm_count = sm;
    info->supported = cached_ok[dev].load(std::memory_order_relaxed) != 0;
    return MOE_OK;
}

namespace {

struct Call {
    Layout L;
    DeviceInfo dev;
    uint8_t* ws;
    int64_t R;
};

// The common checks of the forward-pass stages. Host-only checks first; the device query last.
moe_status_t prepare(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, void* workspace, size_t workspace_bytes,
                     Call* c, bool fused = false) {
    moe_status_t st = check_shape(T, D, F, E, K, true);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
    if (!make_layout(T, D, F, E, K, true, &c->L, fused)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (workspace_bytes < c->L.off[MOE_WS_TOTAL]) return MOE_ERR_WORKSPACE_TOO_SMALL;
    c->ws = static_cast<uint8_t*>(workspace);
    c->R = T * static_cast<int64_t>(K);
    return MOE_OK;
}

moe_status_t check_device(Call* c) {
    moe_status_t st = device_info(&c->dev);
    if (st != MOE_OK) return st;
    return c->dev.supported ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

template <typename P>
P* region(const Call& c, int r) {
    return reinterpret_cast<P*>(c.ws + c.L.off[r]);
}

GemmProblem gemm_problem(const Call& c, int32_t D, int32_t F, int32_t E, int which) {
    GemmProblem p{};
    p.R = c.R;
    p.D = D;
    p.F = F;
    p.E = E;
    p.counts = region<int32_t>(c, MOE_WS_COUNTS);
    p.offsets = region<int32_t>(c, MOE_WS_OFFSETS);
    p.tiles = region<int32_t>(c, which == 1 ? MOE_WS_TILES1 : MOE_WS_TILES2);
    p.status = region<uint32_t>(c, MOE_WS_STATUS);
    p.sm_count = c.dev.sm_count;
    return p;
}

moe_status_t do_dispatch(const Call& c, const void* x, const int32_t* ids, int32_t D, int32_t F, int32_t E, int32_t K,
                         cudaStream_t stream) {
    if (cudaMemsetAsync(region<uint32_t>(c, MOE_WS_STATUS), 0, sizeof(uint32_t), stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    RoutingBuffers b{};
    b.ids = ids;
    b.R = c.R;
    b.E = E;
    b.nblk = c.L.nblk;
    b.block_counts = region<int32_t>(c, MOE_WS_BLOCK_COUNTS);
    b.block_bases = region<int32_t>(c, MOE_WS_BLOCK_BASES);
    b.counts = region<int32_t>(c, MOE_WS_COUNTS);
    b.offsets = region<int32_t>(c, MOE_WS_OFFSETS);
    b.perm = region<int32_t>(c, MOE_WS_PERM);
    b.inv = region<int32_t>(c, MOE_WS_INV);
    b.tiles1 = region<int32_t>(c, MOE_WS_TILES1);
    b.tiles2 = region<int32_t>(c, MOE_WS_TILES2);
    b.ntiles_n1 = static_cast<int32_t>(ceil_div(F, kBN1));
    b.ntiles_n2 = static_cast<int32_t>(ceil_div(D, kBN2));
    b.status = region<uint32_t>(c, MOE_WS_STATUS);
    moe_status_t st = launch_routing(b, stream);
    if (st != MOE_OK) return st;
    return launch_gather(x, b.inv, b.offsets, E, K, c.R, D, region<void>(c, MOE_WS_XP), c.dev.sm_count, stream);
}

moe_status_t do_gemm1(const Call& c, const void* w13, int32_t D, int32_t F, int32_t E, cudaStream_t stream) {
    return launch_gemm1_swiglu(gemm_problem(c, D, F, E, 1), region<void>(c, MOE_WS_XP), w13, region<void>(c, MOE_WS_H),
                               stream);
}

moe_status_t do_gemm2(const Call& c, const void* scores, int32_t scores_dtype, const void* w2, int32_t D, int32_t F,
                      int32_t E, cudaStream_t stream) {
    return launch_gemm2_score(gemm_problem(c, D, F, E, 2), region<void>(c, MOE_WS_H), w2,
                              region<int32_t>(c, MOE_WS_PERM), scores, scores_dtype, region<void>(c, MOE_WS_XP),
                              nullptr, stream);
}

moe_status_t do_combine(const Call& c, const int32_t* ids, void* out, int64_t T, int32_t D, int32_t E, int32_t K,
                        cudaStream_t stream) {
    return launch_combine(region<void>(c, MOE_WS_XP), ids, T, D, E, K, out, c.dev.sm_count, stream);
}

bool bad_scores_dtype(int32_t d) { return d != MOE_SCORES_F32 && d != MOE_SCORES_BF16; }

// Backward workspace: routing arrays, the padded-row maps and the padded activation buffers.
enum {
    BW_STATUS,
    BW_COUNTS,
    BW_OFFSETS,
    BW_BLOCK_COUNTS,
    BW_BLOCK_BASES,
    BW_PERM,
    BW_INV,
    BW_PMT,
    BW_PPERM,
    BW_PINV,
    BW_XPP,
    BW_DOP,
    BW_GU,
    BW_HS,
    BW_DGU,
    BW_PARTIAL,
    BW_DXP,
    BW_TOTAL
};

struct BwdLayout {
    size_t off[BW_TOTAL + 1];
    int nblk;
    int64_t padded_rows;
};

bool make_bwd_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, BwdLayout* L) {
    if (check_shape(T, D, F, E, K, true) != MOE_OK || T == 0) return false;
    const int64_t R = T * static_cast<int64_t>(K);
    const int64_t nonempty = R < E ? R : E;
    L->padded_rows = ceil_div(R + 127 * nonempty, 128) * 128;
    if (L->padded_rows >= (int64_t{1} << 31)) return false;
    L->nblk = static_cast<int>(ceil_div(R, kRouteChunk));
    const size_t e1 = static_cast<size_t>(E) + 1, rp = static_cast<size_t>(L->padded_rows);
    size_t sizes[BW_TOTAL] = {};
    sizes[BW_STATUS] = sizeof(uint32_t);
    sizes[BW_COUNTS] = sizeof(int32_t) * E;
    sizes[BW_OFFSETS] = sizeof(int32_t) * e1;
    sizes[BW_BLOCK_COUNTS] = sizeof(int32_t) * e1 * L->nblk;
    sizes[BW_BLOCK_BASES] = sizeof(int32_t) * e1 * L->nblk;
    sizes[BW_PERM] = sizeof(int32_t) * R;
    sizes[BW_INV] = sizeof(int32_t) * R;
    sizes[BW_PMT] = sizeof(int32_t) * e1;
    sizes[BW_PPERM] = sizeof(int32_t) * rp;
    sizes[BW_PINV] = sizeof(int32_t) * R;
    sizes[BW_XPP] = 2 * rp * D;
    sizes[BW_DOP] = 2 * rp * D;
    sizes[BW_GU] = 2 * rp * 2 * F;
    sizes[BW_HS] = 2 * rp * F;
    sizes[BW_DGU] = 2 * rp * 2 * F;
    sizes[BW_PARTIAL] = sizeof(float) * rp * ceil_div(F, kBN2);
    sizes[BW_DXP] = 2 * rp * D;
    size_t off = 0;
    for (int r = 0; r < BW_TOTAL; ++r) {
        L->off[r] = off;
        off += align_up(sizes[r]);
    }
    L->off[BW_TOTAL] = off;
    return true;
}

// MXFP8: D and F multiples of 128 (whole 128-byte K steps and whole scale groups).
moe_status_t check_mx_shape(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K) {
    moe_status_t st = check_shape(T, D, F, E, K, true);
    if (st != MOE_OK) return st;
    if (D % kMxBK != 0 || F % kMxBK != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t R = T * static_cast<int64_t>(K);
    const int64_t nonempty = R < E ? R : E;
    const int64_t ntn = ceil_div(F, kMxGateUpF) > ceil_div(D, kMxDownN) ? ceil_div(F, kMxGateUpF)
                                                                         : ceil_div(D, kMxDownN);
    if ((ceil_div(R, kBM) + nonempty) * ntn >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((ceil_div(R, kBM) + nonempty) * kBM >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

struct MxLayout {
    size_t off[MOE_MXWS_REGIONS];
    int nblk;
    int64_t padded_rows;
};

// fp4 = true: the NVFP4 sizes (packed E2M1 codes, one UE4M3 scale per 16, K groups padded to whole
// 256-wide stages); false: MXFP8 (E4M3 codes, one UE8M0 scale per 32).
bool make_mx_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, MxLayout* L, bool fp4 = false) {
    if (check_mx_shape(T, D, F, E, K) != MOE_OK || T == 0) return false;
    const int64_t R = T * static_cast<int64_t>(K);
    const int64_t nonempty = R < E ? R : E;
    L->padded_rows = (ceil_div(R, kBM) + nonempty) * kBM;
    L->nblk = static_cast<int>(ceil_div(R, kRouteChunk));
    const size_t e1 = static_cast<size_t>(E) + 1, rp = static_cast<size_t>(L->padded_rows);
    size_t sizes[MOE_MXWS_TOTAL] = {};
    sizes[MOE_MXWS_STATUS] = sizeof(uint32_t);
    sizes[MOE_MXWS_COUNTS] = sizeof(int32_t) * E;
    sizes[MOE_MXWS_OFFSETS] = sizeof(int32_t) * e1;
    sizes[MOE_MXWS_TILES] = sizeof(int32_t) * e1;
    sizes[MOE_MXWS_TILES2] = sizeof(int32_t) * e1;
    sizes[MOE_MXWS_BLOCK_COUNTS] = sizeof(int32_t) * e1 * L->nblk;
    sizes[MOE_MXWS_BLOCK_BASES] = sizeof(int32_t) * e1 * L->nblk;
    sizes[MOE_MXWS_PERM] = sizeof(int32_t) * R;
    sizes[MOE_MXWS_INV] = sizeof(int32_t) * R;
    sizes[MOE_MXWS_XQ] = fp4 ? rp * D / 2 : rp * D;
    sizes[MOE_MXWS_XS] = fp4 ? nv_act_scale_bytes(L->padded_rows, D) : rp * (D / 32);
    sizes[MOE_MXWS_HQ] = fp4 ? rp * F / 2 : rp * F;
    sizes[MOE_MXWS_HS] = fp4 ? nv_act_scale_bytes(L->padded_rows, F) : rp * (F / 32);
    sizes[MOE_MXWS_Y] = 2 * static_cast<size_t>(R) * D;
    size_t off = 0;
    for (int r = 0; r < MOE_MXWS_TOTAL; ++r) {
        L->off[r] = off;
        off += align_up(sizes[r]);
    }
    L->off[MOE_MXWS_TOTAL] = off;
    return true;
}

bool mx_weight_bytes(int32_t which, int32_t D, int32_t F, int32_t E, size_t* data, size_t* scales) {
    if (which == MOE_WEIGHT_W13) {
        *data = static_cast<size_t>(E) * 2 * F * D;
        *scales = static_cast<size_t>(E) * ceil_div(F, kMxGateUpF) * (D / 128) * 1024;
    } else {
        *data = static_cast<size_t>(E) * D * F;
        *scales = static_cast<size_t>(E) * ceil_div(D, kMxDownN) * (F / 128) * 1024;
    }
    return true;
}


// The block-scaled forward stages (MXFP8, or NVFP4 with fp4 = true and its activation scales).
moe_status_t block_scaled_stages(bool fp4, const void* x, const int32_t* topk_ids, const void* topk_scores,
                                 int32_t scores_dtype, const void* w13_data, const void* w13_scales,
                                 const void* w2_data, const void* w2_scales, float x_scale, float h_scale, void* out,
                                 int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, int32_t stage_begin,
                                 int32_t stage_end, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    moe_status_t st = check_mx_shape(T, D, F, E, K);
    if (fp4 && !(x_scale > 0.0f && x_scale < 3.0e38f && h_scale > 0.0f && h_scale < 3.0e38f))
        return MOE_ERR_INVALID_ARG;
    if (st != MOE_OK) return st;
    if (bad_scores_dtype(scores_dtype)) return MOE_ERR_INVALID_ARG;
    if (stage_begin < 0 || stage_end > MOE_MX_STAGES || stage_begin > stage_end) return MOE_ERR_INVALID_ARG;
    if (T == 0 || stage_begin == stage_end) return MOE_OK;
    if (!x || !topk_ids || !topk_scores || !w13_data || !w13_scales || !w2_data || !w2_scales || !out || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(topk_ids, 4) || !aligned(topk_scores, 4) || !aligned(w13_data, 16) ||
        !aligned(w13_scales, 256) || !aligned(w2_data, 16) || !aligned(w2_scales, 256) || !aligned(out, 16) ||
        !aligned(workspace, kAlign))
        return MOE_ERR_MISALIGNED;
    MxLayout L;
    if (!make_mx_layout(T, D, F, E, K, &L, fp4)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (workspace_bytes < L.off[MOE_MXWS_TOTAL]) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    MxProblem p{};
    p.act_scale_x = x_scale;
    p.act_scale_h = h_scale;
    p.T = T;
    p.D = D;
    p.F = F;
    p.E = E;
    p.K = K;
    p.x = x;
    p.ids = topk_ids;
    p.scores = topk_scores;
    p.scores_dtype = scores_dtype;
    p.w13q = w13_data;
    p.w13s = w13_scales;
    p.w2q = w2_data;
    p.w2s = w2_scales;
    p.out = out;
    p.status = reinterpret_cast<uint32_t*>(ws + L.off[MOE_MXWS_STATUS]);
    p.counts = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_COUNTS]);
    p.offsets = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_OFFSETS]);
    p.tiles1 = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_TILES]);
    p.tiles2 = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_TILES2]);
    p.block_counts = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_BLOCK_COUNTS]);
    p.block_bases = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_BLOCK_BASES]);
    p.perm = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_PERM]);
    p.inv = reinterpret_cast<int32_t*>(ws + L.off[MOE_MXWS_INV]);
    p.xq = ws + L.off[MOE_MXWS_XQ];
    p.xs = ws + L.off[MOE_MXWS_XS];
    p.hq = ws + L.off[MOE_MXWS_HQ];
    p.hs = ws + L.off[MOE_MXWS_HS];
    p.y = ws + L.off[MOE_MXWS_Y];
    p.nblk = L.nblk;
    p.padded_rows = L.padded_rows;
    p.sm_count = dev.sm_count;
    return fp4 ? launch_nv_forward(p, stage_begin, stage_end, reinterpret_cast<cudaStream_t>(stream))
               : launch_mx_forward(p, stage_begin, stage_end, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K) {
    Layout L;
    if (T == 0 || !make_layout(T, D, F, E, K, true, &L)) return 0;
    return L.off[MOE_WS_TOTAL];
}

moe_status_t moe_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, size_t* region_offsets) {
    if (region_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, D, F, E, K, true);
    if (st != MOE_OK) return st;
    Layout L;
    if (!make_layout(T, D, F, E, K, true, &L)) return MOE_ERR_UNSUPPORTED_SHAPE;
    std::memcpy(region_offsets, L.off, sizeof(L.off));
    return MOE_OK;
}

size_t moe_mega_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K) {
    Layout L;
    if (T == 0 || !make_layout(T, D, F, E, K, true, &L, true)) return 0;
    return L.off[MOE_WS_TOTAL];
}

moe_status_t moe_mega_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                       size_t* region_offsets) {
    if (region_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, D, F, E, K, true);
    if (st != MOE_OK) return st;
    Layout L;
    if (!make_layout(T, D, F, E, K, true, &L, true)) return MOE_ERR_UNSUPPORTED_SHAPE;
    std::memcpy(region_offsets, L.off, sizeof(L.off));
    return MOE_OK;
}

size_t moe_routing_workspace_bytes(int64_t T, int32_t E, int32_t K) {
    Layout L;
    if (T == 0 || !make_layout(T, 0, 0, E, K, false, &L)) return 0;
    return L.off[MOE_WS_TOTAL];
}

moe_status_t moe_routing(const int32_t* topk_ids, int64_t T, int32_t E, int32_t K, int32_t* counts, int32_t* offsets,
                         int32_t* perm, int32_t* inv, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    moe_status_t st = check_shape(T, 0, 0, E, K, false);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (!topk_ids || !counts || !offsets || !perm || !inv || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4) || !aligned(inv, 4))
        return MOE_ERR_MISALIGNED;
    if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
    Layout L;
    if (!make_layout(T, 0, 0, E, K, false, &L)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (workspace_bytes < L.off[MOE_WS_TOTAL]) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    st = device_info(&dev);
    if (st != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws + L.off[MOE_WS_STATUS], 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    RoutingBuffers b{};
    b.ids = topk_ids;
    b.R = T * static_cast<int64_t>(K);
    b.E = E;
    b.nblk = L.nblk;
    b.block_counts = reinterpret_cast<int32_t*>(ws + L.off[MOE_WS_BLOCK_COUNTS]);
    b.block_bases = reinterpret_cast<int32_t*>(ws + L.off[MOE_WS_BLOCK_BASES]);
    b.counts = counts;
    b.offsets = offsets;
    b.perm = perm;
    b.inv = inv;
    b.status = reinterpret_cast<uint32_t*>(ws + L.off[MOE_WS_STATUS]);
    return launch_routing(b, s);
}

moe_status_t moe_fwd_dispatch(const void* x, const int32_t* topk_ids, int64_t T, int32_t D, int32_t F, int32_t E,
                              int32_t K, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Call c{};
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c);
    if (st != MOE_OK || T == 0) return st;
    if (!x || !topk_ids) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(topk_ids, 4)) return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    return do_dispatch(c, x, topk_ids, D, F, E, K, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_fwd_gemm1(const void* w13, int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream) {
    Call c{};
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c);
    if (st != MOE_OK || T == 0) return st;
    if (!w13) return MOE_ERR_INVALID_ARG;
    if (!aligned(w13, 16)) return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    return do_gemm1(c, w13, D, F, E, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_fwd_gemm2(const void* topk_scores, int32_t scores_dtype, const void* w2, int64_t T, int32_t D,
                           int32_t F, int32_t E, int32_t K, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream) {
    Call c{};
    if (bad_scores_dtype(scores_dtype)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c);
    if (st != MOE_OK || T == 0) return st;
    if (!topk_scores || !w2) return MOE_ERR_INVALID_ARG;
    if (!aligned(w2, 16) || !aligned(topk_scores, scores_dtype == MOE_SCORES_F32 ? 4 : 2)) return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    return do_gemm2(c, topk_scores, scores_dtype, w2, D, F, E, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_fwd_combine(const int32_t* topk_ids, void* out, int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Call c{};
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c);
    if (st != MOE_OK || T == 0) return st;
    if (!topk_ids || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(topk_ids, 4)) return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    return do_combine(c, topk_ids, out, T, D, E, K, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_routed_experts_fwd(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                    int32_t scores_dtype, const void* w13, const void* w2, void* out, int64_t T,
                                    int32_t D, int32_t F, int32_t E, int32_t K, void* workspace,
                                    size_t workspace_bytes, moe_stream_t stream) {
    Call c{};
    if (bad_scores_dtype(scores_dtype)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c);
    if (st != MOE_OK || T == 0) return st;
    if (!x || !topk_ids || !topk_scores || !w13 || !w2 || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_scores, scores_dtype == MOE_SCORES_F32 ? 4 : 2))
        return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = do_dispatch(c, x, topk_ids, D, F, E, K, s)) != MOE_OK) return st;
    if ((st = do_gemm1(c, w13, D, F, E, s)) != MOE_OK) return st;
    if ((st = do_gemm2(c, topk_scores, scores_dtype, w2, D, F, E, s)) != MOE_OK) return st;
    return do_combine(c, topk_ids, out, T, D, E, K, s);
}

size_t moe_bwd_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K) {
    BwdLayout L;
    if (!make_bwd_layout(T, D, F, E, K, &L)) return 0;
    return L.off[BW_TOTAL];
}

moe_status_t moe_bwd_stages(const void* x, const int32_t* topk_ids, const void* topk_scores, int32_t scores_dtype,
                            const void* w13, const void* w2, const void* dout, void* dx, float* dscores, void* dw13,
                            void* dw2, int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, int32_t stage_begin,
                            int32_t stage_end, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    if (bad_scores_dtype(scores_dtype)) return MOE_ERR_INVALID_ARG;
    if (stage_begin < 0 || stage_end > MOE_BWD_STAGES || stage_begin > stage_end) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, D, F, E, K, true);
    if (st != MOE_OK || stage_begin == stage_end) return st;
    if (!w13 || !w2 || !dw13 || !dw2) return MOE_ERR_INVALID_ARG;
    if (!aligned(w13, 16) || !aligned(w2, 16) || !aligned(dw13, 16) || !aligned(dw2, 16)) return MOE_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceInfo dev;
    if (T == 0) {
        // no tokens: the weight gradients are zero (written by the stages that write them)
        if ((st = device_info(&dev)) != MOE_OK) return st;
        const bool w2_stage = stage_begin <= MOE_BWD_STAGE_WGRAD_DOWN && MOE_BWD_STAGE_WGRAD_DOWN < stage_end;
        const bool w13_stage = stage_begin <= MOE_BWD_STAGE_WGRAD_GATE_UP && MOE_BWD_STAGE_WGRAD_GATE_UP < stage_end;
        if ((w13_stage && cudaMemsetAsync(dw13, 0, 2ull * E * 2 * F * D, s) != cudaSuccess) ||
            (w2_stage && cudaMemsetAsync(dw2, 0, 2ull * E * D * F, s) != cudaSuccess))
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!x || !topk_ids || !topk_scores || !dout || !dx || !dscores || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(dout, 16) || !aligned(dx, 16) || !aligned(topk_ids, 4) || !aligned(dscores, 4) ||
        !aligned(topk_scores, scores_dtype == MOE_SCORES_F32 ? 4 : 2))
        return MOE_ERR_MISALIGNED;
    if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
    BwdLayout L;
    if (!make_bwd_layout(T, D, F, E, K, &L)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (workspace_bytes < L.off[BW_TOTAL]) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto at = [&](int r) { return ws + L.off[r]; };
    BwdProblem p{};
    p.T = T;
    p.D = D;
    p.F = F;
    p.E = E;
    p.K = K;
    p.x = x;
    p.ids = topk_ids;
    p.scores = topk_scores;
    p.scores_dtype = scores_dtype;
    p.w13 = w13;
    p.w2 = w2;
    p.dout = dout;
    p.dx = dx;
    p.dscores = dscores;
    p.dw13 = dw13;
    p.dw2 = dw2;
    p.status = reinterpret_cast<uint32_t*>(at(BW_STATUS));
    p.counts = reinterpret_cast<int32_t*>(at(BW_COUNTS));
    p.offsets = reinterpret_cast<int32_t*>(at(BW_OFFSETS));
    p.block_counts = reinterpret_cast<int32_t*>(at(BW_BLOCK_COUNTS));
    p.block_bases = reinterpret_cast<int32_t*>(at(BW_BLOCK_BASES));
    p.perm = reinterpret_cast<int32_t*>(at(BW_PERM));
    p.inv = reinterpret_cast<int32_t*>(at(BW_INV));
    p.pmt = reinterpret_cast<int32_t*>(at(BW_PMT));
    p.pperm = reinterpret_cast<int32_t*>(at(BW_PPERM));
    p.pinv = reinterpret_cast<int32_t*>(at(BW_PINV));
    p.xpp = at(BW_XPP);
    p.dop = at(BW_DOP);
    p.gu = at(BW_GU);
    p.hs = at(BW_HS);
    p.dgu = at(BW_DGU);
    p.partial = reinterpret_cast<float*>(at(BW_PARTIAL));
    p.dxp = at(BW_DXP);
    p.nblk = L.nblk;
    p.padded_rows = L.padded_rows;
    p.sm_count = dev.sm_count;
    return launch_backward(p, stage_begin, stage_end, s);
}

moe_status_t moe_routed_experts_bwd(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                    int32_t scores_dtype, const void* w13, const void* w2, const void* dout, void* dx,
                                    float* dscores, void* dw13, void* dw2, int64_t T, int32_t D, int32_t F, int32_t E,
                                    int32_t K, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return moe_bwd_stages(x, topk_ids, topk_scores, scores_dtype, w13, w2, dout, dx, dscores, dw13, dw2, T, D, F, E, K,
                          0, MOE_BWD_STAGES, workspace, workspace_bytes, stream);
}

moe_status_t moe_fwd_mega_stages(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                 int32_t scores_dtype, const void* w13, const void* w2, void* out, int64_t T,
                                 int32_t D, int32_t F, int32_t E, int32_t K, int32_t stage_begin, int32_t stage_end,
                                 void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Call c{};
    if (bad_scores_dtype(scores_dtype)) return MOE_ERR_INVALID_ARG;
    if (stage_begin < 0 || stage_end > MOE_MEGA_STAGES || stage_begin > stage_end) return MOE_ERR_INVALID_ARG;
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c, true);
    if (st != MOE_OK || T == 0 || stage_begin == stage_end) return st;
    const bool dispatch = stage_begin <= MOE_MEGA_STAGE_DISPATCH && MOE_MEGA_STAGE_DISPATCH < stage_end;
    const bool gemms = stage_begin <= MOE_MEGA_STAGE_GEMMS && MOE_MEGA_STAGE_GEMMS < stage_end;
    const bool combine = stage_begin <= MOE_MEGA_STAGE_COMBINE && MOE_MEGA_STAGE_COMBINE < stage_end;
    if ((dispatch && !x) || !topk_ids || (gemms && (!topk_scores || !w13 || !w2)) || (combine && !out))
        return MOE_ERR_INVALID_ARG;
    if ((dispatch && !aligned(x, 16)) || !aligned(topk_ids, 4) ||
        (gemms && (!aligned(w13, 16) || !aligned(w2, 16) ||
                   !aligned(topk_scores, scores_dtype == MOE_SCORES_F32 ? 4 : 2))) ||
        (combine && !aligned(out, 16)))
        return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dispatch && (st = do_dispatch(c, x, topk_ids, D, F, E, K, s)) != MOE_OK) return st;
    if (gemms) {
        if (cudaMemsetAsync(region<uint32_t>(c, MOE_WS_READY), 0, c.L.off[MOE_WS_Y] - c.L.off[MOE_WS_READY], s) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        if ((st = launch_fused_gemms(gemm_problem(c, D, F, E, 1), region<int32_t>(c, MOE_WS_TILES2),
                                     region<void>(c, MOE_WS_XP), w13, region<void>(c, MOE_WS_H), w2,
                                     region<int32_t>(c, MOE_WS_PERM), topk_scores, scores_dtype,
                                     region<void>(c, MOE_WS_Y), region<uint32_t>(c, MOE_WS_READY), s)) != MOE_OK)
            return st;
    }
    if (combine) return launch_combine(region<void>(c, MOE_WS_Y), topk_ids, T, D, E, K, out, c.dev.sm_count, s);
    return MOE_OK;
}

moe_status_t moe_routed_experts_fwd_mega(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                         int32_t scores_dtype, const void* w13, const void* w2, void* out, int64_t T,
                                         int32_t D, int32_t F, int32_t E, int32_t K, void* workspace,
                                         size_t workspace_bytes, moe_stream_t stream) {
    return moe_fwd_mega_stages(x, topk_ids, topk_scores, scores_dtype, w13, w2, out, T, D, F, E, K, 0,
                               MOE_MEGA_STAGES, workspace, workspace_bytes, stream);
}

moe_status_t moe_routed_experts_fwd_rmsnorm(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                            int32_t scores_dtype, const void* w13, const void* w2, void* out,
                                            int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, float eps,
                                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Call c{};
    if (bad_scores_dtype(scores_dtype) || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = prepare(T, D, F, E, K, workspace, workspace_bytes, &c);
    if (st != MOE_OK || T == 0) return st;
    if (!x || !topk_ids || !topk_scores || !w13 || !w2 || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_scores, scores_dtype == MOE_SCORES_F32 ? 4 : 2))
        return MOE_ERR_MISALIGNED;
    if ((st = check_device(&c)) != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = do_dispatch(c, x, topk_ids, D, F, E, K, s)) != MOE_OK) return st;
    if ((st = do_gemm1(c, w13, D, F, E, s)) != MOE_OK) return st;
    float* sumsq = region<float>(c, MOE_WS_RMS);
    if ((st = launch_gemm2_score(gemm_problem(c, D, F, E, 2), region<void>(c, MOE_WS_H), w2,
                                 region<int32_t>(c, MOE_WS_PERM), topk_scores, scores_dtype, region<void>(c, MOE_WS_XP),
                                 sumsq, s)) != MOE_OK)
        return st;
    return launch_combine_rmsnorm(region<void>(c, MOE_WS_XP), topk_ids, topk_scores, scores_dtype, sumsq, T, D, E, K,
                                  eps, out, c.dev.sm_count, s);
}

moe_status_t moe_mxfp8_weight_bytes(int32_t which, int32_t D, int32_t F, int32_t E, size_t* data_bytes,
                                    size_t* scale_bytes) {
    if (!data_bytes || !scale_bytes) return MOE_ERR_INVALID_ARG;
    if (which != MOE_WEIGHT_W13 && which != MOE_WEIGHT_W2) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(1, D, F, E, 1);
    if (st != MOE_OK) return st;
    mx_weight_bytes(which, D, F, E, data_bytes, scale_bytes);
    return MOE_OK;
}

moe_status_t moe_mxfp8_prepare_weight(int32_t which, const void* w, int32_t D, int32_t F, int32_t E, void* data,
                                      size_t data_bytes, void* scales, size_t scale_bytes, moe_stream_t stream) {
    if (which != MOE_WEIGHT_W13 && which != MOE_WEIGHT_W2) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(1, D, F, E, 1);
    if (st != MOE_OK) return st;
    if (!w || !data || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(data, 16) || !aligned(scales, 256)) return MOE_ERR_MISALIGNED;
    size_t need_data = 0, need_scales = 0;
    mx_weight_bytes(which, D, F, E, &need_data, &need_scales);
    if (data_bytes < need_data || scale_bytes < need_scales) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    return launch_mx_prepare_weight(which, w, D, F, E, data, scales, need_scales, dev.sm_count,
                                    reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_mxfp8_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K) {
    MxLayout L;
    if (T == 0 || !make_mx_layout(T, D, F, E, K, &L)) return 0;
    return L.off[MOE_MXWS_TOTAL];
}

moe_status_t moe_mxfp8_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                        size_t* region_offsets) {
    if (region_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(T, D, F, E, K);
    if (st != MOE_OK) return st;
    MxLayout L;
    if (!make_mx_layout(T, D, F, E, K, &L)) return MOE_ERR_UNSUPPORTED_SHAPE;
    std::memcpy(region_offsets, L.off, sizeof(L.off));
    return MOE_OK;
}

moe_status_t moe_routed_experts_fwd_mxfp8(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                          int32_t scores_dtype, const void* w13_data, const void* w13_scales,
                                          const void* w2_data, const void* w2_scales, void* out, int64_t T,
                                          int32_t D, int32_t F, int32_t E, int32_t K, void* workspace,
                                          size_t workspace_bytes, moe_stream_t stream) {
    return moe_fwd_mxfp8_stages(x, topk_ids, topk_scores, scores_dtype, w13_data, w13_scales, w2_data, w2_scales, out,
                                T, D, F, E, K, 0, MOE_MX_STAGES, workspace, workspace_bytes, stream);
}


moe_status_t moe_fwd_mxfp8_stages(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                  int32_t scores_dtype, const void* w13_data, const void* w13_scales,
                                  const void* w2_data, const void* w2_scales, void* out, int64_t T, int32_t D,
                                  int32_t F, int32_t E, int32_t K, int32_t stage_begin, int32_t stage_end,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return block_scaled_stages(false, x, topk_ids, topk_scores, scores_dtype, w13_data, w13_scales, w2_data,
                               w2_scales, 0.0f, 0.0f, out, T, D, F, E, K, stage_begin, stage_end, workspace,
                               workspace_bytes, stream);
}

moe_status_t moe_nvfp4_weight_bytes(int32_t which, int32_t D, int32_t F, int32_t E, size_t* data_bytes,
                                    size_t* scale_bytes) {
    if (!data_bytes || !scale_bytes) return MOE_ERR_INVALID_ARG;
    if (which != MOE_WEIGHT_W13 && which != MOE_WEIGHT_W2) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(1, D, F, E, 1);
    if (st != MOE_OK) return st;
    *data_bytes = (which == MOE_WEIGHT_W13 ? static_cast<size_t>(E) * 2 * F * D : static_cast<size_t>(E) * D * F) / 2;
    *scale_bytes = nv_weight_scale_bytes(which, D, F, E);
    return MOE_OK;
}

moe_status_t moe_nvfp4_prepare_weight(int32_t which, const void* w, int32_t D, int32_t F, int32_t E, void* data,
                                      size_t data_bytes, void* scales, size_t scale_bytes, moe_stream_t stream) {
    size_t need_data = 0, need_scales = 0;
    moe_status_t st = moe_nvfp4_weight_bytes(which, D, F, E, &need_data, &need_scales);
    if (st != MOE_OK) return st;
    if (!w || !data || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(data, 16) || !aligned(scales, 256)) return MOE_ERR_MISALIGNED;
    if (data_bytes < need_data || scale_bytes < need_scales) return MOE_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != MOE_OK) return st;
    if (!dev.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
    return launch_nv_prepare_weight(which, w, D, F, E, data, scales, need_scales, dev.sm_count,
                                    reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_nvfp4_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K) {
    MxLayout L;
    if (T == 0 || !make_mx_layout(T, D, F, E, K, &L, true)) return 0;
    return L.off[MOE_MXWS_TOTAL];
}

moe_status_t moe_nvfp4_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                        size_t* region_offsets) {
    if (region_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(T, D, F, E, K);
    if (st != MOE_OK) return st;
    MxLayout L;
    if (!make_mx_layout(T, D, F, E, K, &L, true)) return MOE_ERR_UNSUPPORTED_SHAPE;
    std::memcpy(region_offsets, L.off, sizeof(L.off));
    return MOE_OK;
}

moe_status_t moe_routed_experts_fwd_nvfp4(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                          int32_t scores_dtype, const void* w13_data, const void* w13_scales,
                                          const void* w2_data, const void* w2_scales, float x_scale, float h_scale,
                                          void* out, int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return moe_fwd_nvfp4_stages(x, topk_ids, topk_scores, scores_dtype, w13_data, w13_scales, w2_data, w2_scales,
                                x_scale, h_scale, out, T, D, F, E, K, 0, MOE_MX_STAGES, workspace, workspace_bytes,
                                stream);
}

moe_status_t moe_fwd_nvfp4_stages(const void* x, const int32_t* topk_ids, const void* topk_scores,
                                  int32_t scores_dtype, const void* w13_data, const void* w13_scales,
                                  const void* w2_data, const void* w2_scales, float x_scale, float h_scale, void* out,
                                  int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, int32_t stage_begin,
                                  int32_t stage_end, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return block_scaled_stages(true, x, topk_ids, topk_scores, scores_dtype, w13_data, w13_scales, w2_data,
                               w2_scales, x_scale, h_scale, out, T, D, F, E, K, stage_begin, stage_end, workspace,
                               workspace_bytes, stream);
}

moe_status_t moe_get_status(const void* workspace, uint32_t* device_bits, moe_stream_t stream) {
    if (!workspace || !device_bits) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    if (cudaMemcpyAsync(&bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    *device_bits = bits;
    return MOE_OK;
}

const char* moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer, negative size or unknown enum value";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE: sizes outside the supported limits";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: a pointer breaks the alignment rule";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL: workspace below the required size";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime or driver call failed";
        case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE: the current device is not sm_103";
    }
    return "unknown moe_status_t";
}

}  // extern "C"
