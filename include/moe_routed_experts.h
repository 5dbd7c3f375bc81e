/*
 * moe_routed_experts.h -- C ABI of the routed top-k mixture-of-experts expert layer (forward,
 * backward and block-scaled forwards) for NVIDIA GB300 (sm_103a).
 *
 * The layer (the expert path shared by the TeraMoE README, Dist-MoE 0.1.0 and the Primus MegaMoE
 * guide; the MoonEP page describes its weight layout):
 *
 *     out[t] = sum_{k<K} score[t,k] * W2[e] ( SiLU(Wg[e] x_t) * (Wu[e] x_t) ),   e = ids[t,k]
 *
 *  - Dist-MoE 0.1.0, "Understand the execution model": route on the GPU -> W13 -> SwiGLU -> W2 ->
 *    combine. On one GPU the cross-rank "publish rows" / "combine" become a local stable permute of
 *    the (token, k) pairs into expert-contiguous rows and a local weighted unpermute-and-sum.
 *  - Dist-MoE 0.1.0, "BF16 Quickstart": the tensors x_TD [T,D], topk_expert_ids_TK [T,K],
 *    topk_scores_TK [T,K], w13_E2FD [E,2,F,D] (also [E,2F,D] or [E*2F,D], the same memory),
 *    w2_EDF [E,D,F] (also [E*D,F]); contiguous bf16 inputs and weights, expert ids in [0, E),
 *    bf16 or fp32 scores. "Choose a precision and pipeline / BF16": bf16 operands, fp32
 *    accumulation.
 *  - Primus MegaMoE guide, weight-module diagram: w1 [g, 2I, H] is gate then up; w2 [g, H, I].
 *  - MoonEP page, FAQ on the weight layout: one contiguous tensor per projection, experts addressed
 *    by row offset -- the grouped GEMMs here address expert e at row e*2F of w13 and e*D of w2.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device (or managed) memory on the current device; the
 *    caller owns them and keeps them alive until the stream work that uses them has completed.
 *  - bf16 is IEEE bfloat16 (16-bit storage). All arrays are dense row-major (C order).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream). No entry
 *    point allocates memory, synchronises or copies device data to the host, except
 *    moe_get_status, which synchronises `stream`.
 *  - Host-side checks run before anything is enqueued; a non-MOE_OK return means nothing was
 *    enqueued. Device-side problems never trap: they set bits in a status word that
 *    moe_get_status reads.
 *  - One workspace serves one call in flight at a time (sequentially reusable, not reentrant, as
 *    the Dist-MoE context is).
 *  - Shape limits (MOE_ERR_UNSUPPORTED_SHAPE otherwise): D and F multiples of 64; 1 <= E <= 4096;
 *    K >= 1; T*K < 2^31; T >= 0 (T = 0 returns MOE_OK and enqueues nothing).
 *  - Alignment (MOE_ERR_MISALIGNED otherwise): every pointer 16-byte aligned; the workspace
 *    256-byte aligned.
 */
#ifndef MOE_ROUTED_EXPERTS_H
#define MOE_ROUTED_EXPERTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null pointer, negative size, unknown enum value */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* outside the shape limits above */
    MOE_ERR_MISALIGNED = 3,          /* a pointer breaks the alignment rule above */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes below the size the call needs */
    MOE_ERR_CUDA = 5,                /* a CUDA runtime or driver call failed */
    MOE_ERR_UNSUPPORTED_DEVICE = 6   /* the current device is not sm_103 */
} moe_status_t;

/* Bits of the device status word (read with moe_get_status). */
enum {
    MOE_DEV_BAD_EXPERT_ID = 1u, /* an id outside [0, E): that (token, k) pair contributes 0 */
    MOE_DEV_TIMEOUT = 2u        /* a kernel's bounded wait expired; its results are invalid */
};

/* Dtype of topk_scores. */
enum { MOE_SCORES_F32 = 0, MOE_SCORES_BF16 = 1 };

/* Regions of the forward workspace, for moe_workspace_layout. */
enum {
    MOE_WS_STATUS = 0,       /* uint32 device status word (always at byte offset 0)            */
    MOE_WS_COUNTS = 1,       /* int32 [E]    rows routed to each expert                       */
    MOE_WS_OFFSETS = 2,      /* int32 [E+1]  first row of each expert; [E] = valid pairs      */
    MOE_WS_TILES1 = 3,       /* int32 [E+1]  prefix of the gate/up GEMM's tiles per expert     */
    MOE_WS_TILES2 = 4,       /* int32 [E+1]  prefix of the down GEMM's tiles per expert        */
    MOE_WS_BLOCK_COUNTS = 5, /* int32 [(E+1)*B]  per-(expert, routing block) counts            */
    MOE_WS_BLOCK_BASES = 6,  /* int32 [(E+1)*B]  per-(expert, routing block) first rows        */
    MOE_WS_PERM = 7,         /* int32 [T*K]  row -> flat pair t*K+k                            */
    MOE_WS_INV = 8,          /* int32 [T*K]  flat pair -> row                                  */
    MOE_WS_XP = 9,           /* bf16 [T*K, D] rows of x in routed order; after the down GEMM
                                the same bytes hold Y [T, K, D], the score-weighted expert
                                outputs per pair                                              */
    MOE_WS_H = 10,           /* bf16 [T*K, F] SwiGLU output per routed row                     */
    MOE_WS_RMS = 11,         /* fp32 [T*K, ceil(D/256)] per-tile sums of squares (RMSNorm mode) */
    MOE_WS_READY = 12,       /* fused forward only: uint32 [32 + ceil(T*K/128) + min(T*K, E)], the
                                fused grid's tile counter and its row-tile readiness counters */
    MOE_WS_Y = 13,           /* fused forward only: bf16 [T, K, D] score-weighted pair outputs  */
    MOE_WS_TOTAL = 14,       /* total bytes (== moe_workspace_bytes, or moe_mega_workspace_bytes
                                in the fused layout)                                          */
    MOE_WS_REGIONS = 15
};

/*
 * Bytes of device workspace that moe_routed_experts_fwd and the moe_fwd_* stages need for these
 * sizes (0 for T = 0). Pure arithmetic; never touches the GPU. Returns 0 for sizes outside the
 * shape limits.
 */
size_t moe_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K);

/*
 * Byte offsets of the workspace regions (MOE_WS_* above) into region_offsets[MOE_WS_REGIONS]
 * (host memory, caller-owned). Each region starts on a 256-byte boundary. Pure arithmetic.
 */
moe_status_t moe_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                  size_t *region_offsets);

/*
 * Bytes of device workspace that moe_routed_experts_fwd_mega needs, and its region offsets: the
 * layout above with the READY and Y regions filled in (both are empty in the staged layout).
 * Pure arithmetic; 0 / MOE_ERR_* for sizes outside the shape limits.
 */
size_t moe_mega_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K);
moe_status_t moe_mega_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                       size_t *region_offsets);

/*
 * Bytes of device workspace that moe_routing needs (status word and per-block scratch).
 */
size_t moe_routing_workspace_bytes(int64_t T, int32_t E, int32_t K);

/*
 * Routing alone: expert histogram, exclusive scan and stable permutation of the R = T*K
 * (token, k) pairs (the local form of Dist-MoE's "route on GPU"; the MoonEP FAQ's "tokens are
 * written directly to their expert-grouped positions").
 *
 *   topk_ids  device int32 [T,K]
 *   counts    device int32 [E]    counts[e] = #{ pairs with id e }
 *   offsets   device int32 [E+1]  offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   perm      device int32 [T*K]  perm[r] = t*K+k of the pair in row r; rows are ordered by
 *                                 (expert, t*K+k) ascending; pairs with an id outside [0, E) fill
 *                                 rows offsets[E] .. T*K-1 in ascending t*K+k
 *   inv       device int32 [T*K]  inv[t*K+k] = its row
 *   workspace device, moe_routing_workspace_bytes(T, E, K) bytes
 * All four outputs are bit-exact (they are integers with a unique answer). An id outside [0, E)
 * sets MOE_DEV_BAD_EXPERT_ID.
 */
moe_status_t moe_routing(const int32_t *topk_ids, int64_t T, int32_t E, int32_t K, int32_t *counts,
                         int32_t *offsets, int32_t *perm, int32_t *inv, void *workspace,
                         size_t workspace_bytes, moe_stream_t stream);

/*
 * The whole forward pass (Dist-MoE 0.1.0, "Understand the execution model"; TeraMoE README,
 * compute and combine workers): routing, gate/up grouped GEMM with SwiGLU, down grouped GEMM with
 * the score weighting, and a deterministic combine. Equivalent to moe_fwd_dispatch,
 * moe_fwd_gemm1, moe_fwd_gemm2 and moe_fwd_combine in that order.
 *
 *   x            device bf16 [T,D]
 *   topk_ids     device int32 [T,K]
 *   topk_scores  device [T,K], fp32 (scores_dtype = MOE_SCORES_F32) or bf16 (MOE_SCORES_BF16)
 *   w13          device bf16 [E,2,F,D]; w13[e,0] is the gate (through SiLU), w13[e,1] the up
 *   w2           device bf16 [E,D,F]
 *   out          device bf16 [T,D]; may not alias any input or the workspace
 *   workspace    device, moe_workspace_bytes(T, D, F, E, K) bytes
 *
 * Numerics: bf16 operands, fp32 accumulation; the SwiGLU output H and the score-weighted pair
 * outputs Y are rounded to bf16 (nearest even) in the workspace; the combine adds each token's K
 * pair outputs in fp32 in k order and rounds once. The result is deterministic: repeated calls
 * on the same inputs give the same bits. A pair with score 0 contributes exactly 0.
 */
moe_status_t moe_routed_experts_fwd(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                    int32_t scores_dtype, const void *w13, const void *w2, void *out,
                                    int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                    void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * The forward pass with Dist-MoE's typed post-expert processing (Dist-MoE 0.1.0, "Use advanced
 * features / Post-expert processing": route-wise RMSNorm, router-score weighting and top-k
 * reduction fused):
 *     out[t] = sum_k score[t,k] * y / sqrt(mean_d(y^2) + eps),   y = W2[e] (SiLU(Wg[e] x_t) * Wu[e] x_t)
 * The norm has no gain vector (the page names only eps and the dtypes); it is taken in fp32 from
 * the fp32 accumulator, and the weighted sum is fp32 in k order, rounded once to bf16. Arguments
 * and workspace as for moe_routed_experts_fwd, plus eps >= 0 (MOE_ERR_INVALID_ARG otherwise).
 */
moe_status_t moe_routed_experts_fwd_rmsnorm(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                            int32_t scores_dtype, const void *w13, const void *w2, void *out,
                                            int64_t T, int32_t D, int32_t F, int32_t E, int32_t K, float eps,
                                            void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * The forward pass with the two grouped GEMMs fused into one pipeline (Dist-MoE 0.1.0,
 * "Block-scaled execution": the Mega pipeline runs both projections as one chunked pipeline, with
 * the staged pipeline's tensor and memory contracts). One grid walks the gate/up
 * tiles of expert e and the down tiles of an earlier expert in turn; a down tile starts once the
 * gate/up tiles of its 128 rows have written their H rows, so H is read back from L2 and the two
 * GEMMs share one launch and one tail. The tiles and roundings are those of
 * moe_routed_experts_fwd: the output is bit-identical to it.
 *
 * Arguments as for moe_routed_experts_fwd, except
 *   workspace    device, moe_mega_workspace_bytes(T, D, F, E, K) bytes (it adds the READY
 *                counters and a Y region that may not overlap XP, because Y rows are written
 *                while later experts' XP rows are still being read)
 * Errors as for moe_routed_experts_fwd. A row tile whose H never arrives ends the kernel through
 * its bounded wait with MOE_DEV_TIMEOUT. Calls on different workspaces may run at once on
 * different streams.
 */
moe_status_t moe_routed_experts_fwd_mega(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                         int32_t scores_dtype, const void *w13, const void *w2, void *out,
                                         int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                         void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* Stages of the fused forward, for moe_fwd_mega_stages. */
enum {
    MOE_MEGA_STAGE_DISPATCH = 0, /* status word cleared, routing, x rows gathered (XP)             */
    MOE_MEGA_STAGE_GEMMS = 1,    /* readiness counters cleared; both grouped GEMMs in one grid (H, Y) */
    MOE_MEGA_STAGE_COMBINE = 2,  /* out from Y                                                      */
    MOE_MEGA_STAGES = 3
};

/*
 * Stages stage_begin .. stage_end-1 of moe_routed_experts_fwd_mega (0 <= stage_begin <= stage_end
 * <= MOE_MEGA_STAGES; the full range is that call), each needing the previous stages' workspace
 * contents. Arguments as for moe_routed_experts_fwd_mega; an out-of-range stage pair returns
 * MOE_ERR_INVALID_ARG before any launch.
 */
moe_status_t moe_fwd_mega_stages(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                 int32_t scores_dtype, const void *w13, const void *w2, void *out, int64_t T,
                                 int32_t D, int32_t F, int32_t E, int32_t K, int32_t stage_begin,
                                 int32_t stage_end, void *workspace, size_t workspace_bytes,
                                 moe_stream_t stream);

/*
 * Stage 1 of the forward pass: clears the status word, routes the pairs into the workspace's
 * counts/offsets/perm/inv and tile lists, and copies x[t] into row inv[t*K+k] of the workspace's
 * XP region (the expert-contiguous input of the gate/up GEMM).
 */
moe_status_t moe_fwd_dispatch(const void *x, const int32_t *topk_ids, int64_t T, int32_t D, int32_t F,
                              int32_t E, int32_t K, void *workspace, size_t workspace_bytes,
                              moe_stream_t stream);

/*
 * Stage 2: for every expert e, H[rows of e, :] = SiLU(XP_e Wg[e]^T) * (XP_e Wu[e]^T) (TeraMoE
 * README, compute worker: gate/up projection and activation), into the workspace's H region.
 * Needs stage 1's workspace contents.
 */
moe_status_t moe_fwd_gemm1(const void *w13, int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                           void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Stage 3: for every routed row r of expert e with pair p = perm[r],
 * Y[p, :] = score[p] * (H[r, :] W2[e]^T) (the down projection with the pair's routing weight
 * applied before the sum over k), into the workspace's XP region, which now holds Y [T,K,D].
 * Needs stage 2's workspace contents.
 */
moe_status_t moe_fwd_gemm2(const void *topk_scores, int32_t scores_dtype, const void *w2, int64_t T,
                           int32_t D, int32_t F, int32_t E, int32_t K, void *workspace,
                           size_t workspace_bytes, moe_stream_t stream);

/*
 * Stage 4: out[t, :] = bf16( sum_{k<K} Y[t, k, :] ) summed in fp32 in ascending k, skipping pairs
 * whose id is outside [0, E) (TeraMoE README, combine and gather workers: the final weighted
 * accumulation of a token's expert results). Needs stage 3's workspace contents.
 */
moe_status_t moe_fwd_combine(const int32_t *topk_ids, void *out, int64_t T, int32_t D, int32_t F,
                             int32_t E, int32_t K, void *workspace, size_t workspace_bytes,
                             moe_stream_t stream);

/*
 * Bytes of device workspace that moe_routed_experts_bwd needs (0 for T = 0 or sizes outside the
 * shape limits). Pure arithmetic.
 */
size_t moe_bwd_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K);

/*
 * The backward pass of the layer (Dist-MoE 0.1.0, "Understand the execution model": DGRAD computes
 * input gradients and WGRAD weight gradients; the TeraMoE README's example calls
 * output.backward). For the upstream gradient dout of out, with e = ids[t,k], s = scores[t,k]:
 *   dscores[t,k] = < dout[t], W2[e] (SiLU(Wg[e] x_t) * (Wu[e] x_t)) >
 *   dx[t]        = sum_k Wg[e]^T dg + Wu[e]^T du,  dh = s W2[e]^T dout[t],
 *                  dg = dh * (Wu[e] x_t) * SiLU'(Wg[e] x_t),  du = dh * SiLU(Wg[e] x_t)
 *   dw2[e]       = sum over the pairs of e of (s dout[t]) h^T
 *   dw13[e]      = sum over the pairs of e of [dg; du] x_t^T
 * Inputs as for moe_routed_experts_fwd, plus
 *   dout     device bf16 [T,D]
 *   dx       device bf16 [T,D]         (written in full)
 *   dscores  device fp32 [T,K]         (written in full; 0 for ids outside [0, E))
 *   dw13     device bf16 [E,2,F,D]     (written in full; zero for experts with no pairs)
 *   dw2      device bf16 [E,D,F]       (written in full)
 *   workspace device, moe_bwd_workspace_bytes(T, D, F, E, K) bytes; its first 4 bytes are the
 *            device status word (moe_get_status)
 * The forward activations are recomputed (nothing from the forward call is needed). bf16
 * operands, fp32 accumulation, bf16 intermediates; deterministic. T = 0 writes zero weight
 * gradients.
 */
moe_status_t moe_routed_experts_bwd(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                    int32_t scores_dtype, const void *w13, const void *w2, const void *dout,
                                    void *dx, float *dscores, void *dw13, void *dw2, int64_t T, int32_t D,
                                    int32_t F, int32_t E, int32_t K, void *workspace, size_t workspace_bytes,
                                    moe_stream_t stream);

/* Stages of the backward pass, for moe_bwd_stages. */
enum {
    MOE_BWD_STAGE_DISPATCH = 0,      /* status cleared, routing, padded-row maps, x and dout rows gathered */
    MOE_BWD_STAGE_RECOMPUTE = 1,     /* gate/up GEMM again: GU = [g | u] and HS = s h per padded row      */
    MOE_BWD_STAGE_DGRAD_DOWN = 2,    /* dout rows x W2 with the SwiGLU backward: DGU = [dg | du], dscores  */
                                     /* partial sums                                                        */
    MOE_BWD_STAGE_DGRAD_GATE_UP = 3, /* DGU x w13: the pairs' dx rows                                      */
    MOE_BWD_STAGE_WGRAD_DOWN = 4,    /* dw2[e] = (s dout)^T h over the expert's rows                         */
    MOE_BWD_STAGE_WGRAD_GATE_UP = 5, /* dw13[e] = [dg; du]^T x over the expert's rows                        */
    MOE_BWD_STAGE_REDUCE = 6,        /* dscores and dx, each summed in a fixed order                        */
    MOE_BWD_STAGES = 7
};

/*
 * Stages stage_begin .. stage_end-1 (MOE_BWD_STAGE_*) of moe_routed_experts_bwd, on one workspace:
 * a stage reads what the earlier stages left in it, so a caller runs the stages in order (one call
 * per stage lets it time each with events on its stream). 0 <= stage_begin <= stage_end <=
 * MOE_BWD_STAGES; the full range is moe_routed_experts_bwd. Arguments and errors as for that call;
 * MOE_ERR_INVALID_ARG for a bad range. With T = 0 the weight-gradient stages write zeros and the
 * others do nothing.
 */
moe_status_t moe_bwd_stages(const void *x, const int32_t *topk_ids, const void *topk_scores,
                            int32_t scores_dtype, const void *w13, const void *w2, const void *dout,
                            void *dx, float *dscores, void *dw13, void *dw2, int64_t T, int32_t D,
                            int32_t F, int32_t E, int32_t K, int32_t stage_begin, int32_t stage_end,
                            void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* MXFP8 forward (Dist-MoE 0.1.0, "Choose a precision and pipeline / MXFP8": MXFP8 E4M3, the    */
/* activations quantized after routing, the weights prepared once and reused -- "Use advanced   */
/* features / Prepared block-scaled weights" -- and FP32 accumulation).                        */
/*                                                                                              */
/* The format, read as the OCP Microscaling (MX) v1.0 format: a block is 32 consecutive elements */
/* along a GEMM's contraction axis (D for x and w13, F for the SwiGLU output h and for w2); it  */
/* shares the scale 2^e, e = floor(log2 max|v|) - 8 clamped to [-127, 127] (an all-zero block:  */
/* -127), stored as the UE8M0 byte e + 127; each element is the E4M3 value nearest v * 2^-e     */
/* (ties to even, saturating at 448, sign kept). x is quantized per token row, h per (token, k)  */
/* pair from fp32; the score, the expert outputs Y and out are as in the bf16 forward.          */
/* Shape limits of the MXFP8 entry points: those above, with D and F multiples of 128.          */
/* ------------------------------------------------------------------------------------------ */

/* Which weight moe_mxfp8_prepare_weight prepares. */
enum { MOE_WEIGHT_W13 = 0, MOE_WEIGHT_W2 = 1 };

/*
 * Sizes of a prepared weight: *data_bytes of E4M3 codes and *scale_bytes of UE8M0 scales (host
 * memory, caller-owned). Pure arithmetic.
 *   MOE_WEIGHT_W13: data E*2F*D;  scales E * ceil(F/96) * (D/128) * 1024
 *   MOE_WEIGHT_W2:  data E*D*F;   scales E * ceil(D/192) * (F/128) * 1024
 */
moe_status_t moe_mxfp8_weight_bytes(int32_t which, int32_t D, int32_t F, int32_t E, size_t *data_bytes,
                                    size_t *scale_bytes);

/*
 * Prepares one expert weight for the MXFP8 forward (Dist-MoE's prepare_block_scaled_weight):
 *   w       device bf16: w13 [E,2,F,D] (MOE_WEIGHT_W13) or w2 [E,D,F] (MOE_WEIGHT_W2)
 *   data    device, data_bytes: E4M3 codes in w's own element order (w13 as [E*2F, D] rows, w2 as
 *           [E*D, F] rows), each row quantized in blocks of 32 along its contiguous axis
 *   scales  device, scale_bytes: the UE8M0 scales, grouped per GEMM tile so that one tile's
 *           scales for 128 K values are one contiguous 1024-byte group. The scale of row n of
 *           tile (e, j) and 32-block b along the row sits at byte
 *             ((e * NT + j) * (C / 128) + b / 4) * 1024 + 512 * (n / 128)
 *               + 16 * (n % 32) + 4 * ((n % 128) / 32) + b % 4
 *           with C the row length. w13: NT = ceil(F/96), tile j holds gate rows f = 96j + n
 *           (n < 96) then up rows f = 96j + n - 96; w2: NT = ceil(D/192), row d = 192j + n.
 *           Bytes that belong to no row are 0.
 * Deterministic: the same w gives the same bytes. Capacity: data_bytes and scale_bytes at least
 * moe_mxfp8_weight_bytes' (MOE_ERR_WORKSPACE_TOO_SMALL otherwise). scales (here and in
 * moe_routed_experts_fwd_mxfp8) must be 256-byte aligned.
 */
moe_status_t moe_mxfp8_prepare_weight(int32_t which, const void *w, int32_t D, int32_t F, int32_t E,
                                      void *data, size_t data_bytes, void *scales, size_t scale_bytes,
                                      moe_stream_t stream);

/* Regions of the MXFP8 forward workspace, for moe_mxfp8_workspace_layout. Rp (padded rows) =
 * 128 * (ceil(T*K/128) + min(E, T*K)): every expert's rows start on a 128-row boundary. */
enum {
    MOE_MXWS_STATUS = 0,       /* uint32 device status word (always at byte offset 0)           */
    MOE_MXWS_COUNTS = 1,       /* int32 [E]                                                      */
    MOE_MXWS_OFFSETS = 2,      /* int32 [E+1]                                                    */
    MOE_MXWS_TILES = 3,        /* int32 [E+1] prefix of 128-row tiles: expert e's padded rows
                                  start at 128 * tiles[e]                                        */
    MOE_MXWS_TILES2 = 4,       /* int32 [E+1] (the same values; scratch of the routing scan)     */
    MOE_MXWS_BLOCK_COUNTS = 5, /* int32 [(E+1)*B]                                                */
    MOE_MXWS_BLOCK_BASES = 6,  /* int32 [(E+1)*B]                                                */
    MOE_MXWS_PERM = 7,         /* int32 [T*K] routed row -> pair, as in the bf16 forward          */
    MOE_MXWS_INV = 8,          /* int32 [T*K] pair -> routed row                                  */
    MOE_MXWS_XQ = 9,           /* E4M3 [Rp, D] x rows: routed row offsets[e] + i of expert e at
                                  padded row 128 * tiles[e] + i; zeros after each expert's rows  */
    MOE_MXWS_XS = 10,          /* UE8M0 scales of XQ: padded row p, 32-block b at byte
                                  ((p/128) * (D/128) + b/4) * 512 + 16 (p%32) + 4 ((p%128)/32) + b%4 */
    MOE_MXWS_HQ = 11,          /* E4M3 [Rp, F] the SwiGLU output, same rows as XQ                */
    MOE_MXWS_HS = 12,          /* UE8M0 scales of HQ, laid out as XS with F for D                */
    MOE_MXWS_Y = 13,           /* bf16 [T*K, D] score-weighted expert output per pair            */
    MOE_MXWS_TOTAL = 14,       /* total bytes (== moe_mxfp8_workspace_bytes)                     */
    MOE_MXWS_REGIONS = 15
};

/* Bytes of device workspace that moe_routed_experts_fwd_mxfp8 needs (0 for T = 0 or sizes outside
 * the MXFP8 shape limits). Pure arithmetic. */
size_t moe_mxfp8_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K);

/* Byte offsets of the MXFP8 workspace regions into region_offsets[MOE_MXWS_REGIONS] (host,
 * caller-owned); each region starts on a 256-byte boundary. Pure arithmetic. */
moe_status_t moe_mxfp8_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                        size_t *region_offsets);

/*
 * The MXFP8 forward: out as for moe_routed_experts_fwd, computed from MX-quantized x, w13, h and
 * w2 with fp32 accumulation (block-scaled tcgen05 tensor-core GEMMs).
 *   x, topk_ids, topk_scores, scores_dtype, out   as for moe_routed_experts_fwd
 *   w13_data, w13_scales   device, as written by moe_mxfp8_prepare_weight(MOE_WEIGHT_W13)
 *   w2_data, w2_scales     device, as written by moe_mxfp8_prepare_weight(MOE_WEIGHT_W2)
 *   workspace  device, moe_mxfp8_workspace_bytes(T, D, F, E, K) bytes, 256-byte aligned; its
 *              first 4 bytes are the device status word (moe_get_status)
 * Deterministic. An id outside [0, E) sets MOE_DEV_BAD_EXPERT_ID and its pair contributes 0.
 */
moe_status_t moe_routed_experts_fwd_mxfp8(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                          int32_t scores_dtype, const void *w13_data, const void *w13_scales,
                                          const void *w2_data, const void *w2_scales, void *out, int64_t T,
                                          int32_t D, int32_t F, int32_t E, int32_t K, void *workspace,
                                          size_t workspace_bytes, moe_stream_t stream);

/* Stages of the MXFP8 forward, for moe_fwd_mxfp8_stages. */
enum {
    MOE_MX_STAGE_DISPATCH = 0, /* status word cleared, routing, x rows gathered and quantized (XQ) */
    MOE_MX_STAGE_GATE_UP = 1,  /* gate/up GEMM, SwiGLU, H quantized (HQ)                             */
    MOE_MX_STAGE_DOWN = 2,     /* down GEMM with the score (Y)                                        */
    MOE_MX_STAGE_COMBINE = 3,  /* out from Y                                                          */
    MOE_MX_STAGES = 4
};

/*
 * Stages stage_begin .. stage_end-1 of moe_routed_experts_fwd_mxfp8 (0 <= stage_begin <= stage_end
 * <= MOE_MX_STAGES; the full range is that call). Arguments as for moe_routed_experts_fwd_mxfp8;
 * a stage reads what the earlier stages left in the same workspace, so stages run in order on
 * one stream. Lets a caller time each stage with events or read an intermediate region.
 */
moe_status_t moe_fwd_mxfp8_stages(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                  int32_t scores_dtype, const void *w13_data, const void *w13_scales,
                                  const void *w2_data, const void *w2_scales, void *out, int64_t T, int32_t D,
                                  int32_t F, int32_t E, int32_t K, int32_t stage_begin, int32_t stage_end,
                                  void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* NVFP4 forward, inference (Dist-MoE 0.1.0, "Choose a precision and pipeline / NVFP4":          */
/* inference only, prepared weights).                                                          */
/*                                                                                              */
/* The format, read as NVIDIA's two-level NVFP4: E2M1 elements in blocks of 16 along a GEMM's    */
/* contraction axis; a block scale S = E4M3(amax / (6 G)) stored as a UE4M3 byte (nearest even, */
/* saturating at 448); a per-tensor fp32 scale G; elements E2M1(v / (S G)) (nearest even,       */
/* saturating at 6, sign kept; +0 when S = 0), value = e2m1 * S * G. The fp32 steps are fixed:   */
/* t = 6 G, b = amax / t, r = 1 / (S G) (IEEE reciprocal of the fp32 product), v * r. A weight's */
/* G = amax(tensor) / 2688, found by moe_nvfp4_prepare_weight; the activations' G (x_scale for x, */
/* h_scale for the SwiGLU output) are calibration constants passed to the forward call. E2M1    */
/* codes are packed two per byte, the lower K index in the low nibble.                          */
/* Shape limits: those of the MXFP8 entry points (D and F multiples of 128).                    */
/* ------------------------------------------------------------------------------------------ */

/*
 * Sizes of a prepared NVFP4 weight (host outputs, caller-owned). Pure arithmetic.
 *   MOE_WEIGHT_W13: data E*2F*D/2;  scales 256 + E * ceil(F/64) * P(D) * 512
 *   MOE_WEIGHT_W2:  data E*D*F/2;   scales 256 + E * ceil(D/128) * P(F) * 512
 * with P(C) = 4 * ceil(C/256) scale groups of 64 K values per row (padded to whole 256-wide steps).
 */
moe_status_t moe_nvfp4_weight_bytes(int32_t which, int32_t D, int32_t F, int32_t E, size_t *data_bytes,
                                    size_t *scale_bytes);

/*
 * Prepares one expert weight for the NVFP4 forward:
 *   w       device bf16: w13 [E,2,F,D] (MOE_WEIGHT_W13) or w2 [E,D,F] (MOE_WEIGHT_W2)
 *   data    device: packed E2M1 codes in w's element order (w13 as [E*2F, D/2] bytes, w2 as
 *           [E*D, F/2])
 *   scales  device, 256-byte aligned: a 256-byte header (the fp32 tensor scale G at byte 0), then
 *           the UE4M3 scales grouped per GEMM tile: the scale of row n of tile (e, j) and 16-block
 *           b along the row sits at byte
 *             256 + ((e * NT + j) * P(C) + b / 4) * 512 + 16 * (n % 32) + 4 * (n / 32) + b % 4
 *           with C the row length. w13: NT = ceil(F/64), tile j holds gate rows f = 64j + n (n < 64)
 *           then up rows f = 64j + n - 64; w2: NT = ceil(D/128), row d = 128j + n. Bytes that belong
 *           to no row are 0.
 * Deterministic. Capacities at least moe_nvfp4_weight_bytes' (MOE_ERR_WORKSPACE_TOO_SMALL otherwise).
 */
moe_status_t moe_nvfp4_prepare_weight(int32_t which, const void *w, int32_t D, int32_t F, int32_t E,
                                      void *data, size_t data_bytes, void *scales, size_t scale_bytes,
                                      moe_stream_t stream);

/* Bytes of device workspace of the NVFP4 forward, and its layout: the MOE_MXWS_* regions, with XQ
 * and HQ holding packed E2M1 codes ([Rp, D/2] and [Rp, F/2] bytes) and XS and HS UE4M3 scales
 * (padded row p, 16-block b at byte ((p/128) * P(cols) + b/4) * 512 + 16 (p%32) + 4 ((p%128)/32)
 * + b%4). The padding rows after each expert's rows have zero scales in XS and zero codes and
 * scales in HQ / HS; their XQ codes are left unwritten (a zero scale makes them contribute 0).
 * Pure arithmetic. */
size_t moe_nvfp4_workspace_bytes(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K);
moe_status_t moe_nvfp4_workspace_layout(int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                        size_t *region_offsets);

/*
 * The NVFP4 forward: out as for moe_routed_experts_fwd, computed from NVFP4-quantized x (tensor
 * scale x_scale), w13, h (tensor scale h_scale) and w2, with fp32 accumulation (block-scaled
 * tcgen05 tensor-core GEMMs). x_scale and h_scale: finite and > 0 (MOE_ERR_INVALID_ARG otherwise).
 * Other arguments as for moe_routed_experts_fwd_mxfp8, with weights from
 * moe_nvfp4_prepare_weight and a workspace of moe_nvfp4_workspace_bytes.
 */
moe_status_t moe_routed_experts_fwd_nvfp4(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                          int32_t scores_dtype, const void *w13_data, const void *w13_scales,
                                          const void *w2_data, const void *w2_scales, float x_scale,
                                          float h_scale, void *out, int64_t T, int32_t D, int32_t F, int32_t E,
                                          int32_t K, void *workspace, size_t workspace_bytes,
                                          moe_stream_t stream);

/* Stages stage_begin .. stage_end-1 (MOE_MX_STAGE_*) of moe_routed_experts_fwd_nvfp4. */
moe_status_t moe_fwd_nvfp4_stages(const void *x, const int32_t *topk_ids, const void *topk_scores,
                                  int32_t scores_dtype, const void *w13_data, const void *w13_scales,
                                  const void *w2_data, const void *w2_scales, float x_scale, float h_scale,
                                  void *out, int64_t T, int32_t D, int32_t F, int32_t E, int32_t K,
                                  int32_t stage_begin, int32_t stage_end, void *workspace,
                                  size_t workspace_bytes, moe_stream_t stream);

/* Capacity of the library-owned scratch of moe_routing_static_scratch, in int32 entries per
 * array: it serves sizes with (E + 1) * ceil(T*K / 2048) <= this value. */
#define MOE_STATIC_SCRATCH_MAX_ENTRIES 262144

/*
 * Routing (the same results as moe_routing, bit for bit) without any caller-provided workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot allocate device
 * memory at the point of the call -- for example an engine whose device memory is all owned and
 * pre-planned by another allocator, or a plain C host program with no allocator at hand -- and so
 * cannot pass moe_routing a workspace. It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 *   topk_ids, counts, offsets, perm, inv   as for moe_routing (device, caller-owned)
 *   device_status  device uint32, caller-owned, or NULL: cleared, then receives the MOE_DEV_* bits
 *                  of this call (an id outside [0, E) sets MOE_DEV_BAD_EXPERT_ID)
 *
 * Scratch: a fixed array inside the library (a file-scope __device__ variable of
 * 2 * MOE_STATIC_SCRATCH_MAX_ENTRIES int32 plus 256 bytes, about 2 MiB), held on every GPU that
 * loads the library until the process exits. Sizes with (E + 1) * ceil(T*K / 2048) above
 * MOE_STATIC_SCRATCH_MAX_ENTRIES return MOE_ERR_UNSUPPORTED_SHAPE before anything is enqueued.
 *
 * Set-up: every call looks up the array's device address on the current device with
 * cudaGetSymbolAddress (nothing is cached, so a device reset, after which the array may move, needs
 * no special handling). The first lookup on a device may load the library's device code: make the
 * first call on each device before any stream capture. Every call on a device shares the one array
 * and it keeps the previous call's contents; the call clears the status slot it uses and rewrites
 * all of the other scratch it reads. Calls whose GPU work overlaps (on different streams, or from
 * different threads without ordering) race on the array: order them on one stream.
 */
moe_status_t moe_routing_static_scratch(const int32_t *topk_ids, int64_t T, int32_t E, int32_t K,
                                        int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                                        uint32_t *device_status, moe_stream_t stream);

/*
 * Reads the device status word at the start of `workspace` (a forward or a routing workspace)
 * into *device_bits (host memory): 0, or an OR of MOE_DEV_* bits raised since the last
 * moe_fwd_dispatch / moe_routed_experts_fwd / moe_routing on that workspace. Synchronises
 * `stream` first; the only synchronising entry point.
 */
moe_status_t moe_get_status(const void *workspace, uint32_t *device_bits, moe_stream_t stream);

/*
 * Failure-detection self-test. Every wait inside the library's kernels is bounded; when one runs
 * out the kernel sets MOE_DEV_TIMEOUT and returns instead of hanging. This launches one small
 * kernel whose wait can never be satisfied (an mbarrier that nothing arrives on), bounded at
 * timeout_us microseconds (1 .. 2000000), so that path can be checked on a GPU.
 *   device_status  device uint32, caller-owned: cleared, then set to MOE_DEV_TIMEOUT
 */
moe_status_t moe_selftest_wait_timeout(uint32_t timeout_us, uint32_t *device_status,
                                       moe_stream_t stream);

/* A static, human-readable name for a status code. */
const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTED_EXPERTS_H */
