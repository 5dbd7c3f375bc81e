/*
 * moe_oracle.c -- CPU oracle for the routed top-k expert layer (forward pass).
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of bench.py
 * load this library. The CUDA library never calls it, and the two share no code, header, table or
 * helper: the only thing they have in common is the seeded input generator that feeds both.
 *
 * What it computes, for every token t (a plain per-token loop, no blocking or fusion):
 *
 *     out[t] = sum_{k<K} score[t,k] * W2[e] ( SiLU(Wg[e] x_t) * (Wu[e] x_t) ),   e = ids[t,k]
 *
 * Sources for the definition:
 *   - Dist-MoE 0.1.0 (PyPI description), "Understand the execution model": the call routes rows,
 *     then runs W13, SwiGLU, W2 and the combine; "BF16 Quickstart": the tensors x_TD,
 *     topk_expert_ids_TK, topk_scores_TK, w13_E2FD ([E,2,F,D]), w2_EDF ([E,D,F]);
 *     "Choose a precision and pipeline / BF16": BF16 operands, FP32 accumulation.
 *   - TeraMoE README, worker list: the compute worker does the gate/up projection, the activation
 *     and the down projection; the combine worker applies the final weighted accumulation.
 *   - Primus MegaMoE technical guide, introduction and weight-module diagram: dispatch grouped GEMM
 *     -> SwiGLU -> grouped GEMM with weighted reduce; w1 [g, 2I, H] holds gate then up, w2 [g, H, I].
 *
 * Precision: inputs are bf16 bit patterns, decoded here by a 16-bit shift; every product and sum
 * is fp32, summed in ascending index order, as the pages' BF16 path accumulates in FP32. Built
 * with -ffp-contract=off so no multiply-add is fused and x86 and Arm hosts give the same bits.
 *
 * The MXFP8 forward (oracle_routed_experts_mxfp8, after the backward) is the same definition with
 * block-scaled E4M3 operands; its own header states the format it reads.
 *
 * The backward pass (oracle_routed_experts_bwd) is the same definition
 * differentiated by hand; the pages name its parts (Dist-MoE 0.1.0, "Understand the execution
 * model": DGRAD computes input gradients and WGRAD weight gradients; TeraMoE README, usage
 * example: output.backward(...)).
 *
 * Readings where the pages say nothing:
 *   - w13[e,0] is the gate (goes through SiLU), w13[e,1] the up projection.
 *   - SiLU(g) = g / (1 + exp(-g)) (the logistic-sigmoid-weighted linear unit), host libm expf.
 *   - The score multiplies the expert output after W2, before the sum over k.
 *   - An id outside [0, E) contributes nothing (the pages trap on bad input; this layer reports
 *     it instead); duplicate ids within a token simply add.
 *   - The routed order inside one expert's segment is ascending flat pair index t*K+k.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float bf16_to_f32(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a float to the nearest bf16, ties to even (used only by the optional round_h mode, which
 * mirrors a device path that stores the SwiGLU output in bf16). */
static float round_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {
        u &= 0xffff0000u; /* inf stays inf; a NaN keeps its top mantissa bits */
        if ((u & 0x007f0000u) == 0 && (f != f)) u |= 0x00400000u;
    } else {
        u += 0x7fffu + ((u >> 16) & 1u);
        u &= 0xffff0000u;
    }
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Routing (the local form of the pages' dispatch: "route on GPU" in Dist-MoE's execution model;
 * "tokens are written directly to their expert-grouped positions" in the MoonEP FAQ).
 *
 * The R = T*K pairs i = t*K + k get the key key(i) = ids[i] if 0 <= ids[i] < E, else E.
 *   counts[e]  = #{ i : key(i) = e }                          for e < E
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]    (offsets[E] = number of valid pairs)
 *   perm[r]    = the i of row r, rows sorted by (key(i), i) ascending (a stable counting sort;
 *                invalid pairs fill rows offsets[E] .. R-1 in ascending i)
 *   inv[i]     = the row of pair i, so inv[perm[r]] = r.
 * Returns the number of invalid ids, or -1 on a bad argument.
 */
long oracle_routing(const int32_t *ids, int64_t T, int32_t E, int32_t K, int32_t *counts,
                    int32_t *offsets, int32_t *perm, int32_t *inv) {
    if (T < 0 || E <= 0 || K <= 0) return -1;
    int64_t R = T * (int64_t)K;
    int64_t *next = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t *tally = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    if (!next || !tally) {
        free(next);
        free(tally);
        return -1;
    }
    long invalid = 0;
    for (int64_t i = 0; i < R; ++i) {
        int32_t e = ids[i];
        if (e >= 0 && e < E) {
            tally[e] += 1;
        } else {
            tally[E] += 1;
            invalid += 1;
        }
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) {
        counts[e] = (int32_t)tally[e];
        offsets[e + 1] = offsets[e] + counts[e];
    }
    for (int32_t e = 0; e <= E; ++e) next[e] = (e < E) ? offsets[e] : offsets[E];
    for (int64_t i = 0; i < R; ++i) {
        int32_t e = ids[i];
        int32_t key = (e >= 0 && e < E) ? e : E;
        int64_t r = next[key]++;
        perm[r] = (int32_t)i;
        inv[i] = (int32_t)r;
    }
    free(next);
    free(tally);
    return invalid;
}

typedef struct {
    const uint16_t *x;
    const int32_t *ids;
    const void *scores;
    int scores_bf16;
    const uint16_t *w13;
    const uint16_t *w2;
    float *out;
    int64_t t_begin, t_end;
    int32_t D, F, E, K;
    int round_h;
    int rmsnorm;       /* 1: route-wise RMSNorm of each expert output before the score */
    float rms_eps;
    /* MXFP8 forward only: prepared weights as E4M3 codes and UE8M0 block-scale codes */
    const uint8_t *w13q, *w13s, *w2q, *w2s;
    int failed;
} oracle_job;

static float pair_score(const oracle_job *job, int64_t pair) {
    if (job->scores_bf16) return bf16_to_f32(((const uint16_t *)job->scores)[pair]);
    return ((const float *)job->scores)[pair];
}

/* The definition above, for tokens t_begin .. t_end-1. */
static void *oracle_tokens(void *arg) {
    oracle_job *job = (oracle_job *)arg;
    const int32_t D = job->D, F = job->F, E = job->E, K = job->K;
    float *xt = (float *)malloc(sizeof(float) * (size_t)D);
    float *acc = (float *)malloc(sizeof(float) * (size_t)D);
    float *h = (float *)malloc(sizeof(float) * (size_t)F);
    float *xt_y = (float *)malloc(sizeof(float) * (size_t)D);
    if (!xt || !acc || !h || !xt_y) {
        job->failed = 1;
        free(xt);
        free(acc);
        free(h);
        free(xt_y);
        return NULL;
    }
    for (int64_t t = job->t_begin; t < job->t_end; ++t) {
        for (int32_t d = 0; d < D; ++d) xt[d] = bf16_to_f32(job->x[t * D + d]);
        for (int32_t j = 0; j < D; ++j) acc[j] = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = job->ids[t * K + k];
            if (e < 0 || e >= E) continue;
            float s = pair_score(job, t * K + k);
            const uint16_t *wg = job->w13 + ((size_t)e * 2 + 0) * (size_t)F * (size_t)D;
            const uint16_t *wu = job->w13 + ((size_t)e * 2 + 1) * (size_t)F * (size_t)D;
            const uint16_t *w2e = job->w2 + (size_t)e * (size_t)D * (size_t)F;
            /* gate/up projection and SwiGLU */
            for (int32_t f = 0; f < F; ++f) {
                float g = 0.0f, u = 0.0f;
                for (int32_t d = 0; d < D; ++d) {
                    g += bf16_to_f32(wg[(size_t)f * D + d]) * xt[d];
                    u += bf16_to_f32(wu[(size_t)f * D + d]) * xt[d];
                }
                float silu = g / (1.0f + expf(-g));
                h[f] = silu * u;
                if (job->round_h) h[f] = round_to_bf16(h[f]);
            }
            /* down projection, weighted by the pair's score */
            if (!job->rmsnorm) {
                for (int32_t j = 0; j < D; ++j) {
                    float y = 0.0f;
                    for (int32_t f = 0; f < F; ++f) y += bf16_to_f32(w2e[(size_t)j * F + f]) * h[f];
                    acc[j] += s * y;
                }
            } else {
                /* route-wise RMSNorm: y / sqrt(mean(y^2) + eps), then the score */
                float ss = 0.0f;
                for (int32_t j = 0; j < D; ++j) {
                    float y = 0.0f;
                    for (int32_t f = 0; f < F; ++f) y += bf16_to_f32(w2e[(size_t)j * F + f]) * h[f];
                    xt_y[j] = y;
                    ss += y * y;
                }
                const float rstd = 1.0f / sqrtf(ss / (float)D + job->rms_eps);
                for (int32_t j = 0; j < D; ++j) acc[j] += s * (xt_y[j] * rstd);
            }
        }
        for (int32_t j = 0; j < D; ++j) job->out[t * D + j] = acc[j];
    }
    free(xt);
    free(acc);
    free(h);
    free(xt_y);
    return NULL;
}

static int oracle_forward(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                          const uint16_t *w13, const uint16_t *w2, float *out, int64_t T, int32_t D,
                          int32_t F, int32_t E, int32_t K, int round_h, int rmsnorm, float rms_eps,
                          int nthreads);

/*
 * The forward with Dist-MoE's typed post-expert processing (Dist-MoE 0.1.0, "Use advanced
 * features / Post-expert processing": route-wise RMSNorm, router-score weighting and top-k
 * reduction in one step):
 *     out[t] = sum_k score[t,k] * y / sqrt(mean_d(y^2) + eps),   y = W2[e] (SiLU(Wg[e] x_t) * Wu[e] x_t)
 * Reading: the normalisation has no gain vector (the page names only eps and dtypes); the norm
 * is taken in fp32 (its norm_output_dtype) and the sum in fp32.
 */
int oracle_routed_experts_rmsnorm(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                                  const uint16_t *w13, const uint16_t *w2, float *out, int64_t T, int32_t D,
                                  int32_t F, int32_t E, int32_t K, float eps, int nthreads) {
    return oracle_forward(x, ids, scores, scores_bf16, w13, w2, out, T, D, F, E, K, 0, 1, eps, nthreads);
}

/*
 * out[T,D] (fp32) of the routed-experts forward. x [T,D], w13 [E,2,F,D] and w2 [E,D,F] are bf16
 * bit patterns; ids [T,K] int32; scores [T,K] fp32 (scores_bf16 = 0) or bf16 bits (= 1).
 * round_h = 1 rounds the SwiGLU output to bf16 before W2. Tokens are split across nthreads POSIX
 * threads (each token is computed by one thread, in the same order, whatever nthreads is).
 * Returns 0, or -1 on a bad argument or an allocation failure.
 */
static int oracle_forward(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                          const uint16_t *w13, const uint16_t *w2, float *out, int64_t T, int32_t D,
                          int32_t F, int32_t E, int32_t K, int round_h, int rmsnorm, float rms_eps,
                          int nthreads) {
    if (T < 0 || D <= 0 || F <= 0 || E <= 0 || K <= 0) return -1;
    if (T == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > T) nthreads = (int)T;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -1;
    }
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        oracle_job *j = &jobs[i];
        j->x = x;
        j->ids = ids;
        j->scores = scores;
        j->scores_bf16 = scores_bf16;
        j->w13 = w13;
        j->w2 = w2;
        j->out = out;
        j->t_begin = T * i / nthreads;
        j->t_end = T * (i + 1) / nthreads;
        j->D = D;
        j->F = F;
        j->E = E;
        j->K = K;
        j->round_h = round_h;
        j->rmsnorm = rmsnorm;
        j->rms_eps = rms_eps;
    }
    unsigned char *running = (unsigned char *)calloc((size_t)nthreads, 1);
    if (!running) {
        free(jobs);
        free(tids);
        return -1;
    }
    for (int i = 1; i < nthreads; ++i)
        running[i] = (pthread_create(&tids[i], NULL, oracle_tokens, &jobs[i]) == 0);
    oracle_tokens(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (running[i]) pthread_join(tids[i], NULL);
    for (int i = 1; i < nthreads; ++i)
        if (!running[i]) oracle_tokens(&jobs[i]); /* could not start a thread: run its tokens here */
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].failed) rc = -1;
    free(running);
    free(jobs);
    free(tids);
    return rc;
}

int oracle_routed_experts(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                          const uint16_t *w13, const uint16_t *w2, float *out, int64_t T, int32_t D,
                          int32_t F, int32_t E, int32_t K, int round_h, int nthreads) {
    return oracle_forward(x, ids, scores, scores_bf16, w13, w2, out, T, D, F, E, K, round_h, 0, 0.0f, nthreads);
}

/* ------------------------------------------------------------------------------------------ */
/* Backward pass.                                                                              */
/*                                                                                             */
/* For a pair p = (t, k) with e = ids[p], s = scores[p] and upstream gradient dout[t] (D):     */
/*   g = Wg[e] x_t, u = Wu[e] x_t, a = SiLU(g), h = a * u, y = W2[e] h     (the forward)      */
/*   dscores[p]  = <dout[t], y>                                                                */
/*   dh          = s * W2[e]^T dout[t]                                                      */
/*   dg          = dh * u * SiLU'(g),  SiLU'(g) = sig(g) (1 + g (1 - sig(g)))             */
/*   du          = dh * a                                                                     */
/*   dx[t]      += Wg[e]^T dg + Wu[e]^T du                                                    */
/*   dW2[e]     += (s * dout[t]) h^T                                                           */
/*   dWg[e]     += dg x_t^T,   dWu[e] += du x_t^T                                             */
/* Pairs with ids outside [0, E) contribute nothing and get dscores = 0.                       */
/* Pass A (tokens in parallel) gives dx and dscores; pass B (experts in parallel) gives the     */
/* weight gradients, summing each expert's pairs in ascending t*K+k. All of it in fp32.        */

typedef struct {
    const oracle_job *fw; /* shapes and forward inputs */
    const float *dout;
    float *dx, *dscores, *dw13, *dw2;
    int32_t e_begin, e_end; /* pass B range */
    int failed;
} oracle_bwd_job;

/* g, u, a, h and W2^T dout[t] for one pair (the shared recomputation of both passes). */
static void pair_recompute(const oracle_job *fw, const float *xt, const float *dout_t, int32_t e,
                           float *g, float *u, float *a, float *h, float *w2t_dout) {
    const int32_t D = fw->D, F = fw->F;
    const uint16_t *wg = fw->w13 + ((size_t)e * 2 + 0) * (size_t)F * (size_t)D;
    const uint16_t *wu = fw->w13 + ((size_t)e * 2 + 1) * (size_t)F * (size_t)D;
    const uint16_t *w2e = fw->w2 + (size_t)e * (size_t)D * (size_t)F;
    for (int32_t f = 0; f < F; ++f) {
        float gs = 0.0f, us = 0.0f;
        for (int32_t d = 0; d < D; ++d) {
            gs += bf16_to_f32(wg[(size_t)f * D + d]) * xt[d];
            us += bf16_to_f32(wu[(size_t)f * D + d]) * xt[d];
        }
        g[f] = gs;
        u[f] = us;
        a[f] = gs / (1.0f + expf(-gs));
        h[f] = a[f] * us;
    }
    for (int32_t f = 0; f < F; ++f) w2t_dout[f] = 0.0f;
    for (int32_t j = 0; j < D; ++j) {
        const float dj = dout_t[j];
        for (int32_t f = 0; f < F; ++f) w2t_dout[f] += bf16_to_f32(w2e[(size_t)j * F + f]) * dj;
    }
}

static float silu_grad(float g) {
    const float sig = 1.0f / (1.0f + expf(-g));
    return sig * (1.0f + g * (1.0f - sig));
}

/* Pass A: dx[t] and dscores[t, :] for tokens t_begin .. t_end-1 (range in the forward job). */
static void *oracle_bwd_tokens(void *arg) {
    oracle_bwd_job *job = (oracle_bwd_job *)arg;
    const oracle_job *fw = job->fw;
    const int32_t D = fw->D, F = fw->F, E = fw->E, K = fw->K;
    float *buf = (float *)malloc(sizeof(float) * ((size_t)2 * D + (size_t)7 * F));
    if (!buf) {
        job->failed = 1;
        return NULL;
    }
    float *xt = buf, *dxt = buf + D, *g = dxt + D, *u = g + F, *a = u + F, *h = a + F, *w2t = h + F,
          *dg = w2t + F, *du = dg + F;
    for (int64_t t = fw->t_begin; t < fw->t_end; ++t) {
        const float *dout_t = job->dout + t * D;
        for (int32_t d = 0; d < D; ++d) xt[d] = bf16_to_f32(fw->x[t * D + d]);
        for (int32_t d = 0; d < D; ++d) dxt[d] = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
            const int32_t e = fw->ids[t * K + k];
            job->dscores[t * K + k] = 0.0f;
            if (e < 0 || e >= E) continue;
            const float s = pair_score(fw, t * K + k);
            pair_recompute(fw, xt, dout_t, e, g, u, a, h, w2t);
            /* dscores = <dout, W2 h> = <W2^T dout, h> */
            float ds = 0.0f;
            for (int32_t f = 0; f < F; ++f) ds += w2t[f] * h[f];
            job->dscores[t * K + k] = ds;
            for (int32_t f = 0; f < F; ++f) {
                const float dh = s * w2t[f];
                dg[f] = dh * u[f] * silu_grad(g[f]);
                du[f] = dh * a[f];
            }
            const uint16_t *wg = fw->w13 + ((size_t)e * 2 + 0) * (size_t)F * (size_t)D;
            const uint16_t *wu = fw->w13 + ((size_t)e * 2 + 1) * (size_t)F * (size_t)D;
            for (int32_t d = 0; d < D; ++d) {
                float acc = 0.0f;
                for (int32_t f = 0; f < F; ++f)
                    acc += bf16_to_f32(wg[(size_t)f * D + d]) * dg[f] + bf16_to_f32(wu[(size_t)f * D + d]) * du[f];
                dxt[d] += acc;
            }
        }
        for (int32_t d = 0; d < D; ++d) job->dx[t * D + d] = dxt[d];
    }
    free(buf);
    return NULL;
}

/* Pass B: weight gradients of experts e_begin .. e_end-1. */
static void *oracle_bwd_experts(void *arg) {
    oracle_bwd_job *job = (oracle_bwd_job *)arg;
    const oracle_job *fw = job->fw;
    const int32_t D = fw->D, F = fw->F, K = fw->K;
    const int64_t R = fw->t_end * (int64_t)K; /* fw covers all tokens here */
    float *buf = (float *)malloc(sizeof(float) * ((size_t)D + (size_t)7 * F));
    if (!buf) {
        job->failed = 1;
        return NULL;
    }
    float *xt = buf, *g = xt + D, *u = g + F, *a = u + F, *h = a + F, *w2t = h + F, *dg = w2t + F, *du = dg + F;
    for (int32_t e = job->e_begin; e < job->e_end; ++e) {
        float *dwg = job->dw13 + ((size_t)e * 2 + 0) * (size_t)F * (size_t)D;
        float *dwu = job->dw13 + ((size_t)e * 2 + 1) * (size_t)F * (size_t)D;
        float *dw2e = job->dw2 + (size_t)e * (size_t)D * (size_t)F;
        for (size_t i = 0; i < (size_t)F * D; ++i) dwg[i] = dwu[i] = 0.0f;
        for (size_t i = 0; i < (size_t)D * F; ++i) dw2e[i] = 0.0f;
        for (int64_t p = 0; p < R; ++p) {
            if (fw->ids[p] != e) continue;
            const int64_t t = p / K;
            const float s = pair_score(fw, p);
            const float *dout_t = job->dout + t * D;
            for (int32_t d = 0; d < D; ++d) xt[d] = bf16_to_f32(fw->x[t * D + d]);
            pair_recompute(fw, xt, dout_t, e, g, u, a, h, w2t);
            for (int32_t f = 0; f < F; ++f) {
                const float dh = s * w2t[f];
                dg[f] = dh * u[f] * silu_grad(g[f]);
                du[f] = dh * a[f];
            }
            for (int32_t j = 0; j < D; ++j) {
                const float dy = s * dout_t[j];
                for (int32_t f = 0; f < F; ++f) dw2e[(size_t)j * F + f] += dy * h[f];
            }
            for (int32_t f = 0; f < F; ++f)
                for (int32_t d = 0; d < D; ++d) {
                    dwg[(size_t)f * D + d] += dg[f] * xt[d];
                    dwu[(size_t)f * D + d] += du[f] * xt[d];
                }
        }
    }
    free(buf);
    return NULL;
}

/*
 * Gradients of the layer for an upstream gradient dout [T,D] (fp32): dx [T,D], dscores [T,K],
 * dw13 [E,2,F,D], dw2 [E,D,F], all fp32 and written in full. Inputs as for oracle_routed_experts.
 * Returns 0, or -1 on a bad argument or an allocation failure.
 */
int oracle_routed_experts_bwd(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                              const uint16_t *w13, const uint16_t *w2, const float *dout, float *dx,
                              float *dscores, float *dw13, float *dw2, int64_t T, int32_t D, int32_t F,
                              int32_t E, int32_t K, int nthreads) {
    if (T < 0 || D <= 0 || F <= 0 || E <= 0 || K <= 0) return -1;
    if (nthreads < 1) nthreads = 1;
    oracle_job *fws = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    oracle_bwd_job *jobs = (oracle_bwd_job *)calloc((size_t)nthreads, sizeof(oracle_bwd_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    unsigned char *running = (unsigned char *)calloc((size_t)nthreads, 1);
    int rc = 0;
    if (!fws || !jobs || !tids || !running) {
        rc = -1;
        goto done;
    }
    for (int pass = 0; pass < 2; ++pass) {
        for (int i = 0; i < nthreads; ++i) {
            oracle_job *f = &fws[i];
            memset(f, 0, sizeof *f);
            f->x = x;
            f->ids = ids;
            f->scores = scores;
            f->scores_bf16 = scores_bf16;
            f->w13 = w13;
            f->w2 = w2;
            f->D = D;
            f->F = F;
            f->E = E;
            f->K = K;
            if (pass == 0) {
                f->t_begin = T * i / nthreads;
                f->t_end = T * (i + 1) / nthreads;
            } else {
                f->t_begin = 0;
                f->t_end = T;
            }
            oracle_bwd_job *j = &jobs[i];
            memset(j, 0, sizeof *j);
            j->fw = f;
            j->dout = dout;
            j->dx = dx;
            j->dscores = dscores;
            j->dw13 = dw13;
            j->dw2 = dw2;
            j->e_begin = (int32_t)((int64_t)E * i / nthreads);
            j->e_end = (int32_t)((int64_t)E * (i + 1) / nthreads);
        }
        void *(*fn)(void *) = pass == 0 ? oracle_bwd_tokens : oracle_bwd_experts;
        for (int i = 1; i < nthreads; ++i) running[i] = (pthread_create(&tids[i], NULL, fn, &jobs[i]) == 0);
        fn(&jobs[0]);
        for (int i = 1; i < nthreads; ++i)
            if (running[i]) pthread_join(tids[i], NULL);
        for (int i = 1; i < nthreads; ++i)
            if (!running[i]) fn(&jobs[i]);
        for (int i = 0; i < nthreads; ++i)
            if (jobs[i].failed) rc = -1;
    }
done:
    free(fws);
    free(jobs);
    free(tids);
    free(running);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* MXFP8 forward.                                                                              */
/*                                                                                             */
/* Dist-MoE 0.1.0, "Choose a precision and pipeline / MXFP8": the MXFP8 E4M3 format; activations */
/* are quantized after routing and the weights are prepared once ("Use advanced features /      */
/* Prepared block-scaled weights"); tensor-core products accumulate in FP32. The page names the  */
/* format but not its encoding. The reading here is the OCP Microscaling (MX) format, v1.0:     */
/*   - a block is 32 consecutive elements along the contraction axis of a GEMM operand (D for x  */
/*     and w13, F for the SwiGLU output h and w2);                                               */
/*   - the block shares one power-of-two scale X = 2^e, stored as the UE8M0 code e + 127, with  */
/*     e = floor(log2(max|v|)) - 8 (8 = the exponent of E4M3's largest normal, 448 = 1.75*2^8), */
/*     clamped to [-127, 127]; an all-zero block gets e = -127;                                 */
/*   - each element is v / X rounded to the nearest E4M3 value, ties to even, magnitudes beyond  */
/*     448 saturating to 448, the sign kept (so a negative value that rounds to zero is -0);     */
/*   - the block's value is code * X.                                                            */
/* x is quantized per token row (a routed row is a copy of it), h per pair after SwiGLU in fp32. */
/* Every product of dequantized operands and every sum is fp32, in ascending index order.        */

/* Value of an E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 */
/* holds the subnormals m * 2^-9; 0x7F and 0xFF are NaN and never produced here).               */
static double e4m3_value(uint8_t code) {
    const int sign = code >> 7, ex = (code >> 3) & 15, man = code & 7;
    const double mag = ex == 0 ? ldexp((double)man, -9) : ldexp((double)(8 + man), ex - 10);
    return sign ? -mag : mag;
}

/* The E4M3 code nearest to v (ties to even, |v| beyond 448 gives 448, the sign of v kept). The  */
/* representable magnitudes in [2^k, 2^(k+1)) are spaced 2^(k-3) for k >= -6; below 2^-6 they   */
/* are the subnormals, spaced 2^-9.                                                              */
static uint8_t e4m3_code(double v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs(v);
    int ex = 0;
    if (a > 0) (void)frexp(a, &ex); /* a = f 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
    const int k = (a > 0 && ex - 1 > -6) ? ex - 1 : -6;
    double r = ldexp(nearbyint(ldexp(a, 3 - k)), k - 3); /* default rounding mode: ties to even */
    if (r > 448.0) r = 448.0;
    if (r == 0) return sign;
    int rex = 0;
    (void)frexp(r, &rex);
    const int rk = rex - 1;
    if (rk < -6) return (uint8_t)(sign | (uint8_t)ldexp(r, 9)); /* subnormal: m 2^-9 */
    return (uint8_t)(sign | (uint8_t)((rk + 7) << 3) | (uint8_t)((int)ldexp(r, 3 - rk) - 8));
}

/* Scale exponent of a block with largest magnitude amax. */
static int mx_exponent(double amax) {
    if (!(amax > 0)) return -127;
    int ex = 0;
    (void)frexp(amax, &ex);
    int e = (ex - 1) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Quantize n = 32 values: codes[0..31] and the block's UE8M0 scale code. */
static void mx_quantize_block(const float *v, uint8_t *codes, uint8_t *scale_code) {
    double amax = 0;
    for (int i = 0; i < 32; ++i)
        if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
    const int e = mx_exponent(amax);
    for (int i = 0; i < 32; ++i) codes[i] = e4m3_code(ldexp((double)v[i], -e));
    *scale_code = (uint8_t)(e + 127);
}

/*
 * MX quantization of a bf16 matrix [rows, cols] along its rows (cols % 32 == 0): E4M3 codes
 * [rows, cols] and UE8M0 scale codes [rows, cols / 32], both row-major. This is how the MXFP8
 * weights are prepared: w13 [E, 2F, D] as E*2F rows of D, w2 [E, D, F] as E*D rows of F.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_mx_quantize_rows(const uint16_t *in, int64_t rows, int32_t cols, uint8_t *codes, uint8_t *scales) {
    if (rows < 0 || cols <= 0 || cols % 32 != 0) return -1;
    float blk[32];
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t b = 0; b < cols / 32; ++b) {
            for (int i = 0; i < 32; ++i) blk[i] = bf16_to_f32(in[r * cols + b * 32 + i]);
            mx_quantize_block(blk, codes + r * cols + b * 32, scales + r * (cols / 32) + b);
        }
    return 0;
}

/* Dequantized row: out[i] = value(codes[i]) * 2^(scales[i / 32] - 127), exact in fp32. `value`
 * is a table of e4m3_value over all 256 codes (each worker thread fills its own). */
static void mx_dequantize_row(const double *value, const uint8_t *codes, const uint8_t *scales, int32_t cols,
                              float *out) {
    for (int32_t b = 0; b < cols / 32; ++b) {
        const int e = (int)scales[b] - 127;
        for (int i = 0; i < 32; ++i) out[b * 32 + i] = (float)ldexp(value[codes[b * 32 + i]], e);
    }
}

static void *oracle_tokens_mxfp8(void *arg) {
    oracle_job *job = (oracle_job *)arg;
    const int32_t D = job->D, F = job->F, E = job->E, K = job->K;
    float *xt = (float *)malloc(sizeof(float) * (size_t)D);
    float *xd = (float *)malloc(sizeof(float) * (size_t)D);
    float *acc = (float *)malloc(sizeof(float) * (size_t)D);
    float *h = (float *)malloc(sizeof(float) * (size_t)F);
    float *hd = (float *)malloc(sizeof(float) * (size_t)F);
    float *wg = (float *)malloc(sizeof(float) * (size_t)D);
    float *wu = (float *)malloc(sizeof(float) * (size_t)D);
    float *w2r = (float *)malloc(sizeof(float) * (size_t)F);
    uint8_t *q = (uint8_t *)malloc((size_t)(D > F ? D : F));
    uint8_t *qs = (uint8_t *)malloc((size_t)(D > F ? D : F) / 32);
    double value[256];
    if (!xt || !xd || !acc || !h || !hd || !wg || !wu || !w2r || !q || !qs) {
        job->failed = 1;
        goto out;
    }
    for (int c = 0; c < 256; ++c) value[c] = e4m3_value((uint8_t)c);
    for (int64_t t = job->t_begin; t < job->t_end; ++t) {
        /* the token row, quantized and dequantized */
        for (int32_t b = 0; b < D / 32; ++b) {
            for (int i = 0; i < 32; ++i) xt[b * 32 + i] = bf16_to_f32(job->x[t * D + b * 32 + i]);
            mx_quantize_block(xt + b * 32, q + b * 32, qs + b);
        }
        mx_dequantize_row(value, q, qs, D, xd);
        for (int32_t j = 0; j < D; ++j) acc[j] = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
            const int32_t e = job->ids[t * K + k];
            if (e < 0 || e >= E) continue;
            const float s = pair_score(job, t * K + k);
            /* gate/up projection and SwiGLU, from dequantized operands */
            for (int32_t f = 0; f < F; ++f) {
                const size_t grow = ((size_t)e * 2 + 0) * (size_t)F + (size_t)f; /* row of [E*2F, D] */
                const size_t urow = ((size_t)e * 2 + 1) * (size_t)F + (size_t)f;
                mx_dequantize_row(value, job->w13q + grow * (size_t)D, job->w13s + grow * (size_t)(D / 32), D, wg);
                mx_dequantize_row(value, job->w13q + urow * (size_t)D, job->w13s + urow * (size_t)(D / 32), D, wu);
                float g = 0.0f, u = 0.0f;
                for (int32_t d = 0; d < D; ++d) {
                    g += wg[d] * xd[d];
                    u += wu[d] * xd[d];
                }
                h[f] = g / (1.0f + expf(-g)) * u;
            }
            /* h quantized after SwiGLU, then the down projection weighted by the score */
            for (int32_t b = 0; b < F / 32; ++b) mx_quantize_block(h + b * 32, q + b * 32, qs + b);
            mx_dequantize_row(value, q, qs, F, hd);
            for (int32_t j = 0; j < D; ++j) {
                const size_t row = (size_t)e * (size_t)D + (size_t)j; /* row of [E*D, F] */
                mx_dequantize_row(value, job->w2q + row * (size_t)F, job->w2s + row * (size_t)(F / 32), F, w2r);
                float y = 0.0f;
                for (int32_t f = 0; f < F; ++f) y += w2r[f] * hd[f];
                acc[j] += s * y;
            }
        }
        for (int32_t j = 0; j < D; ++j) job->out[t * D + j] = acc[j];
    }
out:
    free(xt);
    free(xd);
    free(acc);
    free(h);
    free(hd);
    free(wg);
    free(wu);
    free(w2r);
    free(q);
    free(qs);
    return NULL;
}

/*
 * out[T,D] (fp32) of the MXFP8 forward. x [T,D] bf16 bits; ids, scores as for
 * oracle_routed_experts; the weights prepared by oracle_mx_quantize_rows: w13q [E,2F,D] codes with
 * w13s [E,2F,D/32] scale codes, w2q [E,D,F] codes with w2s [E,D,F/32]. D and F must be multiples
 * of 32. Tokens are split across nthreads threads as in oracle_routed_experts.
 * Returns 0, or -1 on a bad argument or an allocation failure.
 */
int oracle_routed_experts_mxfp8(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                                const uint8_t *w13q, const uint8_t *w13s, const uint8_t *w2q,
                                const uint8_t *w2s, float *out, int64_t T, int32_t D, int32_t F, int32_t E,
                                int32_t K, int nthreads) {
    if (T < 0 || D <= 0 || F <= 0 || E <= 0 || K <= 0 || D % 32 != 0 || F % 32 != 0) return -1;
    if (T == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > T) nthreads = (int)T;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    unsigned char *running = (unsigned char *)calloc((size_t)nthreads, 1);
    int rc = 0;
    if (!jobs || !tids || !running) {
        rc = -1;
        goto done;
    }
    for (int i = 0; i < nthreads; ++i) {
        oracle_job *j = &jobs[i];
        j->x = x;
        j->ids = ids;
        j->scores = scores;
        j->scores_bf16 = scores_bf16;
        j->w13q = w13q;
        j->w13s = w13s;
        j->w2q = w2q;
        j->w2s = w2s;
        j->out = out;
        j->t_begin = T * i / nthreads;
        j->t_end = T * (i + 1) / nthreads;
        j->D = D;
        j->F = F;
        j->E = E;
        j->K = K;
    }
    for (int i = 1; i < nthreads; ++i)
        running[i] = (pthread_create(&tids[i], NULL, oracle_tokens_mxfp8, &jobs[i]) == 0);
    oracle_tokens_mxfp8(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (running[i]) pthread_join(tids[i], NULL);
    for (int i = 1; i < nthreads; ++i)
        if (!running[i]) oracle_tokens_mxfp8(&jobs[i]);
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].failed) rc = -1;
done:
    free(jobs);
    free(tids);
    free(running);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* NVFP4 forward (inference).                                                                  */
/*                                                                                             */
/* Dist-MoE 0.1.0, "Choose a precision and pipeline / NVFP4": the NVFP4 block-scaled format,     */
/* inference only, with prepared weights. The page names the format, not its encoding; the       */
/* reading here is NVIDIA's published NVFP4 two-level scaling:                                  */
/*   - elements E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3,   */
/*     4, 6), in blocks of 16 consecutive elements along the contraction axis;                  */
/*   - each block has a scale S: a positive E4M3 value (UE4M3); each tensor has an fp32 scale G; */
/*   - a block with largest magnitude amax gets S = E4M3(amax / (6 G)) (nearest, ties to even,   */
/*     saturating at 448); an element v gets E2M1(v / (S G)) (nearest, ties to even, saturating */
/*     at 6, sign kept), or +0 when S = 0; its value is e2m1 * S * G;                          */
/*   - the fp32 steps are fixed so that any implementation decides the same codes:              */
/*     t = 6 G (fp32 product), b = amax / t (fp32 quotient); r = 1 / (S G) as the fp32          */
/*     reciprocal of the fp32 product S G, and v * r (fp32 product) is rounded to E2M1;         */
/*   - a weight's G is amax(whole tensor) / 2688 (= 6 * 448) in fp32 (1 for an all-zero tensor); */
/*     the activations' G (for x and for the SwiGLU output h) are calibration constants given   */
/*     by the caller, as NVFP4 inference takes its activation scales.                           */
/* Codes are kept one per byte here (the low 4 bits).                                          */

/* Value of an E2M1 code (4 bits). */
static double e2m1_value(uint8_t code) {
    const int sign = (code >> 3) & 1, ex = (code >> 1) & 3, man = code & 1;
    const double mag = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -mag : mag;
}

/* The E2M1 code nearest to v: magnitudes 0, 0.5, 1, 1.5 are spaced 0.5, then 2, 3 (spacing 1)
 * and 4, 6 (spacing 2); ties go to the code with an even mantissa bit; beyond 6 gives 6. */
static uint8_t e2m1_code(double v) {
    const uint8_t sign = signbit(v) ? 8 : 0;
    const double a = fabs(v);
    double step = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    /* nearest multiple of the spacing, ties to the even multiple: on this grid an even multiple
     * is a value with an even mantissa bit (1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4) */
    double r = nearbyint(a / step) * step;
    if (r > 6.0) r = 6.0;
    uint8_t code = 0;
    for (uint8_t c = 0; c < 8; ++c)
        if (e2m1_value(c) == r) code = c;
    return (uint8_t)(sign | code);
}

/* One block of 16: codes (one per byte) and the block's UE4M3 scale code, for the tensor scale G. */
static void nvfp4_quantize_block(const float *v, float G, uint8_t *codes, uint8_t *scale_code) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i)
        if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
    const float t = 6.0f * G;
    const float b = amax / t;
    const uint8_t s = (uint8_t)(e4m3_code((double)b) & 0x7F);
    *scale_code = s;
    const float S = (float)e4m3_value(s);
    if (S == 0.0f) {
        for (int i = 0; i < 16; ++i) codes[i] = 0;
        return;
    }
    const float r = 1.0f / (S * G);
    for (int i = 0; i < 16; ++i) codes[i] = e2m1_code((double)(v[i] * r));
}

/* The tensor scale of a weight: amax / 2688 in fp32, 1 for an all-zero tensor. */
float oracle_nvfp4_weight_scale(const uint16_t *in, int64_t n) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf(bf16_to_f32(in[i]));
        if (a > amax) amax = a;
    }
    return amax > 0.0f ? amax / 2688.0f : 1.0f;
}

/*
 * NVFP4 quantization of a bf16 matrix [rows, cols] along its rows (cols % 16 == 0) with the
 * tensor scale G: E2M1 codes [rows, cols] (one per byte) and UE4M3 scale codes [rows, cols / 16].
 * Returns 0, or -1 on a bad argument.
 */
int oracle_nvfp4_quantize_rows(const uint16_t *in, int64_t rows, int32_t cols, float G, uint8_t *codes,
                               uint8_t *scales) {
    if (rows < 0 || cols <= 0 || cols % 16 != 0 || !(G > 0.0f)) return -1;
    float blk[16];
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t b = 0; b < cols / 16; ++b) {
            for (int i = 0; i < 16; ++i) blk[i] = bf16_to_f32(in[r * cols + b * 16 + i]);
            nvfp4_quantize_block(blk, G, codes + r * cols + b * 16, scales + r * (cols / 16) + b);
        }
    return 0;
}

/* Dequantized row: e2m1 * S * G, in fp32 (e2m1 * S exact; the product with G rounded once). */
static void nvfp4_dequantize_row(const uint8_t *codes, const uint8_t *scales, float G, int32_t cols, float *out) {
    for (int32_t b = 0; b < cols / 16; ++b) {
        const float S = (float)e4m3_value(scales[b]);
        for (int i = 0; i < 16; ++i) out[b * 16 + i] = (float)(e2m1_value(codes[b * 16 + i]) * S) * G;
    }
}

typedef struct {
    oracle_job base;
    const uint8_t *w13q, *w13s, *w2q, *w2s;
    float g13, g2, gx, gh;
} oracle_nvfp4_job;

static void *oracle_tokens_nvfp4(void *arg) {
    oracle_nvfp4_job *nj = (oracle_nvfp4_job *)arg;
    oracle_job *job = &nj->base;
    const int32_t D = job->D, F = job->F, E = job->E, K = job->K;
    float *xt = (float *)malloc(sizeof(float) * (size_t)D);
    float *xd = (float *)malloc(sizeof(float) * (size_t)D);
    float *acc = (float *)malloc(sizeof(float) * (size_t)D);
    float *h = (float *)malloc(sizeof(float) * (size_t)F);
    float *hd = (float *)malloc(sizeof(float) * (size_t)F);
    float *wg = (float *)malloc(sizeof(float) * (size_t)D);
    float *wu = (float *)malloc(sizeof(float) * (size_t)D);
    float *w2r = (float *)malloc(sizeof(float) * (size_t)F);
    uint8_t *q = (uint8_t *)malloc((size_t)(D > F ? D : F));
    uint8_t *qs = (uint8_t *)malloc((size_t)(D > F ? D : F) / 16);
    if (!xt || !xd || !acc || !h || !hd || !wg || !wu || !w2r || !q || !qs) {
        job->failed = 1;
        goto out;
    }
    for (int64_t t = job->t_begin; t < job->t_end; ++t) {
        for (int32_t b = 0; b < D / 16; ++b) {
            for (int i = 0; i < 16; ++i) xt[b * 16 + i] = bf16_to_f32(job->x[t * D + b * 16 + i]);
            nvfp4_quantize_block(xt + b * 16, nj->gx, q + b * 16, qs + b);
        }
        nvfp4_dequantize_row(q, qs, nj->gx, D, xd);
        for (int32_t j = 0; j < D; ++j) acc[j] = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
            const int32_t e = job->ids[t * K + k];
            if (e < 0 || e >= E) continue;
            const float s = pair_score(job, t * K + k);
            for (int32_t f = 0; f < F; ++f) {
                const size_t grow = ((size_t)e * 2 + 0) * (size_t)F + (size_t)f;
                const size_t urow = ((size_t)e * 2 + 1) * (size_t)F + (size_t)f;
                nvfp4_dequantize_row(nj->w13q + grow * (size_t)D, nj->w13s + grow * (size_t)(D / 16), nj->g13, D, wg);
                nvfp4_dequantize_row(nj->w13q + urow * (size_t)D, nj->w13s + urow * (size_t)(D / 16), nj->g13, D, wu);
                float g = 0.0f, u = 0.0f;
                for (int32_t d = 0; d < D; ++d) {
                    g += wg[d] * xd[d];
                    u += wu[d] * xd[d];
                }
                h[f] = g / (1.0f + expf(-g)) * u;
            }
            for (int32_t b = 0; b < F / 16; ++b) nvfp4_quantize_block(h + b * 16, nj->gh, q + b * 16, qs + b);
            nvfp4_dequantize_row(q, qs, nj->gh, F, hd);
            for (int32_t j = 0; j < D; ++j) {
                const size_t row = (size_t)e * (size_t)D + (size_t)j;
                nvfp4_dequantize_row(nj->w2q + row * (size_t)F, nj->w2s + row * (size_t)(F / 16), nj->g2, F, w2r);
                float y = 0.0f;
                for (int32_t f = 0; f < F; ++f) y += w2r[f] * hd[f];
                acc[j] += s * y;
            }
        }
        for (int32_t j = 0; j < D; ++j) job->out[t * D + j] = acc[j];
    }
out:
    free(xt);
    free(xd);
    free(acc);
    free(h);
    free(hd);
    free(wg);
    free(wu);
    free(w2r);
    free(q);
    free(qs);
    return NULL;
}

/*
 * out[T,D] (fp32) of the NVFP4 forward. x [T,D] bf16 bits, quantized per token row with the
 * activation scale gx; the SwiGLU output h is quantized per pair with gh; the weights prepared by
 * oracle_nvfp4_quantize_rows: w13q [E,2F,D] codes, w13s [E,2F,D/16] scale codes, tensor scale g13;
 * w2q [E,D,F], w2s [E,D,F/16], g2. D and F multiples of 16. ids, scores as for
 * oracle_routed_experts. Returns 0, or -1 on a bad argument or an allocation failure.
 */
int oracle_routed_experts_nvfp4(const uint16_t *x, const int32_t *ids, const void *scores, int scores_bf16,
                                const uint8_t *w13q, const uint8_t *w13s, float g13, const uint8_t *w2q,
                                const uint8_t *w2s, float g2, float gx, float gh, float *out, int64_t T, int32_t D,
                                int32_t F, int32_t E, int32_t K, int nthreads) {
    if (T < 0 || D <= 0 || F <= 0 || E <= 0 || K <= 0 || D % 16 != 0 || F % 16 != 0) return -1;
    if (!(g13 > 0.0f) || !(g2 > 0.0f) || !(gx > 0.0f) || !(gh > 0.0f)) return -1;
    if (T == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > T) nthreads = (int)T;
    oracle_nvfp4_job *jobs = (oracle_nvfp4_job *)calloc((size_t)nthreads, sizeof(oracle_nvfp4_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    unsigned char *running = (unsigned char *)calloc((size_t)nthreads, 1);
    int rc = 0;
    if (!jobs || !tids || !running) {
        rc = -1;
        goto done;
    }
    for (int i = 0; i < nthreads; ++i) {
        oracle_nvfp4_job *j = &jobs[i];
        j->base.x = x;
        j->base.ids = ids;
        j->base.scores = scores;
        j->base.scores_bf16 = scores_bf16;
        j->base.out = out;
        j->base.t_begin = T * i / nthreads;
        j->base.t_end = T * (i + 1) / nthreads;
        j->base.D = D;
        j->base.F = F;
        j->base.E = E;
        j->base.K = K;
        j->w13q = w13q;
        j->w13s = w13s;
        j->w2q = w2q;
        j->w2s = w2s;
        j->g13 = g13;
        j->g2 = g2;
        j->gx = gx;
        j->gh = gh;
    }
    for (int i = 1; i < nthreads; ++i)
        running[i] = (pthread_create(&tids[i], NULL, oracle_tokens_nvfp4, &jobs[i]) == 0);
    oracle_tokens_nvfp4(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (running[i]) pthread_join(tids[i], NULL);
    for (int i = 1; i < nthreads; ++i)
        if (!running[i]) oracle_tokens_nvfp4(&jobs[i]);
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].base.failed) rc = -1;
done:
    free(jobs);
    free(tids);
    free(running);
    return rc;
}
