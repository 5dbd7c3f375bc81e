// backward.cu -- the backward pass of the routed-experts layer (Dist-MoE 0.1.0, "Understand the
// execution model": FPROP, then DGRAD for input gradients and WGRAD for weight gradients; the
// TeraMoE README's usage example calls output.backward). It recomputes what it needs instead of
// keeping forward activations (the pages' activation recompute).
//
// For a pair p = (t, k) with e = ids[p], s = scores[p] and upstream gradient dout[t]:
//   g = Wg[e] x_t, u = Wu[e] x_t, a = SiLU(g), h = a * u           (recomputed)
//   q = W2[e]^T dout[t]            dscores[p] = <q, h>   (= <dout[t], W2[e] h>)
//   dh = s q, dg = dh * u * SiLU'(g), du = dh * a
//   dx[t] += Wg[e]^T dg + Wu[e]^T du
//   dW2[e] += dout[t] (s h)^T,  dWg[e] += dg x_t^T,  dWu[e] += du x_t^T
//
// Layout: every expert's routed rows are padded to a multiple of 128 ("padded rows"), with zero
// rows in the padding, so that row tiles never straddle two experts and the weight-gradient
// GEMMs, which contract over an expert's rows, never read another expert's rows.
//
// Kernels, in stream order:
//   routing (shared with the forward) -> k_pad_tiles -> k_pad_rows -> k_gather_bwd (token order)
//   -> recompute (A = XPP rows, B = w13): GU = [g | u], HS = s h
//   -> dgrad of the down projection (A = DOP rows, B = W2 read MN-major): q = dout W2, with the
//      SwiGLU backward in the epilogue: DGU = [dg | du] and partial dscores per column tile
//   -> dgrad of gate/up (A = DGU rows, B = w13 read MN-major): DXP = DGU w13
//   -> wgrad of W2 (A = DOP, B = HS, both MN-major, K = the expert's padded rows)
//   -> wgrad of w13 (A = DGU, B = XPP, both MN-major)
//   -> k_dscores (sums the partials in fixed order) and k_dx_combine (sums a token's K rows of
//      DXP in k order) -- both deterministic.
#include "gemm_pipeline.cuh"

namespace moe {
namespace {

constexpr int kPadRows = 128;  // padded segment granularity (= the row tile)

// ---------------------------------------------------------------------------- padded routing

// One block: pmt[e] = sum_{e' < e} ceil(counts[e'] / 128) (padded row tiles), pmt[E] = total.
__global__ void __launch_bounds__(1024) k_pad_tiles(const int32_t* __restrict__ counts, int32_t E,
                                                    int32_t* __restrict__ pmt) {
    __shared__ int32_t warp_sums[32];
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int e0 = static_cast<int>(static_cast<int64_t>(E) * tid / nt);
    const int e1 = static_cast<int>(static_cast<int64_t>(E) * (tid + 1) / nt);
    int32_t m = 0;
    for (int e = e0; e < e1; ++e) m += (counts[e] + kPadRows - 1) / kPadRows;
    int32_t inc = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < (nt >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < (nt >> 5)) warp_sums[lane] = w;
    }
    __syncthreads();
    int32_t run = (warp == 0 ? 0 : warp_sums[warp - 1]) + inc - m;
    for (int e = e0; e < e1; ++e) {
        pmt[e] = run;
        run += (counts[e] + kPadRows - 1) / kPadRows;
    }
    if (tid == nt - 1) pmt[E] = run;
}

// Pair p with routed row r of expert e goes to padded row 128 * pmt[e] + (r - offsets[e]).
__global__ void __launch_bounds__(256) k_pad_rows(const int32_t* __restrict__ ids, const int32_t* __restrict__ inv,
                                                  const int32_t* __restrict__ offsets, const int32_t* __restrict__ pmt,
                                                  int64_t R, int32_t E, int32_t* __restrict__ pperm,
                                                  int32_t* __restrict__ pinv) {
    griddep_wait();
    griddep_launch_dependents();
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < R;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t e = __ldg(ids + p);
        if (e < 0 || e >= E) {
            pinv[p] = -1;
            continue;
        }
        const int32_t prow = kPadRows * __ldg(pmt + e) + (__ldg(inv + p) - __ldg(offsets + e));
        pperm[prow] = static_cast<int32_t>(p);
        pinv[p] = prow;
    }
}

// XPP[pinv[p]] = x[t], DOP[pinv[p]] = dout[t] for every valid pair p = t K + k, in token order: a
// work item is one 1024-column chunk of one token (one warp, 16-byte vectors, four per lane per
// tensor), read once and written to each of the token's K padded rows, so x and dout are read
// once instead of once per pair. The next 128 * pmt[E] items zero the padding rows (pperm < 0).
constexpr int kGatherChunkVec = 128;  // 16-byte vectors per chunk

__global__ void __launch_bounds__(256) k_gather_bwd(const uint4* __restrict__ x, const uint4* __restrict__ dout,
                                                    const int32_t* __restrict__ pperm,
                                                    const int32_t* __restrict__ pinv,
                                                    const int32_t* __restrict__ pmt, int32_t E, int32_t K, int64_t T,
                                                    int vec_per_row, uint4* __restrict__ xpp,
                                                    uint4* __restrict__ dop) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t rows = static_cast<int64_t>(kPadRows) * __ldg(pmt + E);
    const int lane = threadIdx.x & 31;
    const int chunks = (vec_per_row + kGatherChunkVec - 1) / kGatherChunkVec;
    const int64_t token_items = T * chunks;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         item < token_items + rows; item += warps_total) {
        if (item < token_items) {
            const int64_t t = item / chunks;
            const int j = static_cast<int>(item - t * chunks) * kGatherChunkVec + lane;
            uint4 a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j + u * 32 < vec_per_row) {
                    a[u] = __ldg(x + t * vec_per_row + j + u * 32);
                    b[u] = __ldg(dout + t * vec_per_row + j + u * 32);
                }
            for (int k = 0; k < K; ++k) {
                const int32_t prow = __ldg(pinv + t * K + k);
                if (prow < 0) continue;  // a pair with an invalid id (warp-uniform)
                uint4* dx = xpp + static_cast<int64_t>(prow) * vec_per_row;
                uint4* dd = dop + static_cast<int64_t>(prow) * vec_per_row;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (j + u * 32 < vec_per_row) {
                        dx[j + u * 32] = a[u];
                        dd[j + u * 32] = b[u];
                    }
            }
        } else {
            const int64_t r = item - token_items;
            if (__ldg(pperm + r) >= 0) continue;
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int j = lane; j < vec_per_row; j += 32) {
                xpp[r * vec_per_row + j] = z;
                dop[r * vec_per_row + j] = z;
            }
        }
    }
}

// ------------------------------------------------------------------------------ tile policies

struct PadRowTile {
    int32_t e, n, row0, kblocks;
};

// Tile list over padded rows: expert e owns (pmt[e+1] - pmt[e]) row tiles x ntn column tiles,
// rows fastest; tile prefix ntn * pmt[e].
__device__ __forceinline__ PadRowTile decode_pad_row_tile(int32_t tile, const GemmArgs& a, int32_t ntn) {
    PadRowTile t;
    t.e = owning_expert(tile, a.pmt, ntn, a.E);
    const int32_t first = __ldg(a.pmt + t.e);
    const int32_t mt = __ldg(a.pmt + t.e + 1) - first;
    const int32_t local = tile - ntn * first;
    t.n = local / mt;
    t.row0 = kPadRows * (first + local - t.n * mt);
    t.kblocks = a.kblocks;
    return t;
}

__device__ __forceinline__ float silu_of(float g, float* sig_out) {
    const float sig = sigmoid_fast(g);
    *sig_out = sig;
    return g * sig;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Recompute: A = XPP (K-major, K = D), B = w13 gate and up rows (K-major), 128 f per tile.
// out0 = GU [rows, 2F] (g then u), out1 = HS [rows, F] (s * SiLU(g) * u).
struct BwdRecompute {
    using Tile = PadRowTile;
    static constexpr bool kAMnMajor = false, kBMnMajor = false;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows);

    __device__ static int32_t ntn(const GemmArgs& a) { return (a.F + kBN1 - 1) / kBN1; }
    __device__ static int32_t num_tiles(const GemmArgs& a) { return ntn(a) * __ldg(a.pmt + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_pad_row_tile(tile, a, ntn(a)); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        const int32_t gate = t.e * 2 * a.F + t.n * kBN1;
        tma_load_2d(sa, ta, bar, kb * kBK, t.row0);
        tma_load_2d(sb, tb, bar, kb * kBK, gate);
        tma_load_2d(sb + kBBytes / 2, tb, bar, kb * kBK, gate + a.F);
    }

    // Rows leave through the per-warp staging buffer in 64-column groups (F % 64 == 0: a group is all
    // in or all out), so each store instruction writes four whole 128-byte row segments.
    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
        const int32_t pair = __ldg(a.pperm + row);
        const float s = pair >= 0 ? pair_score(a, pair) : 0.0f;
#pragma unroll 1
        for (int cp = 0; cp < kBN1 / 64; ++cp) {
            __syncwarp();
            uint32_t g0[32], g1[32], u0[32], u1[32];
            tmem_ld_32cols(taddr + cp * 64, g0);
            tmem_ld_32cols(taddr + cp * 64 + 32, g1);
            tmem_ld_32cols(taddr + kBN1 + cp * 64, u0);
            tmem_ld_32cols(taddr + kBN1 + cp * 64 + 32, u1);
            tmem_ld_wait(g0);
            tmem_ld_tie(g1);
            tmem_ld_tie(u0);
            tmem_ld_tie(u1);
            const int32_t f0 = t.n * kBN1 + cp * 64;
            const bool ok = f0 < a.F;  // warp-uniform
            uint32_t w[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                w[j] = pack_bf16x2(__uint_as_float(g0[2 * j]), __uint_as_float(g0[2 * j + 1]));
                w[16 + j] = pack_bf16x2(__uint_as_float(g1[2 * j]), __uint_as_float(g1[2 * j + 1]));
            }
            warp_store_row_segments(stage, w, reinterpret_cast<char*>(a.out0 + row * 2 * a.F + f0), ok);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                w[j] = pack_bf16x2(__uint_as_float(u0[2 * j]), __uint_as_float(u0[2 * j + 1]));
                w[16 + j] = pack_bf16x2(__uint_as_float(u1[2 * j]), __uint_as_float(u1[2 * j + 1]));
            }
            warp_store_row_segments(stage, w, reinterpret_cast<char*>(a.out0 + row * 2 * a.F + a.F + f0), ok);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float sg;
                const float ga = __uint_as_float(g0[2 * j]), gb = __uint_as_float(g0[2 * j + 1]);
                const float gc = __uint_as_float(g1[2 * j]), gd = __uint_as_float(g1[2 * j + 1]);
                w[j] = pack_bf16x2(s * silu_of(ga, &sg) * __uint_as_float(u0[2 * j]),
                                   s * silu_of(gb, &sg) * __uint_as_float(u0[2 * j + 1]));
                w[16 + j] = pack_bf16x2(s * silu_of(gc, &sg) * __uint_as_float(u1[2 * j]),
                                        s * silu_of(gd, &sg) * __uint_as_float(u1[2 * j + 1]));
            }
            warp_store_row_segments(stage, w, reinterpret_cast<char*>(a.out1 + row * a.F + f0), ok);
        }
    }
};

// Dgrad of the down projection: A = DOP (K-major, K = D), B = W2[e] read MN-major as
// B[n = f][k = d] (four 64-wide f boxes). Epilogue: SwiGLU backward and partial dscores.
// in0 = GU, out0 = DGU [rows, 2F] (dg then du), fout = partials [rows, ceil(F/256)].
struct BwdDgradDown {
    using Tile = PadRowTile;
    static constexpr bool kAMnMajor = false, kBMnMajor = true;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows, false, true);

    __device__ static int32_t ntn(const GemmArgs& a) { return (a.F + kBN2 - 1) / kBN2; }
    __device__ static int32_t num_tiles(const GemmArgs& a) { return ntn(a) * __ldg(a.pmt + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_pad_row_tile(tile, a, ntn(a)); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * kBK, t.row0);
#pragma unroll
        for (int j = 0; j < kBRows / 64; ++j)
            tma_load_2d(sb + j * kMnBoxBytes, tb, bar, t.n * kBN2 + 64 * j, t.e * a.D + kb * kBK);
    }

    // Per 64-column group (F % 64 == 0: all in or all out): this warp's 32 rows of g and u come in
    // with coalesced loads through the staging buffer, dg and du leave the same way, so every load
    // and store instruction moves four whole 128-byte row segments.
    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        const int lane = threadIdx.x & 31;
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
        const int32_t pair = __ldg(a.pperm + row);
        const float s = pair >= 0 ? pair_score(a, pair) : 0.0f;
        const int64_t pitch = 2 * static_cast<int64_t>(a.F) * 2;  // bytes per GU / DGU row
        const char* gu_warp = reinterpret_cast<const char*>(a.in0 + (row - lane) * 2 * a.F);
        {
            // this row's g and u lines of every column group into L2 now, so that only the first
            // group's loads below wait for DRAM (GU does not fit in L2 at these sizes)
            const char* gu_row = reinterpret_cast<const char*>(a.in0 + row * 2 * a.F);
#pragma unroll
            for (int cp = 0; cp < kBN2 / 64; ++cp) {
                const int32_t f0 = t.n * kBN2 + cp * 64;
                if (f0 < a.F) {
                    prefetch_l2(gu_row + 2 * f0);
                    prefetch_l2(gu_row + 2 * (a.F + f0));
                }
            }
        }
        float partial = 0.0f;
#pragma unroll 1
        for (int cp = 0; cp < kBN2 / 64; ++cp) {
            const int32_t f0 = t.n * kBN2 + cp * 64;
            if (f0 >= a.F) break;  // warp-uniform
            uint32_t gw[32], uw[32];
            warp_load_row_segments(stage, gu_warp + 2 * f0, pitch, gw);
            warp_load_row_segments(stage, gu_warp + 2 * (a.F + f0), pitch, uw);
            __syncwarp();
            uint32_t q0[32], q1[32];
            tmem_ld_32cols(taddr + cp * 64, q0);
            tmem_ld_32cols(taddr + cp * 64 + 32, q1);
            tmem_ld_wait(q0);
            tmem_ld_tie(q1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {  // elements 2j and 2j + 1; dg, du overwrite g, u in place
                float dg2[2], du2[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = 2 * j + h;
                    const float gg = __uint_as_float(h ? (gw[j] & 0xffff0000u) : (gw[j] << 16));
                    const float uu = __uint_as_float(h ? (uw[j] & 0xffff0000u) : (uw[j] << 16));
                    const float qv = __uint_as_float(e < 32 ? q0[e] : q1[e - 32]);
                    float sig;
                    const float act = silu_of(gg, &sig);
                    partial += qv * act * uu;
                    const float dh = s * qv;
                    dg2[h] = dh * uu * sig * (1.0f + gg * (1.0f - sig));
                    du2[h] = dh * act;
                }
                gw[j] = pack_bf16x2(dg2[0], dg2[1]);
                uw[j] = pack_bf16x2(du2[0], du2[1]);
            }
            warp_store_row_segments(stage, gw, reinterpret_cast<char*>(a.out0 + row * 2 * a.F + f0), true);
            warp_store_row_segments(stage, uw, reinterpret_cast<char*>(a.out0 + row * 2 * a.F + a.F + f0), true);
        }
        a.fout[row * ntn(a) + t.n] = partial;
    }
};

// Dgrad of gate/up: A = DGU (K-major, K = 2F), B = w13[e] read MN-major as B[n = d][k = 2F rows].
// out0 = DXP [rows, D].
struct BwdDgradGateUp {
    using Tile = PadRowTile;
    static constexpr bool kAMnMajor = false, kBMnMajor = true;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows, false, true);

    __device__ static int32_t ntn(const GemmArgs& a) { return (a.D + kBN2 - 1) / kBN2; }
    __device__ static int32_t num_tiles(const GemmArgs& a) { return ntn(a) * __ldg(a.pmt + a.E); }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) { return decode_pad_row_tile(tile, a, ntn(a)); }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs& a) {
        tma_load_2d(sa, ta, bar, kb * kBK, t.row0);
#pragma unroll
        for (int j = 0; j < kBRows / 64; ++j)
            tma_load_2d(sb + j * kMnBoxBytes, tb, bar, t.n * kBN2 + 64 * j, t.e * 2 * a.F + kb * kBK);
    }

    // DXP rows leave through the staging buffer in 64-column groups (D % 64 == 0).
    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        const int64_t row = static_cast<int64_t>(t.row0) + row_in_tile;
#pragma unroll 1
        for (int cp = 0; cp < kBN2 / 64; ++cp) {
            uint32_t w[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                __syncwarp();
                uint32_t v[32];
                tmem_ld_32cols(taddr + (2 * cp + half) * 32, v);
                tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[16 * half + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            }
            const int32_t d0 = t.n * kBN2 + cp * 64;
            warp_store_row_segments(stage, w, reinterpret_cast<char*>(a.out0 + row * a.D + d0), d0 < a.D);
        }
    }
};

// Weight gradient of one projection: out0[e] [mdim, ndim] = A_e^T B_e, contracting over expert e's
// padded rows; A = [rows, mdim] and B = [rows, ndim] both read MN-major (two 64-wide m boxes,
// four 64-wide n boxes per 64-row K step). An expert without rows gets zeros.
struct BwdWgrad {
    struct Tile {
        int32_t e, m, n, krow0, kblocks;
    };
    static constexpr bool kAMnMajor = true, kBMnMajor = true;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBRows, true, true);

    __device__ static int32_t num_tiles(const GemmArgs& a) { return a.E * a.mtiles * a.ntiles; }
    __device__ static Tile decode(int32_t tile, const GemmArgs& a) {
        Tile t;
        const int32_t per = a.mtiles * a.ntiles;
        t.e = tile / per;
        const int32_t local = tile - t.e * per;
        t.n = local / a.mtiles;
        t.m = local - t.n * a.mtiles;
        const int32_t first = __ldg(a.pmt + t.e);
        t.krow0 = kPadRows * first;
        t.kblocks = (__ldg(a.pmt + t.e + 1) - first) * (kPadRows / kBK);
        return t;
    }

    __device__ static void load(const Tile& t, int32_t kb, uint8_t* sa, uint8_t* sb, uint64_t* bar,
                                const CUtensorMap* ta, const CUtensorMap* tb, const GemmArgs&) {
        const int32_t k = t.krow0 + kb * kBK;
#pragma unroll
        for (int j = 0; j < kBM / 64; ++j) tma_load_2d(sa + j * kMnBoxBytes, ta, bar, t.m * kBM + 64 * j, k);
#pragma unroll
        for (int j = 0; j < kBRows / 64; ++j) tma_load_2d(sb + j * kMnBoxBytes, tb, bar, t.n * kBRows + 64 * j, k);
    }

    // The tile's K is one expert's padded rows (a few hundred at most sizes), so its mainloop is
    // short and the 64 KB of gradient it writes decide the pace: rows leave through the per-warp
    // staging buffer, so each store instruction writes four whole 128-byte row segments instead
    // of 32 scattered 16-byte pieces.
    __device__ static void epilogue(const Tile& t, uint32_t taddr, int row_in_tile, uint4* stage, const GemmArgs& a) {
        const int32_t r = t.m * kBM + row_in_tile;
        __nv_bfloat16* dst = a.out0 + (static_cast<int64_t>(t.e) * a.mdim + r) * a.ndim;
        uint32_t words[32];  // 64 bf16 of this thread's row: two 32-column chunks
#pragma unroll 1
        for (int cp = 0; cp < kBRows / 64; ++cp) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                __syncwarp();
                uint32_t v[32];
                if (t.kblocks > 0) {  // warp-uniform
                    tmem_ld_32cols(taddr + (2 * cp + half) * 32, v);
                    tmem_ld_wait(v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0u;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    words[half * 16 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            }
            const int32_t c0 = t.n * kBRows + cp * 64;  // ndim % 64 == 0: the 64 columns are all in or all out
            warp_store_row_segments(stage, words, reinterpret_cast<char*>(dst + c0), r < a.mdim && c0 < a.ndim);
        }
    }
};

// dscores[p] = sum over the column tiles of partial[pinv[p]] (fixed order); 0 for invalid pairs.
__global__ void __launch_bounds__(256) k_dscores(const int32_t* __restrict__ pinv, const float* __restrict__ partial,
                                                 int64_t R, int32_t ntd, float* __restrict__ dscores) {
    griddep_wait();
    griddep_launch_dependents();
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < R;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t prow = __ldg(pinv + p);
        float s = 0.0f;
        if (prow >= 0)
            for (int j = 0; j < ntd; ++j) s += __ldg(partial + static_cast<int64_t>(prow) * ntd + j);
        dscores[p] = s;
    }
}

// dx[t] = bf16( sum_{k} DXP[pinv[t*K+k]] ) in k order (fp32), skipping invalid pairs.
__global__ void __launch_bounds__(256) k_dx_combine(const uint4* __restrict__ dxp, const int32_t* __restrict__ pinv,
                                                    int64_t T, int32_t K, int32_t vec_per_row,
                                                    uint4* __restrict__ dx) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t total = T * vec_per_row;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = v / vec_per_row;
        const int64_t j = v - t * vec_per_row;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < K; ++k) {
            const int32_t prow = __ldg(pinv + t * K + k);
            if (prow < 0) continue;
            float f[8];
            unpack_bf16x8(__ldg(dxp + static_cast<int64_t>(prow) * vec_per_row + j), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
        dx[v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                           pack_bf16x2(acc[6], acc[7]));
    }
}

int grid_for(int64_t work, int per_block, int sm_count) {
    const int64_t want = ceil_div(work, per_block);
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    const int64_t g = want < cap ? want : cap;
    return static_cast<int>(g > 0 ? g : 1);
}

}  // namespace

moe_status_t launch_backward(const BwdProblem& p, int stage_begin, int stage_end, cudaStream_t stream) {
    auto run = [&](int stage) { return stage_begin <= stage && stage < stage_end; };
    const int64_t R = p.T * p.K;
    const int64_t rp = p.padded_rows;  // capacity of the padded buffers
    const int32_t D = p.D, F = p.F, E = p.E;
    RoutingBuffers b{};
    b.ids = p.ids;
    b.R = R;
    b.E = E;
    b.nblk = p.nblk;
    b.block_counts = p.block_counts;
    b.block_bases = p.block_bases;
    b.counts = p.counts;
    b.offsets = p.offsets;
    b.perm = p.perm;
    b.inv = p.inv;
    b.status = p.status;
    moe_status_t st = MOE_OK;
    if (run(MOE_BWD_STAGE_DISPATCH)) {
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream) != cudaSuccess ||
        cudaMemsetAsync(p.pperm, 0xff, sizeof(int32_t) * rp, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if ((st = launch_routing(b, stream)) != MOE_OK) return st;
    if (launch_pdl(k_pad_tiles, dim3(1), dim3(1024), 0, stream, static_cast<const int32_t*>(p.counts), E, p.pmt) !=
            cudaSuccess ||
        launch_pdl(k_pad_rows, dim3(grid_for(R, 256, p.sm_count)), dim3(256), 0, stream, p.ids,
                   static_cast<const int32_t*>(p.inv), static_cast<const int32_t*>(p.offsets),
                   static_cast<const int32_t*>(p.pmt), R, E, p.pperm, p.pinv) != cudaSuccess ||
        launch_pdl(k_gather_bwd, dim3(grid_for(rp + p.T * ceil_div(D / 8, kGatherChunkVec), 8, p.sm_count)),
                   dim3(256), 0, stream, static_cast<const uint4*>(p.x), static_cast<const uint4*>(p.dout),
                   static_cast<const int32_t*>(p.pperm), static_cast<const int32_t*>(p.pinv),
                   static_cast<const int32_t*>(p.pmt), E, p.K, p.T, D / 8, static_cast<uint4*>(p.xpp),
                   static_cast<uint4*>(p.dop)) != cudaSuccess)
        return MOE_ERR_CUDA;
    }

    GemmArgs a{};
    a.pmt = p.pmt;
    a.pperm = p.pperm;
    a.E = E;
    a.D = D;
    a.F = F;
    a.scores = p.scores;
    a.scores_bf16 = p.scores_dtype == MOE_SCORES_BF16 ? 1 : 0;
    a.status = p.status;
    const int64_t max_row_tiles = ceil_div(rp, kPadRows);
    CUtensorMap ta, tb;

    // recompute: GU = [g | u], HS = s h
    if (run(MOE_BWD_STAGE_RECOMPUTE)) {
    if (!make_tmap(&ta, p.xpp, D, rp, kBK, kBM) || !make_tmap(&tb, p.w13, D, static_cast<uint64_t>(E) * 2 * F, kBK, kBN1))
        return MOE_ERR_CUDA;
    a.kblocks = D / kBK;
    a.out0 = static_cast<__nv_bfloat16*>(p.gu);
    a.out1 = static_cast<__nv_bfloat16*>(p.hs);
    if ((st = launch_gemm<BwdRecompute>(ta, tb, a, sm_count_grid(max_row_tiles * ceil_div(F, kBN1), p.sm_count),
                                        stream)) != MOE_OK)
        return st;
    }

    // dgrad of the down projection + SwiGLU backward
    if (run(MOE_BWD_STAGE_DGRAD_DOWN)) {
    if (!make_tmap(&ta, p.dop, D, rp, kBK, kBM) || !make_tmap(&tb, p.w2, F, static_cast<uint64_t>(E) * D, 64, kBK))
        return MOE_ERR_CUDA;
    a.kblocks = D / kBK;
    a.in0 = static_cast<const __nv_bfloat16*>(p.gu);
    a.out0 = static_cast<__nv_bfloat16*>(p.dgu);
    a.fout = p.partial;
    if ((st = launch_gemm<BwdDgradDown>(ta, tb, a, sm_count_grid(max_row_tiles * ceil_div(F, kBN2), p.sm_count),
                                        stream)) != MOE_OK)
        return st;
    }

    // dgrad of gate/up
    if (run(MOE_BWD_STAGE_DGRAD_GATE_UP)) {
    if (!make_tmap(&ta, p.dgu, 2ull * F, rp, kBK, kBM) ||
        !make_tmap(&tb, p.w13, D, static_cast<uint64_t>(E) * 2 * F, 64, kBK))
        return MOE_ERR_CUDA;
    a.kblocks = 2 * F / kBK;
    a.out0 = static_cast<__nv_bfloat16*>(p.dxp);
    if ((st = launch_gemm<BwdDgradGateUp>(ta, tb, a, sm_count_grid(max_row_tiles * ceil_div(D, kBN2), p.sm_count),
                                          stream)) != MOE_OK)
        return st;
    }

    // wgrad of W2: dW2[e] [D, F] = DOP_e^T HS_e
    if (run(MOE_BWD_STAGE_WGRAD_DOWN)) {
    if (!make_tmap(&ta, p.dop, D, rp, 64, kBK) || !make_tmap(&tb, p.hs, F, rp, 64, kBK)) return MOE_ERR_CUDA;
    a.mdim = D;
    a.ndim = F;
    a.mtiles = static_cast<int32_t>(ceil_div(D, kBM));
    a.ntiles = static_cast<int32_t>(ceil_div(F, kBRows));
    a.out0 = static_cast<__nv_bfloat16*>(p.dw2);
    if ((st = launch_gemm<BwdWgrad>(ta, tb, a,
                                    sm_count_grid(static_cast<int64_t>(E) * a.mtiles * a.ntiles, p.sm_count),
                                    stream)) != MOE_OK)
        return st;
    }

    // wgrad of w13: dW13[e] [2F, D] = DGU_e^T XPP_e
    if (run(MOE_BWD_STAGE_WGRAD_GATE_UP)) {
    if (!make_tmap(&ta, p.dgu, 2ull * F, rp, 64, kBK) || !make_tmap(&tb, p.xpp, D, rp, 64, kBK)) return MOE_ERR_CUDA;
    a.mdim = 2 * F;
    a.ndim = D;
    a.mtiles = static_cast<int32_t>(ceil_div(2 * F, kBM));
    a.ntiles = static_cast<int32_t>(ceil_div(D, kBRows));
    a.out0 = static_cast<__nv_bfloat16*>(p.dw13);
    if ((st = launch_gemm<BwdWgrad>(ta, tb, a,
                                    sm_count_grid(static_cast<int64_t>(E) * a.mtiles * a.ntiles, p.sm_count),
                                    stream)) != MOE_OK)
        return st;
    }

    if (!run(MOE_BWD_STAGE_REDUCE)) return MOE_OK;
    if (launch_pdl(k_dscores, dim3(grid_for(R, 256, p.sm_count)), dim3(256), 0, stream,
                   static_cast<const int32_t*>(p.pinv), static_cast<const float*>(p.partial), R,
                   static_cast<int32_t>(ceil_div(F, kBN2)), p.dscores) != cudaSuccess ||
        launch_pdl(k_dx_combine, dim3(grid_for(p.T * (D / 8), 256, p.sm_count)), dim3(256), 0, stream,
                   static_cast<const uint4*>(p.dxp), static_cast<const int32_t*>(p.pinv), p.T, p.K, D / 8,
                   static_cast<uint4*>(p.dx)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace moe
