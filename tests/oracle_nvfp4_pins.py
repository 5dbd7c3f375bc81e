"""Pins of the oracle's NVFP4 path: checks against things other than the oracle itself.

The format read for the pages' NVFP4 (Dist-MoE 0.1.0, "Choose a precision and pipeline / NVFP4")
is NVIDIA's published NVFP4: E2M1 elements in blocks of 16, a UE4M3 block scale
S = E4M3(amax / (6 G)), an fp32 tensor scale G (amax / 2688 for a weight; given for activations),
elements E2M1(v / (S G)), with the fp32 steps fixed (t = 6 G, b = amax / t, r = 1 / (S G), v * r).

What pins what:
  * E2M1 codes -- a brute-force search over the eight E2M1 magnitudes (nearest, ties to the even
    mantissa bit, saturating at 6), on blocks with ties, saturation, zeros and -0;
  * block scales -- a brute-force search over all finite E4M3 values (ties to even), run on b
    evaluated with numpy's IEEE float32 arithmetic; the S = 0 and saturated cases;
  * the weight tensor scale -- its closed form amax / 2688 and the all-zero case;
  * three blocks worked out by hand in ``golden/nvfp4_blocks.txt``;
  * the NVFP4 forward -- a float64 brute force over ALL experts with a dense [T,E] score matrix
    and its own quantizer, exact invariants (token permutation, power-of-two scaling of w2,
    zero-score pairs, thread count) and its distance to the bf16 forward.
"""

from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from common import bf16_bits, bits_to_f64, max_rel_err
from oracle_mx_pins import nearest_e4m3
from oracle_pins import GOLDEN, small_problem

NV_FP32_TOL = 1e-5
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E4M3_POS = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
f32 = np.float32


def nearest_e2m1(v) -> np.ndarray:
    """Brute force: nearest E2M1 code, ties to the even code (= even mantissa bit), sign kept."""
    v = np.asarray(v, np.float64).reshape(-1)
    a = np.abs(v)
    dist = np.abs(a[:, None] - E2M1_MAGNITUDES[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    first = cand.argmax(axis=1)
    two = cand.sum(axis=1) > 1
    code = np.where(two & (first % 2 == 1), first + 1, first)
    return np.where(np.signbit(v), code | 8, code).astype(np.uint8)


def e2m1_values(codes) -> np.ndarray:
    c = np.asarray(codes, np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def reference_quantize(vals32: np.ndarray, G: float):
    """Independent block quantizer: the reading's fp32 steps in numpy float32, every rounding to a
    format by brute-force search. vals32: float32 [nblocks, 16]. Returns (codes, scale codes)."""
    G = f32(G)
    amax = np.abs(vals32).max(axis=1).astype(f32)
    b = (amax / (f32(6.0) * G)).astype(f32)
    s = nearest_e4m3(b.astype(np.float64)) & 0x7F
    S = E4M3_POS[s].astype(f32)
    codes = np.zeros(vals32.shape, np.uint8)
    nz = S > 0
    r = (f32(1.0) / (S[nz] * G)).astype(f32)
    y = (vals32[nz] * r[:, None]).astype(f32)
    codes[nz] = nearest_e2m1(y.astype(np.float64)).reshape(y.shape)
    return codes, s.astype(np.uint8)


def random_blocks(seed: int, n: int) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(n, 16, generator=g, dtype=torch.float64)
    v *= torch.exp2(torch.randint(-12, 12, (n, 1), generator=g).double())
    q = n // 4
    v[:q] = torch.randint(-13, 14, (q, 16), generator=g).double() * 0.25  # exact ties at S G = 1 style
    v[q] = 0.0
    v[q + 1] = -0.0
    v[q + 2, :] = 1e-4
    v[q + 2, 3] = 50.0  # a spike
    return bf16_bits(v.to(torch.bfloat16))


def check_nvfp4_codes_and_scales_vs_brute_force(lib=None):
    for seed, G in ((31, 2.0 ** -4), (32, 0.0123), (33, 1.0), (34, 3.7e-5)):
        bits = random_blocks(seed, 200)
        codes, scales = oracle.nvfp4_quantize_rows(bits.reshape(20, -1), G, lib=lib)
        vals = bits_to_f64(bits).reshape(-1, 16).astype(f32)
        ref_codes, ref_scales = reference_quantize(vals, G)
        assert np.array_equal(scales.reshape(-1), ref_scales), (seed, G)
        assert np.array_equal(codes.reshape(-1, 16), ref_codes), (seed, G)


def check_nvfp4_weight_scale(lib=None):
    g = torch.Generator().manual_seed(35)
    w = (torch.randn(3, 64, generator=g) * 0.05).to(torch.bfloat16)
    bits = bf16_bits(w)
    amax = f32(np.abs(bits_to_f64(bits)).max())
    assert oracle.nvfp4_weight_scale(bits, lib=lib) == float(amax / f32(2688.0))
    assert oracle.nvfp4_weight_scale(np.zeros(64, np.uint16), lib=lib) == 1.0
    # the block holding the tensor's largest magnitude gets the largest scale code, 448
    codes, scales, G = oracle.nvfp4_prepare(bits, lib=lib)
    assert scales.max() == 0x7E


def read_nv_golden() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "nvfp4_blocks.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            if key.endswith("_values"):
                out[key] = np.array([float.fromhex(v) for v in vals], np.float64)
            else:
                out[key] = np.array([int(v, 16) for v in vals], np.uint8)
    return out


def check_nvfp4_golden_blocks(lib=None):
    gold = read_nv_golden()
    for blk in "ABC":
        bits = bf16_bits(torch.from_numpy(gold[f"{blk}_values"]).to(torch.bfloat16))
        assert np.array_equal(bits_to_f64(bits), gold[f"{blk}_values"]), blk
        codes, scales = oracle.nvfp4_quantize_rows(bits.reshape(1, 16), 2.0 ** -4, lib=lib)
        assert np.array_equal(scales.reshape(-1), gold[f"{blk}_scale"]), (blk, scales)
        assert np.array_equal(codes.reshape(-1), gold[f"{blk}_codes"]), (blk, codes)


# ---------------------------------------------------------------------------------- forward

ACT_GX = 2.0 ** -9  # activation tensor scales of the pins (x ~ N(0,1), |x| < 6 * 448 * 2^-9 = 5.25)
ACT_GH = 2.0 ** -9


def nv_problem(T, D, F, E, K, seed, **kw):
    p = small_problem(T, D, F, E, K, seed, **kw)
    p["w13_nv"] = oracle.nvfp4_prepare(p["w13"])
    p["w2_nv"] = oracle.nvfp4_prepare(p["w2"])
    return p


def run_nv(p, lib=None, gx=ACT_GX, gh=ACT_GH, **kw):
    w13 = oracle.nvfp4_prepare(p["w13"], lib=lib) if lib is not None else p["w13_nv"]
    w2 = oracle.nvfp4_prepare(p["w2"], lib=lib) if lib is not None else p["w2_nv"]
    return oracle.routed_experts_nvfp4(p["x"], p["ids"], p["scores"], w13, w2, gx, gh, lib=lib, **kw)


def nv_quantize_f64(v: np.ndarray, G: float):
    """Dequantized float64 values of the independent quantizer, plus a per-block ambiguity flag:
    b within 1e-5 of an E4M3 rounding boundary or an element within 1e-5 of an E2M1 one."""
    shape = v.shape
    blocks = np.asarray(v, np.float64).reshape(-1, 16)
    vals32 = blocks.astype(f32)
    codes, s = reference_quantize(vals32, G)
    S = E4M3_POS[s]
    deq = e2m1_values(codes) * S[:, None] * f32(G)
    # ambiguity of the element roundings: |y| close to a midpoint of the E2M1 grid
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.abs(blocks) / (S[:, None] * G)
    near = np.zeros(blocks.shape[0], bool)
    ok = S > 0
    near[ok] = (np.abs(y[ok][:, :, None] - mids[None, None, :]) <= 1e-5 * np.maximum(y[ok][:, :, None], 1)).any(axis=(1, 2))
    # ambiguity of the scale: b close to a midpoint of consecutive E4M3 values
    b = np.abs(blocks).max(axis=1) / (6 * G)
    e4 = np.sort(E4M3_POS)
    mid4 = (e4[1:] + e4[:-1]) / 2
    near |= (np.abs(b[:, None] - mid4[None, :]) <= 1e-5 * np.maximum(b[:, None], 1e-30)).any(axis=1)
    return deq.reshape(shape), near.reshape(shape[:-1] + (shape[-1] // 16,))


def nv_brute_force_f64(p, E, gx=ACT_GX, gh=ACT_GH):
    x, _ = nv_quantize_f64(bits_to_f64(p["x"]), gx)
    w13, _ = nv_quantize_f64(bits_to_f64(p["w13"]), oracle.nvfp4_weight_scale(p["w13"]))
    w2, _ = nv_quantize_f64(bits_to_f64(p["w2"]), oracle.nvfp4_weight_scale(p["w2"]))
    gate = np.einsum("efd,td->tef", w13[:, 0], x)
    up = np.einsum("efd,td->tef", w13[:, 1], x)
    h = gate / (1.0 + np.exp(-gate)) * up
    hq, amb = nv_quantize_f64(h, gh)
    y_all = np.einsum("edf,tef->ted", w2, hq)
    T, K = p["ids"].shape
    S = np.zeros((T, E))
    used = np.zeros((T, E), bool)
    for t in range(T):
        for k in range(K):
            e = int(p["ids"][t, k])
            if 0 <= e < E:
                S[t, e] += float(p["scores"][t, k])
                used[t, e] = True
    token_ok = ~(amb.any(axis=2) & used).any(axis=1)
    return np.einsum("te,ted->td", S, y_all), token_ok


def check_nvfp4_brute_force(lib=None):
    cases = [
        dict(T=9, D=64, F=96, E=5, K=3, seed=41),
        dict(T=17, D=96, F=64, E=8, K=2, seed=42, dup=True, invalid_frac=0.2, zero_frac=0.2),
        dict(T=6, D=32, F=32, E=1, K=3, seed=43, dup=True),
        dict(T=12, D=64, F=128, E=4, K=4, seed=44),
    ]
    for c in cases:
        p = nv_problem(**c)
        got = run_nv(p, lib=lib)
        ref, ok = nv_brute_force_f64(p, c["E"])
        assert ok.sum() >= max(1, len(ok) // 2), (c, ok)
        err = max_rel_err(got[ok], ref[ok])
        assert err <= NV_FP32_TOL, (c, err)


def check_nvfp4_token_permutation(lib=None):
    p = nv_problem(T=11, D=64, F=64, E=6, K=3, seed=45)
    base = run_nv(p, lib=lib)
    perm = np.random.default_rng(6).permutation(11)
    q = dict(p, x=p["x"][perm], ids=p["ids"][perm], scores=p["scores"][perm])
    assert np.array_equal(run_nv(q, lib=lib), base[perm])


def check_nvfp4_w2_power_of_two(lib=None):
    # w2 * 4: the tensor scale is 4x, every code and block scale the same, so out is exactly 4x
    p = nv_problem(T=7, D=64, F=64, E=4, K=2, seed=46)
    base = run_nv(p, lib=lib)
    w2x4 = bf16_bits(torch.from_numpy(bits_to_f64(p["w2"]) * 4.0).to(torch.bfloat16))
    q = dict(p, w2=w2x4, w2_nv=oracle.nvfp4_prepare(w2x4))
    assert np.array_equal(run_nv(q, lib=lib), base * 4.0)


def check_nvfp4_zero_score_pairs(lib=None):
    p = nv_problem(T=10, D=32, F=64, E=5, K=3, seed=47)
    s = p["scores"].copy()
    s[:, 2] = 0.0
    ids = p["ids"].copy()
    ids[:, 2] = -1
    assert np.array_equal(run_nv(dict(p, scores=s), lib=lib), run_nv(dict(p, ids=ids), lib=lib))


def check_nvfp4_thread_count(lib=None):
    p = nv_problem(T=13, D=64, F=32, E=4, K=2, seed=48)
    assert np.array_equal(run_nv(p, lib=lib, nthreads=1), run_nv(p, lib=lib, nthreads=4))


def check_nvfp4_near_bf16(lib=None):
    # E2M1 keeps one mantissa bit: a relative rounding error of up to 1/6 per element (RMS about
    # 7 % for values spread over the grid); four operands rounded once compound to ~15-25 % RMS
    p = nv_problem(T=16, D=128, F=128, E=4, K=2, seed=49)
    nv = run_nv(p, lib=lib)
    bf = oracle.routed_experts(p["x"], p["ids"], p["scores"], p["w13"], p["w2"])
    rms = float(np.linalg.norm(nv - bf) / np.linalg.norm(bf))
    assert 0.05 < rms < 0.4, rms


NV_PINS = [
    check_nvfp4_codes_and_scales_vs_brute_force,
    check_nvfp4_weight_scale,
    check_nvfp4_golden_blocks,
    check_nvfp4_brute_force,
    check_nvfp4_token_permutation,
    check_nvfp4_w2_power_of_two,
    check_nvfp4_zero_score_pairs,
    check_nvfp4_thread_count,
    check_nvfp4_near_bf16,
]
