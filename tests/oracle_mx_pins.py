"""Pins of the oracle's MXFP8 path: checks against things other than the oracle itself.

The format read for the pages' MXFP8_E4M3 (Dist-MoE 0.1.0, "Choose a precision and pipeline /
MXFP8") is the OCP Microscaling (MX) format v1.0: blocks of 32 along the contraction axis, a
shared UE8M0 power-of-two scale 2^e with e = floor(log2(max|v|)) - 8, E4M3 elements rounded to
nearest, ties to even, saturating at 448.

What pins what:
  * E4M3 element codes -- a brute-force search over all 254 finite E4M3 values (nearest value,
    ties to the even code), and torch's own float8_e4m3fn cast (a library routine), on random
    blocks spanning normal, subnormal, tie and saturating cases;
  * the shared scale -- its defining property (2^8 <= max|v| * 2^-e < 2^9 unless clamped) and
    the all-zero and clamped-tiny special cases;
  * four blocks worked out by hand in ``golden/mx_e4m3_blocks.txt``;
  * exact round trips of blocks that are already MX numbers;
  * the MXFP8 forward -- a float64 brute force over ALL experts with a dense [T,E] score matrix
    and its own quantizer (the brute-force search), exact invariants (token permutation, a
    power-of-two scaling of w2, zero-score pairs, thread count) and its distance to the bf16
    forward (non-zero, and within the format's error).
Each check takes an optional ``lib`` so that ``test_oracle_mutants.py`` can run it on mutants.
"""

from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from common import bf16_bits, bits_to_f64, max_rel_err
from oracle_pins import GOLDEN, small_problem

MX_FP32_TOL = 1e-5

# every finite E4M3 magnitude, by code 0x00 .. 0x7E (ascending), from torch's float8 type
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = torch.from_numpy(_POS_CODES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def nearest_e4m3(v: np.ndarray) -> np.ndarray:
    """Brute force: the finite E4M3 code nearest to each value, ties to the even code, sign kept."""
    v = np.asarray(v, np.float64).reshape(-1)
    a = np.abs(v)
    dist = np.abs(a[:, None] - _POS_VALUES[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    first = cand.argmax(axis=1)
    two = cand.sum(axis=1) > 1
    code = np.where(two & (first % 2 == 1), first + 1, first).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    """torch's float8_e4m3fn cast (round to nearest even) of values clamped to +-448."""
    t = torch.from_numpy(np.clip(np.asarray(v, np.float64), -448.0, 448.0).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(np.shape(v))


def e4m3_value(codes) -> np.ndarray:
    c = np.asarray(codes, np.uint8)
    return torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def block_values(bits: np.ndarray) -> np.ndarray:
    return bits_to_f64(np.asarray(bits, np.uint16)).reshape(-1, 32)


def random_blocks(seed: int, nblocks: int) -> np.ndarray:
    """bf16 bit patterns [nblocks, 32]: random magnitudes over a wide exponent range, plus blocks
    with exact E4M3 ties, spikes, zeros, negative zeros and subnormals."""
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(nblocks, 32, generator=g, dtype=torch.float64)
    v *= torch.exp2(torch.randint(-30, 30, (nblocks, 1), generator=g).double())
    # a quarter of the blocks hold values with at most 5 significant bits (frequent exact ties)
    q = nblocks // 4
    coarse = torch.randint(-31, 32, (q, 32), generator=g).double()
    v[:q] = coarse * torch.exp2(torch.randint(-12, 12, (q, 1), generator=g).double())
    v[q] = 0.0
    v[q + 1] = -0.0
    v[q + 2, :] = 1e-3
    v[q + 2, 5] = 300.0  # one spike: everything else near the bottom of the range
    v[q + 3] = torch.randn(32, generator=g, dtype=torch.float64) * 2.0 ** -128  # bf16 subnormals
    v[q + 4] = torch.randn(32, generator=g, dtype=torch.float64) * 2.0 ** 120
    return bf16_bits(v.to(torch.bfloat16))


def _scaled(vals: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return np.ldexp(vals, -(scales.astype(np.int64) - 127)[:, None])


def check_e4m3_values_vs_torch(lib=None):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_values(codes), e4m3_value(codes))


def check_mx_codes_vs_brute_force(lib=None):
    bits = random_blocks(11, 400)
    codes, scales = oracle.mx_quantize_rows(bits.reshape(20, -1), lib=lib)
    vals = block_values(bits)
    scaled = _scaled(vals, scales.reshape(-1))
    assert np.array_equal(codes.reshape(-1), nearest_e4m3(scaled))


def check_mx_codes_vs_torch_cast(lib=None):
    bits = random_blocks(12, 400)
    codes, scales = oracle.mx_quantize_rows(bits.reshape(40, -1), lib=lib)
    scaled = _scaled(block_values(bits), scales.reshape(-1))
    assert np.array_equal(codes.reshape(-1, 32), torch_e4m3(scaled))


def check_mx_scale_rule(lib=None):
    bits = random_blocks(13, 400)
    codes, scales = oracle.mx_quantize_rows(bits.reshape(10, -1), lib=lib)
    vals = block_values(bits)
    e = scales.reshape(-1).astype(np.int64) - 127
    amax = np.abs(vals).max(axis=1)
    for b in range(vals.shape[0]):
        if amax[b] == 0:
            assert e[b] == -127 and np.all((codes.reshape(-1, 32)[b] & 0x7F) == 0), b
            continue
        top = math.ldexp(amax[b], -int(e[b]))
        if e[b] == -127:
            assert top < 512.0, b  # clamped from below: the block is tiny
        else:
            assert 256.0 <= top < 512.0, (b, amax[b], e[b])


def read_mx_golden() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "mx_e4m3_blocks.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            if key.endswith("_values"):
                out[key] = np.array([float.fromhex(v) for v in vals], np.float64)
            else:
                out[key] = np.array([int(v, 16) for v in vals], np.uint8)
    return out


def check_mx_golden_blocks(lib=None):
    gold = read_mx_golden()
    for blk in "ABCD":
        v = torch.from_numpy(gold[f"{blk}_values"])
        bits = bf16_bits(v.to(torch.bfloat16))
        assert np.array_equal(bits_to_f64(bits), gold[f"{blk}_values"]), blk  # exact bf16 inputs
        codes, scales = oracle.mx_quantize_rows(bits.reshape(1, 32), lib=lib)
        assert np.array_equal(scales.reshape(-1), gold[f"{blk}_scale"]), (blk, scales)
        assert np.array_equal(codes.reshape(-1), gold[f"{blk}_codes"]), (blk, codes)


def check_mx_roundtrip_exact(lib=None):
    # blocks that are MX numbers already: random finite codes, the first one with magnitude in
    # [256, 448] (so the block's max sets e exactly), times 2^e; quantizing gives them back.
    rng = np.random.default_rng(14)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    big = np.array([c for c in finite if 256 <= abs(e4m3_value(np.array([c]))[0]) <= 448], np.uint8)
    codes = rng.choice(finite, size=(64, 32)).astype(np.uint8)
    codes[:, 0] = rng.choice(big, size=64)
    e = rng.integers(-40, 40, size=64)
    vals = np.ldexp(e4m3_value(codes), e[:, None])
    bits = bf16_bits(torch.from_numpy(vals).to(torch.bfloat16))
    assert np.array_equal(bits_to_f64(bits), vals)
    got_codes, got_scales = oracle.mx_quantize_rows(bits.reshape(8, -1), lib=lib)
    assert np.array_equal(got_scales.reshape(-1).astype(np.int64), e + 127)
    assert np.array_equal(got_codes.reshape(64, 32), codes)  # -0 keeps its sign through bf16


# ---------------------------------------------------------------------------------- forward

def mx_quantize_f64(v: np.ndarray):
    """The independent quantizer of the brute force: e from the scale rule, codes by search.
    Returns (dequantized values, ambiguous mask per block): a block is ambiguous when its max is
    within 1e-6 of a power of two or an element is within 1e-6 of a rounding midpoint, where an
    fp32 evaluation of the same value may legitimately round the other way."""
    shape = v.shape
    blocks = np.asarray(v, np.float64).reshape(-1, 32)
    amax = np.abs(blocks).max(axis=1)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.clip(np.where(amax > 0, ex - 1 - 8, -127), -127, 127)
    scaled = np.ldexp(blocks, -e[:, None])
    codes = nearest_e4m3(scaled).reshape(blocks.shape)
    deq = np.ldexp(e4m3_value(codes), e[:, None])
    # ambiguity: distance to the nearest rounding midpoint, relative to the value
    a = np.abs(scaled)
    _, aex = np.frexp(np.where(a > 0, a, 1.0))
    k = np.maximum(aex - 1, -6)
    spacing = np.ldexp(1.0, k - 3)
    frac = a / spacing - np.floor(a / spacing)
    near_mid = np.abs(frac - 0.5) * spacing <= 1e-6 * np.maximum(a, 2.0 ** -9)
    mant, _ = np.frexp(np.where(amax > 0, amax, 1.0))
    near_pow2 = (np.abs(mant - 0.5) <= 1e-6) | (np.abs(mant - 1.0) <= 1e-6)
    ambiguous = near_mid.any(axis=1) | (near_pow2 & (amax > 0))
    return deq.reshape(shape), ambiguous.reshape(shape[:-1] + (shape[-1] // 32,))


def mx_problem(T, D, F, E, K, seed, **kw):
    p = small_problem(T, D, F, E, K, seed, **kw)
    p["w13_mx"] = oracle.mx_quantize_rows(p["w13"])
    p["w2_mx"] = oracle.mx_quantize_rows(p["w2"])
    return p


def run_mx(p, lib=None, **kw):
    w13_mx = oracle.mx_quantize_rows(p["w13"], lib=lib) if lib is not None else p["w13_mx"]
    w2_mx = oracle.mx_quantize_rows(p["w2"], lib=lib) if lib is not None else p["w2_mx"]
    return oracle.routed_experts_mxfp8(p["x"], p["ids"], p["scores"], w13_mx, w2_mx, lib=lib, **kw)


def mx_brute_force_f64(p, E):
    """Every expert on every token in float64 with the independent quantizer, contracted with a
    dense [T,E] score matrix. Returns (out [T,D], token_ok [T]): token_ok is False for tokens with
    an ambiguous quantization of h for one of their experts."""
    x, _ = mx_quantize_f64(bits_to_f64(p["x"]))
    w13, _ = mx_quantize_f64(bits_to_f64(p["w13"]))
    w2, _ = mx_quantize_f64(bits_to_f64(p["w2"]))
    gate = np.einsum("efd,td->tef", w13[:, 0], x)
    up = np.einsum("efd,td->tef", w13[:, 1], x)
    h = gate / (1.0 + np.exp(-gate)) * up
    hq, amb = mx_quantize_f64(h)  # [T,E,F], [T,E,F/32]
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


def check_mxfp8_brute_force(lib=None):
    cases = [
        dict(T=9, D=64, F=96, E=5, K=3, seed=21),
        dict(T=17, D=96, F=64, E=8, K=2, seed=22, dup=True, invalid_frac=0.2, zero_frac=0.2),
        dict(T=6, D=32, F=32, E=1, K=3, seed=23, dup=True),
        dict(T=12, D=64, F=128, E=4, K=4, seed=24),  # K = E
    ]
    for c in cases:
        p = mx_problem(**c)
        got = run_mx(p, lib=lib)
        ref, ok = mx_brute_force_f64(p, c["E"])
        assert ok.sum() >= max(1, len(ok) // 2), (c, ok)
        err = max_rel_err(got[ok], ref[ok])
        assert err <= MX_FP32_TOL, (c, err)


def check_mxfp8_token_permutation(lib=None):
    p = mx_problem(T=11, D=64, F=64, E=6, K=3, seed=25)
    base = run_mx(p, lib=lib)
    perm = np.random.default_rng(5).permutation(11)
    q = dict(p, x=p["x"][perm], ids=p["ids"][perm], scores=p["scores"][perm])
    assert np.array_equal(run_mx(q, lib=lib), base[perm])


def check_mxfp8_w2_power_of_two(lib=None):
    # w2 * 8 keeps every E4M3 code and raises every w2 scale by 3: out is exactly 8x
    p = mx_problem(T=7, D=64, F=64, E=4, K=2, seed=26)
    base = run_mx(p, lib=lib)
    w2x8 = bf16_bits(torch.from_numpy(bits_to_f64(p["w2"]) * 8.0).to(torch.bfloat16))
    q = dict(p, w2=w2x8, w2_mx=oracle.mx_quantize_rows(w2x8))
    assert np.array_equal(run_mx(q, lib=lib), base * 8.0)


def check_mxfp8_zero_score_pairs(lib=None):
    p = mx_problem(T=10, D=32, F=64, E=5, K=3, seed=27)
    s = p["scores"].copy()
    s[:, 1] = 0.0
    ids = p["ids"].copy()
    ids[:, 1] = -1  # the same pairs dropped by an invalid id
    a = run_mx(dict(p, scores=s), lib=lib)
    b = run_mx(dict(p, ids=ids), lib=lib)
    assert np.array_equal(a, b)


def check_mxfp8_thread_count(lib=None):
    p = mx_problem(T=13, D=64, F=32, E=4, K=2, seed=28)
    assert np.array_equal(run_mx(p, lib=lib, nthreads=1), run_mx(p, lib=lib, nthreads=5))


def check_mxfp8_near_bf16(lib=None):
    # The block-scaled result differs from the bf16 one (something was quantized) by about the
    # format's rounding: an E4M3 element carries a uniform relative error of up to 2^-4 (RMS
    # 2^-4/sqrt(3) = 3.6 %); x, w13, h and w2 are each rounded once, which compounds to ~8 % RMS.
    p = mx_problem(T=16, D=128, F=128, E=4, K=2, seed=29)
    mx = run_mx(p, lib=lib)
    bf = oracle.routed_experts(p["x"], p["ids"], p["scores"], p["w13"], p["w2"])
    rms = float(np.linalg.norm(mx - bf) / np.linalg.norm(bf))
    assert 0.02 < rms < 0.2, rms


MX_PINS = [
    check_e4m3_values_vs_torch,
    check_mx_codes_vs_brute_force,
    check_mx_codes_vs_torch_cast,
    check_mx_scale_rule,
    check_mx_golden_blocks,
    check_mx_roundtrip_exact,
    check_mxfp8_brute_force,
    check_mxfp8_token_permutation,
    check_mxfp8_w2_power_of_two,
    check_mxfp8_zero_score_pairs,
    check_mxfp8_thread_count,
    check_mxfp8_near_bf16,
]
