"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each check takes an optional ``lib`` (a loaded oracle library) so that
``test_oracle_mutants.py`` can run the same checks against copies of the oracle with a planted
mistake; every check raises ``AssertionError`` when it fails.

What pins what:
  * routing -- numpy's stable argsort and bincount (an independent sort); structural invariants;
    the round-robin closed form and the hand-derived fixture in ``golden/``.
  * output -- a dense SwiGLU MLP computed by torch in float64 (K=1, one expert, score 1);
    a brute-force float64 evaluation over ALL experts contracted with a dense [T,E] score
    matrix (a different algorithm from the per-token loop); a scalar closed form evaluated with
    Python's math module; exact invariants (token permutation, power-of-two score scaling,
    zero-score pairs, thread count).
  * error bound -- the fp32 oracle agrees with the float64 brute force to 1e-5 of max|ref|.
"""

from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as Fnn

import oracle
from common import bf16_bits, bits_to_f64, max_rel_err

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ORACLE_FP32_TOL = 1e-5


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            out[key] = np.array([int(v) for v in vals], dtype=np.int64)
    return out


def small_problem(T, D, F, E, K, seed, invalid_frac=0.0, dup=False, zero_frac=0.0):
    """Random bf16 inputs for the pins (torch CPU generator, fixed seed)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, 2, F, D, generator=g) / math.sqrt(D)).to(torch.bfloat16)
    w2 = (torch.randn(E, D, F, generator=g) / math.sqrt(F)).to(torch.bfloat16)
    ids = torch.randint(0, E, (T, K), generator=g, dtype=torch.int32)
    if not dup and K <= E:
        ids = torch.rand(T, E, generator=g).topk(K, dim=1).indices.to(torch.int32)
    if invalid_frac > 0:
        m = torch.rand(T, K, generator=g) < invalid_frac
        bad = torch.where(torch.rand(T, K, generator=g) < 0.5, torch.full_like(ids, -1), torch.full_like(ids, E + 3))
        ids = torch.where(m, bad, ids)
    scores = torch.softmax(torch.randn(T, K, generator=g), dim=1)
    if zero_frac > 0:
        scores = torch.where(torch.rand(T, K, generator=g) < zero_frac, torch.zeros_like(scores), scores)
    return {
        "x": bf16_bits(x),
        "w13": bf16_bits(w13),
        "w2": bf16_bits(w2),
        "ids": ids.numpy().astype(np.int32),
        "scores": scores.numpy().astype(np.float32),
    }


def run_oracle(p, lib=None, **kw):
    return oracle.routed_experts(p["x"], p["ids"], p["scores"], p["w13"], p["w2"], lib=lib, **kw)


# ------------------------------------------------------------------------------------------ routing

def routing_reference(ids: np.ndarray, E: int) -> dict:
    """Independent routing: numpy bincount + stable argsort on the key (invalid ids -> E)."""
    flat = ids.reshape(-1).astype(np.int64)
    key = np.where((flat >= 0) & (flat < E), flat, E)
    counts = np.bincount(key, minlength=E + 1)[:E]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm = np.argsort(key, kind="stable")
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv, "n_invalid": int((key == E).sum())}


def check_routing_vs_stable_argsort(lib=None):
    rng = np.random.default_rng(7)
    cases = [(1, 1, 1), (0, 4, 2), (3, 5, 7), (33, 8, 2), (100, 64, 6), (257, 256, 8), (500, 3, 4)]
    for (T, E, K) in cases:
        ids = rng.integers(-2, E + 2, size=(T, K), dtype=np.int32)  # includes invalid ids and duplicates
        got = oracle.routing(ids, E, lib=lib)
        ref = routing_reference(ids, E)
        for key in ("counts", "offsets", "perm", "inv"):
            assert np.array_equal(got[key], ref[key]), (key, T, E, K)
        assert got["n_invalid"] == ref["n_invalid"]


def check_routing_invariants(lib=None):
    rng = np.random.default_rng(11)
    for (T, E, K) in [(64, 16, 4), (129, 7, 3), (1000, 256, 8)]:
        ids = rng.integers(0, E, size=(T, K), dtype=np.int32)
        r = oracle.routing(ids, E, lib=lib)
        R = T * K
        assert r["counts"].sum() == R and r["offsets"][E] == R and r["offsets"][0] == 0
        assert np.array_equal(np.sort(r["perm"]), np.arange(R))  # bijection
        assert np.array_equal(r["inv"][r["perm"]], np.arange(R))
        flat = ids.reshape(-1)
        keys = flat[r["perm"]]
        assert np.all(np.diff(keys) >= 0)  # expert-contiguous
        for e in range(E):
            seg = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)  # stable: ascending pair index inside a segment


def check_round_robin_golden(lib=None):
    g = read_golden("tiny_round_robin_routing.txt")
    T, K, E = int(g["T"][0]), int(g["K"][0]), int(g["E"][0])
    t = np.arange(T)[:, None]
    k = np.arange(K)[None, :]
    ids = ((t * K + k) % E).astype(np.int32)
    r = oracle.routing(ids, E, lib=lib)
    for key in ("counts", "offsets", "perm", "inv"):
        assert np.array_equal(r[key], g[key]), key


def check_round_robin_closed_form(lib=None):
    # Round robin (t*K + k) % E over T*K pairs gives exactly T*K/E per expert when E divides T*K.
    for (T, K, E) in [(16, 2, 8), (4096, 6, 64), (64, 8, 256), (96, 8, 256)]:
        ids = ((np.arange(T)[:, None] * K + np.arange(K)[None, :]) % E).astype(np.int32)
        r = oracle.routing(ids, E, lib=lib)
        if (T * K) % E == 0:
            assert np.all(r["counts"] == T * K // E)
        else:
            q = (T * K) // E
            assert np.all((r["counts"] == q) | (r["counts"] == q + 1))
            assert np.all(r["counts"][: (T * K) % E] == q + 1)


# ------------------------------------------------------------------------------------------- output

def _silu_mlp_f64(x, wg, wu, w2):
    """Dense SwiGLU MLP in float64 with torch's own SiLU: W2 (SiLU(Wg x) * (Wu x))."""
    xt = torch.from_numpy(x)
    h = Fnn.silu(Fnn.linear(xt, torch.from_numpy(wg))) * Fnn.linear(xt, torch.from_numpy(wu))
    return Fnn.linear(h, torch.from_numpy(w2)).numpy()


def check_dense_swiglu_special_case(lib=None):
    # K = 1, every token routed to expert 0 with score 1: the layer is a dense SwiGLU MLP.
    T, D, F, E = 24, 64, 96, 3
    p = small_problem(T, D, F, E, 1, seed=3)
    p["ids"][:] = 0
    p["scores"][:] = 1.0
    got = run_oracle(p, lib=lib)
    ref = _silu_mlp_f64(bits_to_f64(p["x"]), bits_to_f64(p["w13"][0, 0]), bits_to_f64(p["w13"][0, 1]),
                        bits_to_f64(p["w2"][0]))
    assert max_rel_err(got, ref) <= ORACLE_FP32_TOL, max_rel_err(got, ref)


def brute_force_all_experts_f64(p, E):
    """Every expert on every token (float64), contracted with a dense [T,E] score matrix."""
    x = torch.from_numpy(bits_to_f64(p["x"]))
    w13 = torch.from_numpy(bits_to_f64(p["w13"]))
    w2 = torch.from_numpy(bits_to_f64(p["w2"]))
    gate = torch.einsum("efd,td->tef", w13[:, 0], x)
    up = torch.einsum("efd,td->tef", w13[:, 1], x)
    y_all = torch.einsum("edf,tef->ted", w2, Fnn.silu(gate) * up)  # [T,E,D]
    T, K = p["ids"].shape
    S = np.zeros((T, E))
    for t in range(T):
        for k in range(K):
            e = int(p["ids"][t, k])
            if 0 <= e < E:
                S[t, e] += float(p["scores"][t, k])
    return torch.einsum("te,ted->td", torch.from_numpy(S), y_all).numpy()


def check_brute_force_dense(lib=None):
    cases = [
        dict(T=9, D=32, F=48, E=5, K=3, seed=1),
        dict(T=17, D=64, F=32, E=8, K=2, seed=2, dup=True, invalid_frac=0.2, zero_frac=0.2),
        dict(T=5, D=16, F=16, E=1, K=4, seed=4, dup=True),  # one expert, duplicates in every token
        dict(T=12, D=48, F=80, E=6, K=6, seed=5),  # K = E
    ]
    for c in cases:
        E = c["E"]
        p = small_problem(**c)
        got = run_oracle(p, lib=lib)
        ref = brute_force_all_experts_f64(p, E)
        err = max_rel_err(got, ref)
        assert err <= ORACLE_FP32_TOL, (c, err)


def check_scalar_closed_form(lib=None):
    # D = F = E = K = 1: out = s * w2 * SiLU(wg x) * (wu x), with SiLU(z) = z / (1 + e^-z).
    for (xv, wg, wu, w2v, s) in [(1.5, 0.75, -2.0, 0.5, 0.25), (-3.0, 1.25, 0.5, -1.0, 1.0), (0.0, 1.0, 1.0, 1.0, 1.0)]:
        to_bits = lambda v: bf16_bits(torch.tensor([v], dtype=torch.bfloat16))
        p = {
            "x": to_bits(xv).reshape(1, 1),
            "w13": np.concatenate([to_bits(wg), to_bits(wu)]).reshape(1, 2, 1, 1),
            "w2": to_bits(w2v).reshape(1, 1, 1),
            "ids": np.zeros((1, 1), np.int32),
            "scores": np.full((1, 1), s, np.float32),
        }
        g = wg * xv
        ref = s * w2v * (g / (1.0 + math.exp(-g))) * (wu * xv)
        got = float(run_oracle(p, lib=lib)[0, 0])
        assert abs(got - ref) <= 1e-6 * max(1.0, abs(ref)), (got, ref)


def check_token_permutation(lib=None):
    p = small_problem(T=20, D=32, F=32, E=6, K=3, seed=8)
    out = run_oracle(p, lib=lib)
    pi = np.random.default_rng(0).permutation(20)
    q = dict(p, x=p["x"][pi], ids=p["ids"][pi], scores=p["scores"][pi])
    assert np.array_equal(run_oracle(q, lib=lib), out[pi])


def check_score_scaling(lib=None):
    p = small_problem(T=10, D=32, F=48, E=4, K=2, seed=9)
    out = run_oracle(p, lib=lib)
    for c in (2.0, 0.25, 8.0):
        q = dict(p, scores=(p["scores"] * np.float32(c)).astype(np.float32))
        assert np.array_equal(run_oracle(q, lib=lib), out * np.float32(c))


def check_zero_score_pairs(lib=None):
    # A zero-score pair contributes nothing: same output as dropping the pair (column removed).
    p = small_problem(T=8, D=32, F=32, E=4, K=3, seed=10)
    p["scores"][:, 2] = 0.0
    q = dict(p, ids=np.ascontiguousarray(p["ids"][:, :2]), scores=np.ascontiguousarray(p["scores"][:, :2]))
    assert np.array_equal(run_oracle(p, lib=lib), run_oracle(q, lib=lib))
    # ... and the same as marking it with an invalid id
    r = dict(p, ids=p["ids"].copy())
    r["ids"][:, 2] = -1
    assert np.array_equal(run_oracle(p, lib=lib), run_oracle(r, lib=lib))


def check_bf16_scores(lib=None):
    p = small_problem(T=6, D=32, F=32, E=4, K=2, seed=12)
    sb = bf16_bits(torch.from_numpy(p["scores"]).to(torch.bfloat16))
    q = dict(p, scores=sb)
    r = dict(p, scores=bits_to_f64(sb).astype(np.float32))
    assert np.array_equal(run_oracle(q, lib=lib), run_oracle(r, lib=lib))


def check_round_h(lib=None):
    # round_h rounds SwiGLU's output to bf16 (nearest, ties to even) before W2; compare with a
    # float64 evaluation that rounds the same place with torch's bf16 cast.
    T, D, F, E = 7, 32, 64, 1
    p = small_problem(T, D, F, E, 1, seed=13)
    p["ids"][:] = 0
    p["scores"][:] = 1.0
    got = run_oracle(p, lib=lib, round_h=True)
    x = torch.from_numpy(bits_to_f64(p["x"]))
    wg, wu = (torch.from_numpy(bits_to_f64(p["w13"][0, i])) for i in (0, 1))
    h = (Fnn.silu(Fnn.linear(x, wg)) * Fnn.linear(x, wu)).float().to(torch.bfloat16).double()
    ref = Fnn.linear(h, torch.from_numpy(bits_to_f64(p["w2"][0]))).numpy()
    assert max_rel_err(got, ref) <= ORACLE_FP32_TOL


def check_thread_count_invariance(lib=None):
    p = small_problem(T=13, D=32, F=32, E=4, K=2, seed=14)
    a = run_oracle(p, lib=lib, nthreads=1)
    b = run_oracle(p, lib=lib, nthreads=5)
    assert np.array_equal(a, b)


ROUTING_PINS = [
    check_routing_vs_stable_argsort,
    check_routing_invariants,
    check_round_robin_golden,
    check_round_robin_closed_form,
]
OUTPUT_PINS = [
    check_dense_swiglu_special_case,
    check_brute_force_dense,
    check_scalar_closed_form,
    check_token_permutation,
    check_score_scaling,
    check_zero_score_pairs,
    check_bf16_scores,
    check_round_h,
    check_thread_count_invariance,
]
ALL_PINS = ROUTING_PINS + OUTPUT_PINS


# -------------------------------------------------------------------- RMSNorm post-processing

def run_rms(p, eps, lib=None):
    return oracle.routed_experts_rmsnorm(p["x"], p["ids"], p["scores"], p["w13"], p["w2"], eps, lib=lib)


def check_rmsnorm_vs_torch(lib=None):
    # every expert on every token in float64, torch's own rms_norm per (token, expert), contracted
    # with the dense score matrix
    for c in (dict(T=9, D=32, F=48, E=5, K=3, seed=31), dict(T=11, D=64, F=32, E=4, K=2, seed=32, dup=True,
                                                                 invalid_frac=0.2, zero_frac=0.2)):
        p = small_problem(**c)
        x = torch.from_numpy(bits_to_f64(p["x"]))
        w13 = torch.from_numpy(bits_to_f64(p["w13"]))
        w2 = torch.from_numpy(bits_to_f64(p["w2"]))
        h = Fnn.silu(torch.einsum("efd,td->tef", w13[:, 0], x)) * torch.einsum("efd,td->tef", w13[:, 1], x)
        y = torch.einsum("edf,tef->ted", w2, h)
        z = Fnn.rms_norm(y, (c["D"],), eps=1e-6)
        E = c["E"]
        S = np.zeros((c["T"], E))
        for t in range(c["T"]):
            for k in range(c["K"]):
                e = int(p["ids"][t, k])
                if 0 <= e < E:
                    S[t, e] += float(p["scores"][t, k])
        ref = torch.einsum("te,ted->td", torch.from_numpy(S), z).numpy()
        assert max_rel_err(run_rms(p, 1e-6, lib), ref) <= ORACLE_FP32_TOL


def check_rmsnorm_scale_invariance(lib=None):
    # with eps = 0 the normalised output does not depend on the scale of W2: x4 is exact in bf16
    # and in every fp32 step, so the outputs are bit-identical
    p = small_problem(T=10, D=32, F=32, E=3, K=2, seed=33)
    a = run_rms(p, 0.0, lib)
    w2 = torch.from_numpy(bits_to_f64(p["w2"])).float() * 4.0
    b = run_rms(dict(p, w2=bf16_bits(w2.to(torch.bfloat16))), 0.0, lib)
    assert np.array_equal(a, b)


def check_rmsnorm_scalar_sign(lib=None):
    # D = 1 and eps = 0: RMSNorm of a scalar is its sign, so out = sum_k s * sign(y_k)
    p = small_problem(T=6, D=1, F=8, E=3, K=2, seed=34)
    y = oracle.routed_experts(p["x"], p["ids"][:, :1].copy(), np.ones((6, 1), np.float32), p["w13"], p["w2"],
                              lib=lib)[:, 0]
    y2 = oracle.routed_experts(p["x"], p["ids"][:, 1:].copy(), np.ones((6, 1), np.float32), p["w13"], p["w2"],
                               lib=lib)[:, 0]
    ref = p["scores"][:, 0] * np.sign(y) + p["scores"][:, 1] * np.sign(y2)
    got = run_rms(p, 0.0, lib)[:, 0]
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-7)


OUTPUT_PINS += [check_rmsnorm_vs_torch, check_rmsnorm_scale_invariance, check_rmsnorm_scalar_sign]
ALL_PINS = ROUTING_PINS + OUTPUT_PINS
