"""Pins of the backward oracle, against things other than the oracle itself.

  * torch autograd in float64 through the dense brute-force formulation (every expert on every
    token, contracted with a dense [T,E] score matrix) -- a different algorithm differentiated by
    a library, covering duplicates, invalid ids and zero scores;
  * a scalar closed form (D = F = E = K = 1) differentiated by hand and evaluated with math;
  * exact invariants: linearity in the upstream gradient, zero-score pairs, thread count.
"""

from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as Fnn

import oracle
from common import bf16_bits, bits_to_f64, max_rel_err
from oracle_pins import small_problem

BWD_TOL = 2e-5


def run_bwd(p, dout, lib=None, **kw):
    return oracle.routed_experts_bwd(p["x"], p["ids"], p["scores"], p["w13"], p["w2"], dout, lib=lib, **kw)


def autograd_reference(p, dout):
    """float64 autograd through the dense all-experts formulation."""
    x = torch.from_numpy(bits_to_f64(p["x"])).requires_grad_()
    w13 = torch.from_numpy(bits_to_f64(p["w13"])).requires_grad_()
    w2 = torch.from_numpy(bits_to_f64(p["w2"])).requires_grad_()
    sc = torch.from_numpy(p["scores"].astype(np.float64)).requires_grad_()
    ids = torch.from_numpy(p["ids"].astype(np.int64))
    T, K = ids.shape
    E = w13.shape[0]
    valid = (ids >= 0) & (ids < E)
    onehot = Fnn.one_hot(torch.where(valid, ids, 0), E).double() * valid[..., None].double()  # [T,K,E]
    S = torch.einsum("tk,tke->te", sc, onehot)
    gate = torch.einsum("efd,td->tef", w13[:, 0], x)
    up = torch.einsum("efd,td->tef", w13[:, 1], x)
    y_all = torch.einsum("edf,tef->ted", w2, Fnn.silu(gate) * up)
    out = torch.einsum("te,ted->td", S, y_all)
    out.backward(torch.from_numpy(dout.astype(np.float64)))
    return {"dx": x.grad.numpy(), "dscores": sc.grad.numpy(), "dw13": w13.grad.numpy(), "dw2": w2.grad.numpy()}


def random_dout(T, D, seed):
    return torch.randn(T, D, generator=torch.Generator().manual_seed(seed)).numpy().astype(np.float32)


def check_bwd_vs_autograd(lib=None):
    cases = [
        dict(T=9, D=32, F=48, E=5, K=3, seed=21),
        dict(T=13, D=64, F=32, E=6, K=2, seed=22, dup=True, invalid_frac=0.2, zero_frac=0.2),
        dict(T=6, D=16, F=16, E=1, K=3, seed=23, dup=True),
    ]
    for c in cases:
        p = small_problem(**c)
        dout = random_dout(c["T"], c["D"], c["seed"])
        got = run_bwd(p, dout, lib=lib)
        ref = autograd_reference(p, dout)
        for key in ("dx", "dscores", "dw13", "dw2"):
            err = max_rel_err(got[key], ref[key])
            assert err <= BWD_TOL, (c, key, err)


def check_bwd_scalar_closed_form(lib=None):
    to_bits = lambda v: bf16_bits(torch.tensor([v], dtype=torch.bfloat16))
    for (xv, wg, wu, w2v, s, go) in [(1.5, 0.75, -2.0, 0.5, 0.25, 1.0), (-0.5, 1.25, 0.5, -1.0, 0.75, -2.0)]:
        p = {
            "x": to_bits(xv).reshape(1, 1),
            "w13": np.concatenate([to_bits(wg), to_bits(wu)]).reshape(1, 2, 1, 1),
            "w2": to_bits(w2v).reshape(1, 1, 1),
            "ids": np.zeros((1, 1), np.int32),
            "scores": np.full((1, 1), s, np.float32),
        }
        g, u = wg * xv, wu * xv
        sig = 1.0 / (1.0 + math.exp(-g))
        silu, dsilu = g * sig, sig * (1.0 + g * (1.0 - sig))
        ref = {
            "dx": go * s * w2v * (dsilu * wg * u + silu * wu),
            "dscores": go * w2v * silu * u,
            "dwg": go * s * w2v * dsilu * xv * u,
            "dwu": go * s * w2v * silu * xv,
            "dw2": go * s * silu * u,
        }
        got = run_bwd(p, np.full((1, 1), go, np.float32), lib=lib)
        vals = {"dx": got["dx"][0, 0], "dscores": got["dscores"][0, 0], "dwg": got["dw13"][0, 0, 0, 0],
                "dwu": got["dw13"][0, 1, 0, 0], "dw2": got["dw2"][0, 0, 0]}
        for key, r in ref.items():
            assert abs(vals[key] - r) <= 1e-5 * max(1.0, abs(r)), (key, vals[key], r)


def check_bwd_linear_in_dout(lib=None):
    p = small_problem(T=8, D=32, F=32, E=4, K=2, seed=24)
    dout = random_dout(8, 32, 24)
    a = run_bwd(p, dout, lib=lib)
    b = run_bwd(p, dout * np.float32(4.0), lib=lib)
    for key in ("dx", "dw13", "dw2", "dscores"):
        assert np.array_equal(b[key], a[key] * np.float32(4.0)), key


def check_bwd_zero_score_pair(lib=None):
    # a zero-score pair adds nothing to dx or the weight gradients, but its own dscore is <dout, y>
    p = small_problem(T=7, D=32, F=32, E=4, K=3, seed=25)
    p["scores"][:, 2] = 0.0
    dout = random_dout(7, 32, 25)
    a = run_bwd(p, dout, lib=lib)
    q = dict(p, ids=p["ids"].copy())
    q["ids"][:, 2] = -1
    b = run_bwd(q, dout, lib=lib)
    for key in ("dx", "dw13", "dw2"):
        assert np.array_equal(a[key], b[key]), key
    assert np.all(b["dscores"][:, 2] == 0.0)
    y = oracle.routed_experts(p["x"][:, :], p["ids"][:, 2:3].copy(), np.ones((7, 1), np.float32), p["w13"], p["w2"],
                              lib=lib)
    assert max_rel_err(a["dscores"][:, 2], np.sum(y * dout, axis=1)) <= 1e-5


def check_bwd_thread_count(lib=None):
    p = small_problem(T=11, D=32, F=32, E=3, K=2, seed=26)
    dout = random_dout(11, 32, 26)
    a = run_bwd(p, dout, lib=lib, nthreads=1)
    b = run_bwd(p, dout, lib=lib, nthreads=4)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


BWD_PINS = [
    check_bwd_vs_autograd,
    check_bwd_scalar_closed_form,
    check_bwd_linear_in_dout,
    check_bwd_zero_score_pair,
    check_bwd_thread_count,
]
