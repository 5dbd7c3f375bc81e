"""The seeded input generators: shapes, determinism and the routing distributions."""

import numpy as np
import pytest
import torch

from mixture_experts_routed_topk_gb300 import workloads as W


def test_shapes_and_dtypes_tiny():
    inp = W.make_inputs("tiny", seed=0)
    wl = inp["workload"]
    assert inp["x"].shape == (16, 256) and inp["x"].dtype == torch.bfloat16
    assert inp["topk_ids"].shape == (16, 2) and inp["topk_ids"].dtype == torch.int32
    assert inp["topk_scores"].dtype == torch.float32 and torch.all(inp["topk_scores"] == 0.5)
    assert inp["w13"].shape == (wl.E, 2, wl.F, wl.D) and inp["w2"].shape == (wl.E, wl.D, wl.F)
    ids = inp["topk_ids"].numpy()
    assert np.array_equal(ids, (np.arange(16)[:, None] * 2 + np.arange(2)[None, :]) % 8)


def test_deterministic_and_independent_streams():
    a = W.make_inputs("tiny", seed=3)
    b = W.make_inputs("tiny", seed=3)
    for k in ("x", "topk_ids", "topk_scores", "w13", "w2"):
        assert torch.equal(a[k], b[k])
    c = W.make_inputs("tiny", seed=4)
    assert not torch.equal(a["x"], c["x"])
    # one expert's weights do not depend on which other experts are drawn
    w13_all, w2_all = W.make_weights(8, 64, 64, seed=5)
    w13_one, w2_one = W.make_weights(8, 64, 64, seed=5, experts=[6])
    assert torch.equal(w13_all[6], w13_one[6]) and torch.equal(w2_all[6], w2_one[6])


def test_weight_scale():
    w13, w2 = W.make_weights(2, 512, 256, seed=0)
    assert abs(w13.float().std().item() * 512**0.5 - 1.0) < 0.02
    assert abs(w2.float().std().item() * 256**0.5 - 1.0) < 0.02


def test_uniform_routing_distinct_and_balanced():
    ids = W.make_topk_ids(4096, 64, 6, "uniform", seed=0).numpy()
    assert all(len(set(r)) == 6 for r in ids[:512])
    counts = np.bincount(ids.ravel(), minlength=64)
    mean = 4096 * 6 / 64
    assert counts.min() > 0.75 * mean and counts.max() < 1.25 * mean


def test_scores_softmax_normalised():
    s = W.make_scores(1000, 8, "softmax", seed=1)
    assert torch.allclose(s.sum(1), torch.ones(1000), atol=1e-6)
    assert torch.all(s > 0)


def _inclusion_probability(p, i, K, n=40000):
    # successive sampling without replacement as an exponential race (see SKEW_ZIPF_S)
    p = np.asarray(p, float) / np.sum(p)
    others = np.delete(p, i)
    t = np.linspace(0.0, 400.0, n)
    dp = np.zeros((n, K))
    dp[:, 0] = 1.0
    for pj in others:
        q = 1.0 - np.exp(-pj * t)
        nxt = dp * (1.0 - q)[:, None]
        nxt[:, 1:] += dp[:, :-1] * q[:, None]
        dp = nxt
    return np.trapezoid(p[i] * np.exp(-p[i] * t) * dp.sum(1), t)


def test_skew_exponent_gives_peak_to_mean_three():
    E, K = 128, 8
    p = W.skew_zipf_probs(E).numpy()
    assert int((p == 0).sum()) == round(0.05 * E) == 6
    assert np.all(p[-6:] == 0)
    ratio = _inclusion_probability(p[p > 0], 0, K) / (K / E)
    assert abs(ratio - W.SKEW_PEAK_TO_MEAN) < 1e-3, ratio


def test_skew_routing_empirical():
    ids = W.make_topk_ids(16384, 128, 8, "zipf", seed=0).numpy()
    assert all(len(set(r)) == 8 for r in ids[:256])
    counts = np.bincount(ids.ravel(), minlength=128)
    assert np.all(counts[122:] == 0)
    ratio = counts.max() / (16384 * 8 / 128)
    assert 2.85 < ratio < 3.15, ratio
