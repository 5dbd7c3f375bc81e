"""Parity at the workloads' full sizes, in the launch configuration the benchmark times.

The whole pass runs on the full inputs (generated on the GPU). Routing is checked in full
(bit-exact); the layer's arithmetic is checked on samples the oracle can evaluate one by one:
pairs of the hottest expert, of the coldest non-empty expert and of random experts (including
the first and last rows of each sampled segment, i.e. tile edges), and a few whole tokens.
"""

import gc

import numpy as np
import pytest
import torch

from common import max_rel_err
from gpu_common import OUT_TOL, oracle_pairs, oracle_routing_of, oracle_tokens, run_fwd, workspace_view
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def sample_pairs(routing: dict, rng, per_extreme=64, per_random=6) -> np.ndarray:
    """Up to 64 pairs each of the hottest and the coldest non-empty expert, 6 each of two random
    experts, always with the first and last row of every sampled segment (tile edges)."""
    counts, offsets, perm = routing["counts"], routing["offsets"], routing["perm"]
    nonempty = np.flatnonzero(counts)
    hot = int(np.argmax(counts))
    cold = int(nonempty[np.argmin(counts[nonempty])])
    picks = {e: per_random for e in rng.choice(nonempty, size=min(2, nonempty.size), replace=False).tolist()}
    picks[hot] = picks[cold] = per_extreme
    rows = []
    for e in sorted(picks):
        a, b = int(offsets[e]), int(offsets[e + 1])
        chosen = {a, b - 1}
        if b - a > 2:
            chosen.update(rng.choice(np.arange(a + 1, b - 1), size=min(picks[e] - 2, b - a - 2), replace=False).tolist())
        rows.extend(sorted(chosen))
    return perm[np.asarray(rows, dtype=np.int64)].astype(np.int64)


@pytest.mark.parametrize("name", ["medium", "decode", "skewed", "large"])
def test_full_size_workload(name):
    d = W.make_inputs(name, seed=0, device="cuda")
    wl = d["workload"]
    T, D, F, E, K = wl.dims()
    out, ws = run_fwd(d)
    assert binding.moe_get_status(ws) == 0
    dims = (T, D, F, E, K)

    ref_routing = oracle_routing_of(d)
    for key, n in (("counts", E), ("offsets", E + 1), ("perm", T * K), ("inv", T * K)):
        got = workspace_view(ws, dims, key, torch.int32, n).cpu().numpy()
        assert np.array_equal(got, ref_routing[key]), key

    rng = np.random.default_rng(1)
    pairs = sample_pairs(ref_routing, rng)
    y = workspace_view(ws, dims, "xp", torch.bfloat16, T * K * D).reshape(T * K, D)
    got_y = y[torch.from_numpy(pairs).cuda()].float().cpu().numpy()
    assert max_rel_err(got_y, oracle_pairs(d, pairs)) <= OUT_TOL

    tokens = rng.choice(T, size=2, replace=False)
    ref_out, tok = oracle_tokens(d, tokens)
    assert max_rel_err(out[torch.from_numpy(tok).cuda()].float().cpu().numpy(), ref_out) <= OUT_TOL

    again, _ = run_fwd(d, workspace=ws)
    assert torch.equal(out, again)

    del d, out, again, ws, y
    gc.collect()
    torch.cuda.empty_cache()
