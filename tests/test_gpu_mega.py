"""The fused (Mega) forward on the GPU: one grid runs the gate/up and down grouped GEMMs,
a down tile starting once the gate/up tiles of its rows have written H. It computes the same tiles
with the same roundings as the staged forward, so its output must be bit-identical to the staged
one (and therefore within the oracle tolerance) on every case: ragged tails, empty experts,
skewed routing, K = 1, T = 1, invalid ids, bf16 scores, and shapes where the interleaved schedule
(down tiles of expert e running beside gate/up tiles of later experts) really interleaves."""

import numpy as np
import pytest
import torch

from common import max_rel_err
from gpu_common import OUT_TOL, oracle_tokens, run_fwd, to_device
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W
from test_gpu_parity import CASES, problem

pytestmark = pytest.mark.gpu


def run_mega(d, workspace=None):
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    if workspace is None:
        workspace = binding.alloc_workspace(binding.moe_mega_workspace_bytes(T, D, F, E, K), x.device)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=x.device)
    binding.moe_routed_experts_fwd_mega(x, ids, d["topk_scores"], w13, d["w2"], out, workspace)
    return out, workspace


@pytest.mark.parametrize("name", sorted(CASES))
def test_mega_equals_staged_and_oracle(name):
    T, D, F, E, K, routing = CASES[name]
    d = problem(T, D, F, E, K, routing)
    staged, _ = run_fwd(d)
    out, ws = run_mega(d)
    assert binding.moe_get_status(ws) == 0
    assert torch.equal(out, staged)
    ref, _ = oracle_tokens(d)
    assert max_rel_err(out.float().cpu().numpy(), ref) <= OUT_TOL


# Enough gate/up tiles per expert that an expert's down slot trails its gate/up slot by fewer
# experts than there are (the schedule interleaves the two GEMMs instead of running them in turn).
INTERLEAVED = {
    # name: (T, D, F, E, K, routing)
    "interleaved_uniform": (2048, 256, 1024, 32, 6, "uniform"),
    "interleaved_zipf": (2048, 256, 1024, 32, 6, "zipf"),
    "interleaved_ragged_f": (1536, 320, 1088, 24, 4, "uniform"),  # F % 128 = 64, D % 256 = 64
}


@pytest.mark.parametrize("name", sorted(INTERLEAVED))
def test_mega_interleaved_schedule(name):
    T, D, F, E, K, routing = INTERLEAVED[name]
    d = problem(T, D, F, E, K, routing, seed=3)
    staged, _ = run_fwd(d)
    out, ws = run_mega(d)
    assert binding.moe_get_status(ws) == 0
    assert torch.equal(out, staged)
    tokens = np.random.default_rng(1).choice(T, 48, replace=False)
    ref, tok = oracle_tokens(d, tokens)
    assert max_rel_err(out[torch.from_numpy(tok).cuda()].float().cpu().numpy(), ref) <= OUT_TOL


def test_mega_medium_workload():
    d = to_device(W.make_inputs("medium", seed=0), "cuda")
    staged, _ = run_fwd(d)
    out, ws = run_mega(d)
    assert binding.moe_get_status(ws) == 0
    assert torch.equal(out, staged)
    tokens = np.random.default_rng(0).choice(d["x"].shape[0], 16, replace=False)
    ref, tok = oracle_tokens(d, tokens)
    assert max_rel_err(out[torch.from_numpy(tok).cuda()].float().cpu().numpy(), ref) <= OUT_TOL


def test_mega_deterministic_and_reusable():
    d = problem(*INTERLEAVED["interleaved_uniform"][:5], seed=5)
    a, ws = run_mega(d)
    b, _ = run_mega(d, workspace=ws)  # the readiness counters are cleared by every call
    c, _ = run_mega(d)
    assert torch.equal(a, b) and torch.equal(a, c)
    assert binding.moe_get_status(ws) == 0


def test_mega_invalid_ids_and_bf16_scores():
    d = problem(300, 256, 192, 6, 3)
    ids = d["topk_ids"].clone()
    ids[::7, 1] = -1
    ids[3::11, 2] = 6
    d["topk_ids"] = ids
    d["topk_scores"] = d["topk_scores"].to(torch.bfloat16)
    staged, _ = run_fwd(d)
    out, ws = run_mega(d)
    assert binding.moe_get_status(ws) & binding.MOE_DEV_BAD_EXPERT_ID
    assert not binding.moe_get_status(ws) & binding.MOE_DEV_TIMEOUT
    assert torch.equal(out, staged)


def test_mega_all_ids_invalid():
    # no valid pair: no tiles at all; every output row is zero
    d = problem(40, 128, 128, 4, 2)
    d["topk_ids"] = torch.full_like(d["topk_ids"], 9)
    out, ws = run_mega(d)
    assert binding.moe_get_status(ws) == binding.MOE_DEV_BAD_EXPERT_ID
    assert torch.count_nonzero(out) == 0


def test_mega_stage_calls_equal_whole_call():
    d = problem(*INTERLEAVED["interleaved_ragged_f"][:5], seed=7)
    a, _ = run_mega(d)
    T, D = d["x"].shape
    E, _, F, _ = d["w13"].shape
    K = d["topk_ids"].shape[1]
    ws = binding.alloc_workspace(binding.moe_mega_workspace_bytes(T, D, F, E, K), "cuda")
    out = torch.empty_like(d["x"])
    for s in range(binding.MEGA_STAGES):
        binding.moe_fwd_mega_stages(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], d["w2"], out, ws, s, s + 1)
    assert torch.equal(a, out)
    assert binding.moe_get_status(ws) == 0
