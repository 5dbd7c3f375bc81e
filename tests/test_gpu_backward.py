"""The backward pass on the GPU against the CPU oracle's backward on the same seeded inputs.

All four gradients (dx, dscores, dw13, dw2) are compared with max|got - ref| / max|ref| <= 1e-2
(bf16 operands and intermediates, fp32 accumulation), at sizes that span several padded row
tiles per expert, partial column tiles and experts without rows; plus invalid ids, duplicate
ids, zero scores, determinism, and subset checks on the medium workload.
"""

import numpy as np
import pytest
import torch

import oracle
from common import bf16_bits, max_rel_err
from gpu_common import scores_host, to_device
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2


def problem(T, D, F, E, K, routing="uniform", seed=0, ids=None):
    d = {
        "x": W.make_x(T, D, seed),
        "topk_ids": ids if ids is not None else W.make_topk_ids(T, E, K, routing, seed),
        "topk_scores": W.make_scores(T, K, "softmax", seed),
        "dout": W.make_x(T, D, seed + 101),
    }
    d["w13"], d["w2"] = W.make_weights(E, D, F, seed)
    return to_device(d)


def run_bwd(d):
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    ws = binding.alloc_workspace(binding.moe_bwd_workspace_bytes(T, D, F, E, K), x.device)
    g = {
        "dx": torch.empty_like(x),
        "dscores": torch.empty((T, K), dtype=torch.float32, device=x.device),
        "dw13": torch.empty_like(w13),
        "dw2": torch.empty_like(d["w2"]),
    }
    binding.moe_routed_experts_bwd(x, ids, d["topk_scores"], w13, d["w2"], d["dout"], g["dx"], g["dscores"],
                                   g["dw13"], g["dw2"], ws)
    return g, ws


def oracle_bwd(d):
    return oracle.routed_experts_bwd(bf16_bits(d["x"]), d["topk_ids"].cpu().numpy(), scores_host(d["topk_scores"]),
                                     bf16_bits(d["w13"]), bf16_bits(d["w2"]), d["dout"].float().cpu().numpy())


def check_all(got, ref):
    errs = {}
    for key in ("dx", "dscores", "dw13", "dw2"):
        errs[key] = max_rel_err(got[key].float().cpu().numpy(), ref[key])
        assert errs[key] <= TOL, (key, errs)
    return errs


CASES = {
    # name: (T, D, F, E, K, routing)
    "multi_tile": (300, 256, 192, 6, 3, "uniform"),  # ~150 rows/expert: 2 padded row tiles
    "partial_tiles": (70, 320, 128, 5, 2, "uniform"),  # D % 256 = 64, F < 256
    "wide": (96, 512, 384, 4, 2, "uniform"),
    "empty_experts": (20, 128, 128, 64, 2, "uniform"),  # most experts get no rows: zero dW
    "k1": (129, 128, 256, 3, 1, "uniform"),
    "skew": (400, 128, 192, 16, 4, "zipf"),
    "k_over_32": (24, 128, 128, 48, 40, "uniform"),  # 40 padded rows per token in the gather
    "max_experts": (48, 64, 64, 4096, 4, "uniform"),  # E at its maximum: almost every dW block zero
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bwd_matches_oracle(name):
    T, D, F, E, K, routing = CASES[name]
    d = problem(T, D, F, E, K, routing)
    got, ws = run_bwd(d)
    check_all(got, oracle_bwd(d))
    assert binding.moe_get_status(ws) == 0


def test_bwd_invalid_duplicate_and_zero_score_pairs():
    d = problem(64, 128, 128, 6, 4)
    ids = d["topk_ids"].clone()
    ids[::5, 1] = -1  # invalid: contributes nothing, dscores 0
    ids[1::7, 2] = ids[1::7, 0]  # duplicate id within a token
    d["topk_ids"] = ids
    sc = d["topk_scores"].clone()
    sc[::3, 3] = 0.0  # zero score: nothing in dx / dW, dscores still <dout, y>
    d["topk_scores"] = sc
    got, ws = run_bwd(d)
    ref = oracle_bwd(d)
    check_all(got, ref)
    assert torch.all(got["dscores"][::5, 1] == 0)
    assert binding.moe_get_status(ws) & binding.MOE_DEV_BAD_EXPERT_ID


def test_bwd_deterministic():
    d = problem(200, 256, 192, 5, 2)
    a, _ = run_bwd(d)
    b, _ = run_bwd(d)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_bwd_medium_workload_subsets():
    d = to_device(W.make_inputs("medium", seed=0), "cuda")
    d["dout"] = W.make_x(4096, 2048, 101, "cuda")
    got, ws = run_bwd(d)
    assert binding.moe_get_status(ws) == 0
    ids = d["topk_ids"].cpu().numpy()
    E = d["w13"].shape[0]

    def compact(tokens):
        sub = {k: d[k][torch.from_numpy(tokens).cuda()] for k in ("x", "topk_ids", "topk_scores", "dout")}
        experts = np.unique(ids[tokens])
        remap = np.full(E, -1, np.int64)
        remap[experts] = np.arange(experts.size)
        sub_ids = remap[ids[tokens]].astype(np.int32)
        ex = torch.from_numpy(experts).cuda()
        ref = oracle.routed_experts_bwd(bf16_bits(sub["x"]), sub_ids, scores_host(sub["topk_scores"]),
                                        bf16_bits(d["w13"].index_select(0, ex)), bf16_bits(d["w2"].index_select(0, ex)),
                                        sub["dout"].float().cpu().numpy())
        return ref, remap

    # whole tokens: dx and dscores depend only on the token's own pairs
    tokens = np.random.default_rng(0).choice(4096, 12, replace=False)
    ref, _ = compact(tokens)
    tt = torch.from_numpy(tokens).cuda()
    assert max_rel_err(got["dx"][tt].float().cpu().numpy(), ref["dx"]) <= TOL
    assert max_rel_err(got["dscores"][tt].cpu().numpy(), ref["dscores"]) <= TOL
    # one expert's weight gradients need every pair routed to it: take exactly those tokens
    counts = np.bincount(ids.ravel(), minlength=E)
    e = int(np.argmin(counts))
    tokens = np.flatnonzero((ids == e).any(axis=1))
    ref, remap = compact(tokens)
    assert max_rel_err(got["dw13"][e].float().cpu().numpy(), ref["dw13"][remap[e]]) <= TOL
    assert max_rel_err(got["dw2"][e].float().cpu().numpy(), ref["dw2"][remap[e]]) <= TOL


def test_bwd_bf16_scores():
    d = problem(90, 256, 128, 4, 2)
    d["topk_scores"] = d["topk_scores"].to(torch.bfloat16)
    got, _ = run_bwd(d)
    check_all(got, oracle_bwd(d))


def test_bwd_no_tokens_gives_zero_weight_gradients():
    E, D, F = 3, 128, 64
    w13, w2 = W.make_weights(E, D, F, 0, "cuda")
    dw13 = torch.full_like(w13, 7.0)
    dw2 = torch.full_like(w2, 7.0)
    x = torch.empty((0, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    sc = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    ws = binding.alloc_workspace(256, "cuda")
    binding.moe_routed_experts_bwd(x, ids, sc, w13, w2, x, torch.empty_like(x), sc.clone(), dw13, dw2, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw13) == 0 and torch.count_nonzero(dw2) == 0


@pytest.mark.parametrize("split", [[0, 7], [0, 1, 2, 3, 4, 5, 6, 7], [0, 3, 5, 7]])
def test_stage_calls_equal_the_whole_call(split):
    # the backward run as consecutive stage ranges on one workspace gives the whole call's bits
    d = problem(300, 256, 192, 6, 3)
    ref, _ = run_bwd(d)
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    ws = binding.alloc_workspace(binding.moe_bwd_workspace_bytes(T, D, F, E, K), x.device)
    g = {k: torch.full_like(v, 7) for k, v in ref.items()}
    for b, e in zip(split[:-1], split[1:]):
        binding.moe_bwd_stages(x, ids, d["topk_scores"], w13, d["w2"], d["dout"], g["dx"], g["dscores"], g["dw13"],
                               g["dw2"], ws, b, e)
    assert binding.moe_get_status(ws) == 0
    for k in ref:
        assert torch.equal(g[k], ref[k]), k


def test_each_stage_writes_only_its_outputs():
    # the stages before the reductions leave dx and dscores untouched; the weight-gradient stages
    # write dw2 and dw13 and nothing of each other
    d = problem(300, 256, 192, 6, 3)
    ref, _ = run_bwd(d)
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    ws = binding.alloc_workspace(binding.moe_bwd_workspace_bytes(T, D, F, E, K), x.device)
    g = {k: torch.full_like(v, 7) for k, v in ref.items()}
    call = lambda b, e: binding.moe_bwd_stages(x, ids, d["topk_scores"], w13, d["w2"], d["dout"], g["dx"],
                                               g["dscores"], g["dw13"], g["dw2"], ws, b, e)
    call(0, 4)
    torch.cuda.synchronize()
    assert all(torch.all(g[k] == 7) for k in ("dx", "dscores", "dw13", "dw2"))
    call(4, 5)
    torch.cuda.synchronize()
    assert torch.equal(g["dw2"], ref["dw2"]) and torch.all(g["dw13"] == 7) and torch.all(g["dx"] == 7)
    call(5, 6)
    torch.cuda.synchronize()
    assert torch.equal(g["dw13"], ref["dw13"]) and torch.all(g["dx"] == 7) and torch.all(g["dscores"] == 7)
    call(6, 7)
    assert torch.equal(g["dx"], ref["dx"]) and torch.equal(g["dscores"], ref["dscores"])


def test_stage_range_validation():
    d = problem(16, 128, 128, 4, 2)
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    g, ws = run_bwd(d)
    for b, e in ((-1, 2), (3, 2), (0, 8)):
        with pytest.raises(binding.MoeError):
            binding.moe_bwd_stages(x, ids, d["topk_scores"], w13, d["w2"], d["dout"], g["dx"], g["dscores"],
                                   g["dw13"], g["dw2"], ws, b, e)
