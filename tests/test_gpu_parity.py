"""The whole forward pass on the GPU against the CPU oracle on the same seeded inputs.

Sizes are chosen so the oracle finishes in seconds while the GPU path still runs several row
tiles per expert, partial column tiles and ragged expert tails. Also checked: the per-pair
score-weighted outputs Y in the workspace, the routing arrays in the workspace (bit-exact),
determinism, invalid ids, zero scores and bf16 scores.
"""

import numpy as np
import pytest
import torch

from common import max_rel_err
from gpu_common import (OUT_TOL, oracle_pairs, oracle_routing_of, oracle_tokens, run_fwd, to_device,
                        workspace_view)
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def problem(T, D, F, E, K, routing="uniform", seed=0, ids=None):
    d = {
        "x": W.make_x(T, D, seed),
        "topk_ids": ids if ids is not None else W.make_topk_ids(T, E, K, routing, seed),
        "topk_scores": W.make_scores(T, K, "softmax", seed),
    }
    d["w13"], d["w2"] = W.make_weights(E, D, F, seed)
    return to_device(d)


CASES = {
    # name: (T, D, F, E, K, routing)
    "ragged_multi_tile": (300, 256, 192, 6, 3, "uniform"),  # ~150 rows/expert: 2 row tiles, F tail of 64
    "partial_down_tile": (70, 320, 128, 5, 2, "uniform"),  # D % 256 = 64
    "wide": (96, 512, 384, 4, 2, "uniform"),  # 8 K-steps in the gate/up GEMM, 3 f tiles
    "many_empty_experts": (20, 128, 128, 64, 2, "uniform"),
    "k1": (129, 128, 256, 3, 1, "uniform"),
    "t1": (1, 256, 128, 8, 4, "uniform"),
    "k_equals_e": (40, 128, 128, 8, 8, "uniform"),
    "k_over_32": (24, 256, 128, 48, 40, "uniform"),  # a token's destination rows in two groups of lanes
    "max_experts": (64, 128, 128, 4096, 4, "uniform"),  # E at its maximum, almost every expert empty
    # one row tile per expert and 8 gate/up column tiles: 184 (200) tiles on a 152-SM grid leave a
    # partial wave of 32 (48) tiles, which the gate/up GEMM splits into quarters (halves)
    "tail_quarters": (2000, 128, 1024, 23, 1, "uniform"),
    "tail_halves": (2000, 128, 1024, 25, 1, "uniform"),
    "skew": (400, 128, 192, 16, 4, "zipf"),
    # several 128-token tiles per expert with ragged last tiles of every size class, wide D and F
    "multi_tile_wide": (600, 320, 384, 4, 2, "uniform"),  # D % 256 = 64; ~300 rows/expert
    "hot_experts": (2000, 128, 192, 16, 4, "zipf"),  # hot experts with several token tiles
}


def check_against_oracle(d, out, ws=None):
    ref, _ = oracle_tokens(d)
    err = max_rel_err(out.float().cpu().numpy(), ref)
    assert err <= OUT_TOL, err
    return err


@pytest.mark.parametrize("name", sorted(CASES))
def test_fwd_matches_oracle(name):
    T, D, F, E, K, routing = CASES[name]
    d = problem(T, D, F, E, K, routing)
    out, ws = run_fwd(d)
    check_against_oracle(d, out)
    assert binding.moe_get_status(ws) == 0


def test_tiny_workload_matches_oracle():
    d = to_device(W.make_inputs("tiny", seed=0))
    out, ws = run_fwd(d)
    err = check_against_oracle(d, out)
    assert err < 5e-3
    # routing arrays in the workspace are bit-exact
    T, D = d["x"].shape
    E, _, F, _ = d["w13"].shape
    K = d["topk_ids"].shape[1]
    dims = (T, D, F, E, K)
    ref = oracle_routing_of(d)
    for key, n in (("counts", E), ("offsets", E + 1), ("perm", T * K), ("inv", T * K)):
        got = workspace_view(ws, dims, key, torch.int32, n).cpu().numpy()
        assert np.array_equal(got, ref[key]), key
    assert np.all(ref["counts"] == 4)


def test_pair_outputs_match_oracle():
    # Y[p] = score[p] * W2[e] h(x_t) for every pair, read from the workspace after the pass
    T, D, F, E, K = 150, 256, 128, 5, 2
    d = problem(T, D, F, E, K)
    out, ws = run_fwd(d)
    y = workspace_view(ws, (T, D, F, E, K), "xp", torch.bfloat16, T * K * D).reshape(T * K, D)
    ref = oracle_pairs(d, np.arange(T * K))
    assert max_rel_err(y.float().cpu().numpy(), ref) <= OUT_TOL


def test_deterministic():
    d = problem(257, 256, 192, 7, 3)
    a, ws = run_fwd(d)
    b, _ = run_fwd(d, workspace=ws)
    c, _ = run_fwd(d)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_invalid_ids_contribute_zero_and_raise_status():
    d = problem(64, 128, 128, 6, 3)
    ids = d["topk_ids"].clone()
    ids[::7, 1] = -1
    ids[3::11, 2] = 6
    d["topk_ids"] = ids
    out, ws = run_fwd(d)
    assert binding.moe_get_status(ws) & binding.MOE_DEV_BAD_EXPERT_ID
    check_against_oracle(d, out)


def test_zero_score_pair_is_exactly_dropped():
    d = problem(48, 128, 128, 4, 3)
    sc = d["topk_scores"].clone()
    sc[:, 2] = 0.0
    d["topk_scores"] = sc
    a, _ = run_fwd(d)
    ids = d["topk_ids"].clone()
    ids[:, 2] = -1
    b, _ = run_fwd(dict(d, topk_ids=ids))
    assert torch.equal(a, b)


def test_bf16_scores():
    d = problem(100, 256, 128, 4, 2)
    d["topk_scores"] = d["topk_scores"].to(torch.bfloat16)
    out, _ = run_fwd(d)
    check_against_oracle(d, out)


def test_dense_special_case():
    # K = 1, one expert, score 1: a dense SwiGLU MLP over all tokens (many row tiles of one expert)
    T, D, F, E = 600, 256, 256, 1
    ids = torch.zeros((T, 1), dtype=torch.int32)
    d = problem(T, D, F, E, 1, ids=ids)
    d["topk_scores"] = torch.ones((T, 1), device="cuda")
    out, _ = run_fwd(d)
    check_against_oracle(d, out)


def test_stage_calls_equal_fused_call():
    d = problem(200, 256, 192, 6, 2)
    a, _ = run_fwd(d)
    T, D = d["x"].shape
    E, _, F, _ = d["w13"].shape
    K = d["topk_ids"].shape[1]
    dims = (T, D, F, E, K)
    ws = binding.alloc_workspace(binding.moe_workspace_bytes(*dims), "cuda")
    out = torch.empty_like(d["x"])
    binding.moe_fwd_dispatch(d["x"], d["topk_ids"], dims, ws)
    binding.moe_fwd_gemm1(d["w13"], dims, ws)
    binding.moe_fwd_gemm2(d["topk_scores"], d["w2"], dims, ws)
    binding.moe_fwd_combine(d["topk_ids"], out, dims, ws)
    assert torch.equal(a, out)


def test_token_without_valid_pairs_gets_zero_row():
    d = problem(300, 256, 128, 6, 3)
    ids = d["topk_ids"].clone()
    ids[5] = -1  # every pair of token 5 invalid
    ids[77, :] = 6
    ids[78, 1] = 9
    d["topk_ids"] = ids
    out = torch.full_like(d["x"], float("nan"))
    ws = binding.alloc_workspace(binding.moe_workspace_bytes(300, 256, 128, 6, 3), "cuda")
    binding.moe_routed_experts_fwd(d["x"], ids, d["topk_scores"], d["w13"], d["w2"], out, ws)
    # the combine writes every token's row, a token without any valid pair as zeros
    assert binding.moe_get_status(ws) & binding.MOE_DEV_BAD_EXPERT_ID
    assert torch.all(out[5] == 0) and torch.all(out[77] == 0)
    check_against_oracle(d, out)


def test_gather_stage_copies_rows():
    d = problem(90, 192, 128, 5, 3)
    T, D = d["x"].shape
    E, _, F, _ = d["w13"].shape
    K = d["topk_ids"].shape[1]
    dims = (T, D, F, E, K)
    ws = binding.alloc_workspace(binding.moe_workspace_bytes(*dims), "cuda")
    binding.moe_fwd_dispatch(d["x"], d["topk_ids"], dims, ws)
    xp = workspace_view(ws, dims, "xp", torch.bfloat16, T * K * D).reshape(T * K, D)
    perm = torch.from_numpy(oracle_routing_of(d)["perm"]).long().cuda()
    assert torch.equal(xp, d["x"][perm // K])


def test_medium_workload_token_subset():
    d = to_device(W.make_inputs("medium", seed=0), "cuda")
    out, ws = run_fwd(d)
    assert binding.moe_get_status(ws) == 0
    tokens = np.random.default_rng(0).choice(d["x"].shape[0], 24, replace=False)
    ref, tok = oracle_tokens(d, tokens)
    assert max_rel_err(out[torch.from_numpy(tok).cuda()].float().cpu().numpy(), ref) <= OUT_TOL


@pytest.mark.parametrize("name", ["ragged_multi_tile", "partial_down_tile", "skew"])
def test_fwd_rmsnorm_matches_oracle(name):
    import oracle
    from common import bf16_bits
    from gpu_common import scores_host

    T, D, F, E, K, routing = CASES[name]
    d = problem(T, D, F, E, K, routing)
    out = torch.empty_like(d["x"])
    ws = binding.alloc_workspace(binding.moe_workspace_bytes(T, D, F, E, K), "cuda")
    binding.moe_routed_experts_fwd_rmsnorm(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], d["w2"], out, ws,
                                           eps=1e-6)
    ref = oracle.routed_experts_rmsnorm(bf16_bits(d["x"]), d["topk_ids"].cpu().numpy(), scores_host(d["topk_scores"]),
                                        bf16_bits(d["w13"]), bf16_bits(d["w2"]), 1e-6)
    assert max_rel_err(out.float().cpu().numpy(), ref) <= OUT_TOL
    assert binding.moe_get_status(ws) == 0


def test_fwd_rmsnorm_ignores_w2_scale():
    # RMSNorm makes each expert output scale-free: scaling W2 by 4 leaves the result (nearly) unchanged
    d = problem(120, 256, 128, 4, 2)
    ws = binding.alloc_workspace(binding.moe_workspace_bytes(120, 256, 128, 4, 2), "cuda")
    a = torch.empty_like(d["x"])
    b = torch.empty_like(d["x"])
    binding.moe_routed_experts_fwd_rmsnorm(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], d["w2"], a, ws, eps=0.0)
    w2x4 = (d["w2"].float() * 4).to(torch.bfloat16)
    binding.moe_routed_experts_fwd_rmsnorm(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], w2x4, b, ws, eps=0.0)
    assert torch.equal(a, b)
