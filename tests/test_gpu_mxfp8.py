"""The MXFP8 forward on the GPU against the CPU oracle on the same seeded inputs.

Bit-exact: the prepared weights (E4M3 codes and UE8M0 scales, read back through the documented
tile-grouped scale layout) and the quantized activation rows in the workspace (integers decided
from the same bf16 inputs in fp32 on both sides). Within the layer's tolerance: out, against
the oracle's MXFP8 forward fed with weights the oracle quantized itself. Also: padding rows,
determinism, invalid ids, zero and bf16 scores, and every workload at full size on sampled
tokens.
"""

import numpy as np
import pytest
import torch

import oracle
from common import bf16_bits, max_rel_err
from gpu_common import OUT_TOL, scores_host, to_device
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu

W13, W2 = binding.MOE_WEIGHT_W13, binding.MOE_WEIGHT_W2


# ------------------------------------------------------------------------- layout helpers

def sf_in_chunk(n):
    n = np.asarray(n)
    return 16 * (n % 32) + 4 * ((n % 128) // 32)


def untile_weight_scales(scales: np.ndarray, which: int, D: int, F: int, E: int) -> np.ndarray:
    """Row-major [rows, C/32] scales from the tile-grouped layout (the header's formula)."""
    if which == W13:
        rows, C, NT, tile_rows = E * 2 * F, D, -(-F // 96), 96
        r = np.arange(rows)
        e, rem = r // (2 * F), r % (2 * F)
        half, f = rem // F, rem % F
        j, n = f // tile_rows, half * tile_rows + f % tile_rows
    else:
        rows, C, NT, tile_rows = E * D, F, -(-D // 192), 192
        r = np.arange(rows)
        e, d = r // D, r % D
        j, n = d // tile_rows, d % tile_rows
    b = np.arange(C // 32)
    off = (((e * NT + j) * (C // 128))[:, None] + (b // 4)[None, :]) * 1024 + (512 * (n // 128) + sf_in_chunk(n))[:, None] \
        + (b % 4)[None, :]
    return scales[off], off


def untile_act_scales(xs: np.ndarray, rows: np.ndarray, cols: int) -> np.ndarray:
    b = np.arange(cols // 32)
    off = (((rows // 128) * (cols // 128))[:, None] + (b // 4)[None, :]) * 512 + sf_in_chunk(rows)[:, None] \
        + (b % 4)[None, :]
    return xs[off]


# ------------------------------------------------------------------------------ problems

def problem(T, D, F, E, K, routing="uniform", seed=0, ids=None):
    d = {
        "x": W.make_x(T, D, seed),
        "topk_ids": ids if ids is not None else W.make_topk_ids(T, E, K, routing, seed),
        "topk_scores": W.make_scores(T, K, "softmax", seed),
    }
    d["w13"], d["w2"] = W.make_weights(E, D, F, seed)
    return to_device(d)


def prepare(d):
    return (binding.moe_mxfp8_prepare_weight(W13, d["w13"]), binding.moe_mxfp8_prepare_weight(W2, d["w2"]))


def run_mx(d, mx=None, workspace=None):
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    mx = mx or prepare(d)
    if workspace is None:
        workspace = binding.alloc_workspace(binding.moe_mxfp8_workspace_bytes(T, D, F, E, K), x.device)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=x.device)
    binding.moe_routed_experts_fwd_mxfp8(x, ids, d["topk_scores"], mx[0], mx[1], out, workspace, dims_FE=(F, E))
    return out, workspace


def oracle_mx_tokens(d, tokens=None):
    """The oracle's MXFP8 out for the given tokens; only the experts they touch are copied and
    quantized (by the oracle), ids renumbered into that compact set."""
    ids_all = d["topk_ids"]
    T = ids_all.shape[0]
    E = d["w13"].shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    tok_t = torch.from_numpy(tok).to(ids_all.device)
    ids = ids_all.index_select(0, tok_t).cpu().numpy()
    valid = (ids >= 0) & (ids < E)
    experts = np.unique(ids[valid])
    remap = np.full(E, -1, np.int64)
    remap[experts] = np.arange(experts.size)
    ids_c = np.where(valid, remap[np.clip(ids, 0, E - 1)], -1).astype(np.int32)
    if experts.size == 0:
        experts = np.zeros(1, np.int64)
    ex_t = torch.from_numpy(experts).to(d["w13"].device)
    w13 = oracle.mx_quantize_rows(bf16_bits(d["w13"].index_select(0, ex_t)))
    w2 = oracle.mx_quantize_rows(bf16_bits(d["w2"].index_select(0, ex_t)))
    x = bf16_bits(d["x"].index_select(0, tok_t))
    sc = scores_host(d["topk_scores"].index_select(0, tok_t))
    return oracle.routed_experts_mxfp8(x, ids_c, sc, w13, w2), tok


# ------------------------------------------------------------------------------------ tests

def special_weights(E, D, F, seed):
    w13, w2 = W.make_weights(E, D, F, seed)
    w13 = w13.clone()
    w13[0, 0, 0, :64] = 0.0  # all-zero blocks
    w13[0, 1, 1, :32] = -0.0
    w13[0, 0, 2, :32] *= 2.0 ** -120  # tiny (bf16 subnormals included)
    w13[-1, 1, -1, 5] = 300.0  # a spike: the rest of its block near the bottom of the range
    w2 = w2.clone()
    w2[0, 0, 32:64] = 0.0
    w2[-1, -1, :32] *= 2.0 ** 100
    return w13, w2


@pytest.mark.parametrize("dims", [(3, 384, 256), (2, 256, 384), (1, 128, 128), (5, 640, 1024)])
def test_prepared_weights_bit_exact(dims):
    E, D, F = dims
    w13, w2 = special_weights(E, D, F, 7)
    for which, w in ((W13, w13), (W2, w2)):
        data, scales = binding.moe_mxfp8_prepare_weight(which, w.cuda())
        codes, sc = oracle.mx_quantize_rows(bf16_bits(w))
        got = data.cpu().numpy()
        assert np.array_equal(got, codes.reshape(-1)), (which, int((got != codes.reshape(-1)).sum()))
        sc_host = scales.cpu().numpy()
        tiled, off = untile_weight_scales(sc_host, which, D, F, E)
        assert np.array_equal(tiled, sc.reshape(tiled.shape)), which
        unused = np.ones(sc_host.size, bool)
        unused[off.reshape(-1)] = False
        assert not sc_host[unused].any(), "bytes of no row must be 0"


CASES = {
    # name: (T, D, F, E, K, routing)
    "tiny_round_robin": (16, 256, 256, 8, 2, "round_robin"),
    "ragged_multi_tile": (300, 256, 256, 6, 3, "uniform"),  # 2 row tiles per expert; F tail 64 of 96
    "partial_down_tile": (70, 384, 128, 5, 2, "uniform"),  # D = 2 * 192, F a single K step
    "wide": (96, 640, 512, 4, 2, "uniform"),  # 5 K steps, D tail 64 of 192
    "many_empty_experts": (20, 128, 128, 64, 2, "uniform"),
    "k1": (129, 128, 256, 3, 1, "uniform"),
    "t1": (1, 256, 128, 8, 4, "uniform"),
    "k_equals_e": (40, 128, 128, 8, 8, "uniform"),
    "k_over_32": (24, 256, 128, 48, 40, "uniform"),  # a token's destination rows in two groups of lanes
    "max_experts": (64, 128, 128, 4096, 4, "uniform"),  # E at its maximum, almost every expert empty
    "skewed_small": (256, 256, 384, 16, 4, "zipf"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_mxfp8_forward_matches_oracle(name):
    T, D, F, E, K, routing = CASES[name]
    d = problem(T, D, F, E, K, routing, seed=3)
    out, ws = run_mx(d)
    assert binding.moe_get_status(ws) == 0
    ref, _ = oracle_mx_tokens(d)
    err = max_rel_err(out.float().cpu().numpy(), ref)
    assert err <= OUT_TOL, (name, err)


def test_mxfp8_every_pair_on_two_experts():
    # experts 0 and E-1 take every pair (six row tiles each, many column tiles and K steps in a
    # row through the same stages and scale slots); the other experts are empty
    T, D, F, E, K = 700, 512, 384, 8, 2
    ids = torch.zeros((T, K), dtype=torch.int32)
    ids[:, 1] = E - 1
    d = problem(T, D, F, E, K, seed=5, ids=ids)
    out, ws = run_mx(d)
    assert binding.moe_get_status(ws) == 0
    ref, _ = oracle_mx_tokens(d)
    err = max_rel_err(out.float().cpu().numpy(), ref)
    assert err <= OUT_TOL, err


@pytest.mark.parametrize("T", [300, 2100])  # 1024-column work items, and whole rows (T >= 2048)
def test_activation_rows_bit_exact_and_padding_zero(T):
    D, F, E, K = 384, 256, 6, 3
    d = problem(T, D, F, E, K, seed=4)
    out, ws = run_mx(d)
    dims = (T, D, F, E, K)
    lay = binding.moe_mxfp8_workspace_layout(*dims)
    R = T * K
    rp = 128 * (-(-R // 128) + min(E, R))
    tiles = ws[lay["tiles"]:lay["tiles"] + 4 * (E + 1)].view(torch.int32).cpu().numpy()
    xq = ws[lay["xq"]:lay["xq"] + rp * D].cpu().numpy().reshape(rp, D)
    xs = ws[lay["xs"]:lay["xs"] + rp * D // 32].cpu().numpy()
    rt = oracle.routing(d["topk_ids"].cpu().numpy(), E)
    codes, sc = oracle.mx_quantize_rows(bf16_bits(d["x"].cpu()))
    valid_rows = []
    for e in range(E):
        n = int(rt["counts"][e])
        assert tiles[e + 1] - tiles[e] == -(-n // 128)
        prows = 128 * int(tiles[e]) + np.arange(n)
        toks = rt["perm"][rt["offsets"][e]:rt["offsets"][e] + n] // K
        assert np.array_equal(xq[prows], codes[toks]), e
        assert np.array_equal(untile_act_scales(xs, prows, D), sc[toks]), e
        valid_rows.append(prows)
    used = 128 * int(tiles[E])
    pad = np.setdiff1d(np.arange(used), np.concatenate(valid_rows))
    assert pad.size > 0
    assert not xq[pad].any()
    assert not untile_act_scales(xs, pad, D).any()


def test_mxfp8_deterministic_and_reusable_workspace():
    d = problem(200, 256, 256, 7, 3, seed=5)
    mx = prepare(d)
    a, ws = run_mx(d, mx)
    b, _ = run_mx(d, mx, workspace=ws)
    assert torch.equal(a, b)
    # the same workspace, now for a smaller problem and back
    small = problem(9, 256, 256, 7, 3, seed=6)
    run_mx(small, workspace=ws)
    c, _ = run_mx(d, mx, workspace=ws)
    assert torch.equal(a, c)


def test_mxfp8_invalid_ids_zero_and_bf16_scores():
    T, D, F, E, K = 64, 256, 128, 5, 3
    d = problem(T, D, F, E, K, seed=8)
    mx = prepare(d)
    ids = d["topk_ids"].clone()
    ids[::3, 1] = -1
    ids[1::7, 2] = E + 2
    dropped = dict(d, topk_ids=ids)
    out, ws = run_mx(dropped, mx)
    assert binding.moe_get_status(ws) & binding.MOE_DEV_BAD_EXPERT_ID
    ref, _ = oracle_mx_tokens(dropped)
    assert max_rel_err(out.float().cpu().numpy(), ref) <= OUT_TOL
    # zero scores on the same pairs give exactly the same output
    sc = d["topk_scores"].clone()
    bad = (ids < 0) | (ids >= E)
    sc[bad] = 0.0
    zero, _ = run_mx(dict(d, topk_scores=sc), mx)
    assert torch.equal(zero, out)
    # bf16 scores
    sb = d["topk_scores"].to(torch.bfloat16)
    outb, _ = run_mx(dict(d, topk_scores=sb), mx)
    refb, _ = oracle_mx_tokens(dict(d, topk_scores=sb))
    assert max_rel_err(outb.float().cpu().numpy(), refb) <= OUT_TOL


# sampled tokens beyond the first and last; the oracle quantizes every expert they touch (about a
# second per large expert on one core), so the counts stay small
@pytest.mark.parametrize("name,ntok", [("medium", 10), ("decode", 1), ("skewed", 2), ("large", 0)])
def test_mxfp8_full_size_sampled_tokens(name, ntok):
    d = W.make_inputs(name, seed=0, device="cuda")
    T = d["workload"].T
    out, ws = run_mx(d)
    assert binding.moe_get_status(ws) == 0
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, ntok, replace=False)]))
    ref, tok = oracle_mx_tokens(d, tokens)
    err = max_rel_err(out.float().cpu().numpy()[tok], ref)
    assert err <= OUT_TOL, err


def test_mxfp8_stages_equal_fused_call():
    T, D, F, E, K = 150, 256, 384, 5, 3
    d = problem(T, D, F, E, K, seed=9)
    mx = prepare(d)
    fused, ws = run_mx(d, mx)
    out = torch.empty_like(fused)
    for s in range(binding.MX_STAGES):
        binding.moe_fwd_mxfp8_stages(d["x"], d["topk_ids"], d["topk_scores"], mx[0], mx[1], out, ws, (F, E), s, s + 1)
    assert torch.equal(out, fused)
