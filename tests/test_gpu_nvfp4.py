"""The NVFP4 forward on the GPU against the CPU oracle on the same seeded inputs.

Bit-exact: the prepared weights (packed E2M1 codes, the tensor scale in the scale header and the
UE4M3 block scales read back through the documented tile-grouped layout) and the quantized x rows
in the workspace (integers decided from the same inputs with the same fp32 steps on both sides).
Within the layer's tolerance: out, against the oracle's NVFP4 forward fed with weights the oracle
quantized itself. Also: padding rows and padding scale groups, determinism, invalid ids, zero and
bf16 scores, the stage calls, and every workload at full size on sampled tokens.
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
HEADER = 256
H_SCALE = 2.0 ** -8  # tensor scale of the SwiGLU output: |h| up to 6 * 448 * 2^-8 = 10.5 without saturating


def groups(cols):
    return -(-cols // 256) * 4


def sf_in_chunk(n):
    n = np.asarray(n)
    return 16 * (n % 32) + 4 * ((n % 128) // 32)


def unpack(packed: np.ndarray) -> np.ndarray:
    """Packed E2M1 bytes [..., c/2] -> one code per byte [..., c] (low nibble first)."""
    lo, hi = packed & 15, packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))


def untile_weight_scales(scales: np.ndarray, which: int, D: int, F: int, E: int):
    if which == W13:
        rows, C, NT, tr = E * 2 * F, D, -(-F // 64), 64
        r = np.arange(rows)
        e, rem = r // (2 * F), r % (2 * F)
        half, f = rem // F, rem % F
        j, n = f // tr, half * tr + f % tr
    else:
        rows, C, NT, tr = E * D, F, -(-D // 128), 128
        r = np.arange(rows)
        e, d = r // D, r % D
        j, n = d // tr, d % tr
    b = np.arange(C // 16)
    off = HEADER + (((e * NT + j) * groups(C))[:, None] + (b // 4)[None, :]) * 512 + sf_in_chunk(n)[:, None] \
        + (b % 4)[None, :]
    return scales[off], off


def untile_act_scales(xs: np.ndarray, rows: np.ndarray, cols: int) -> np.ndarray:
    b = np.arange(cols // 16)
    off = (((rows // 128) * groups(cols))[:, None] + (b // 4)[None, :]) * 512 + sf_in_chunk(rows)[:, None] \
        + (b % 4)[None, :]
    return xs[off]


def problem(T, D, F, E, K, routing="uniform", seed=0, ids=None):
    d = {
        "x": W.make_x(T, D, seed),
        "topk_ids": ids if ids is not None else W.make_topk_ids(T, E, K, routing, seed),
        "topk_scores": W.make_scores(T, K, "softmax", seed),
    }
    d["w13"], d["w2"] = W.make_weights(E, D, F, seed)
    return to_device(d)


def x_scale_of(x: torch.Tensor) -> float:
    """Calibration of x's tensor scale: amax / 2688 in fp32 (computed on the host)."""
    amax = np.float32(x.detach().abs().max().float().cpu().item())
    return float(amax / np.float32(2688.0))


def prepare(d):
    return (binding.moe_nvfp4_prepare_weight(W13, d["w13"]), binding.moe_nvfp4_prepare_weight(W2, d["w2"]))


def run_nv(d, nv=None, workspace=None, gx=None, gh=H_SCALE):
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    nv = nv or prepare(d)
    gx = x_scale_of(x) if gx is None else gx
    if workspace is None:
        workspace = binding.alloc_workspace(binding.moe_nvfp4_workspace_bytes(T, D, F, E, K), x.device)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=x.device)
    binding.moe_routed_experts_fwd_nvfp4(x, ids, d["topk_scores"], nv[0], nv[1], out, workspace, (F, E), gx, gh)
    return out, workspace


def oracle_nv_tokens(d, tokens=None, gx=None, gh=H_SCALE):
    """The oracle's NVFP4 out for the given tokens. The weights' tensor scales come from the whole
    tensors (as prepared); only the experts the tokens touch are quantized and passed."""
    ids_all = d["topk_ids"]
    T = ids_all.shape[0]
    E = d["w13"].shape[0]
    gx = x_scale_of(d["x"]) if gx is None else gx
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
    out = []
    for name in ("w13", "w2"):
        w = d[name]
        amax = np.float32(w.abs().max().float().cpu().item())
        G = float(amax / np.float32(2688.0)) if amax > 0 else 1.0
        codes, scales = oracle.nvfp4_quantize_rows(bf16_bits(w.index_select(0, ex_t)), G)
        out.append((codes, scales, G))
    x = bf16_bits(d["x"].index_select(0, tok_t))
    sc = scores_host(d["topk_scores"].index_select(0, tok_t))
    return oracle.routed_experts_nvfp4(x, ids_c, sc, out[0], out[1], gx, gh), tok


def special_weights(E, D, F, seed):
    w13, w2 = W.make_weights(E, D, F, seed)
    w13 = w13.clone()
    w13[0, 0, 0, :32] = 0.0
    w13[0, 1, 1, :16] = -0.0
    w13[0, 0, 2, :16] *= 2.0 ** -20  # tiny blocks: scale 0
    w13[-1, 1, -1, 5] = 3.0  # the tensor's largest magnitude
    w2 = w2.clone()
    w2[0, 0, 16:48] = 0.0
    return w13, w2


@pytest.mark.parametrize("dims", [(3, 384, 256), (2, 256, 384), (1, 128, 128), (4, 640, 1152)])
def test_prepared_weights_bit_exact(dims):
    E, D, F = dims
    w13, w2 = special_weights(E, D, F, 7)
    for which, w in ((W13, w13), (W2, w2)):
        data, scales = binding.moe_nvfp4_prepare_weight(which, w.cuda())
        bits = bf16_bits(w)
        G = oracle.nvfp4_weight_scale(bits)
        codes, sc = oracle.nvfp4_quantize_rows(bits, G)
        sc_host = scales.cpu().numpy()
        assert sc_host[:4].view(np.float32)[0] == np.float32(G), which
        got = unpack(data.cpu().numpy().reshape(-1, (D if which == W13 else F) // 2))
        assert np.array_equal(got, codes.reshape(got.shape)), (which, int((got != codes.reshape(got.shape)).sum()))
        tiled, off = untile_weight_scales(sc_host, which, D, F, E)
        assert np.array_equal(tiled, sc.reshape(tiled.shape)), which
        unused = np.ones(sc_host.size, bool)
        unused[:8] = False  # the tensor scale and its amax
        unused[off.reshape(-1)] = False
        assert not sc_host[unused].any(), "bytes of no row must be 0"


CASES = {
    # name: (T, D, F, E, K, routing)
    "tiny_round_robin": (16, 256, 256, 8, 2, "round_robin"),
    "ragged_multi_tile": (300, 256, 384, 6, 3, "uniform"),  # 2 row tiles per expert; F = 1.5 stages
    "partial_down_tile": (70, 384, 128, 5, 2, "uniform"),  # D tail 0 of 128, F a half stage
    "wide": (96, 640, 512, 4, 2, "uniform"),  # D = 2.5 stages, 5 down tiles
    "many_empty_experts": (20, 128, 128, 64, 2, "uniform"),
    "k1": (129, 128, 256, 3, 1, "uniform"),
    "t1": (1, 256, 128, 8, 4, "uniform"),
    "k_equals_e": (40, 128, 128, 8, 8, "uniform"),
    "k_over_32": (24, 256, 128, 48, 40, "uniform"),  # a token's destination rows in two groups of lanes
    "max_experts": (64, 128, 128, 4096, 4, "uniform"),  # E at its maximum, almost every expert empty
    "skewed_small": (256, 256, 384, 16, 4, "zipf"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_nvfp4_forward_matches_oracle(name):
    T, D, F, E, K, routing = CASES[name]
    d = problem(T, D, F, E, K, routing, seed=3)
    out, ws = run_nv(d)
    assert binding.moe_get_status(ws) == 0
    ref, _ = oracle_nv_tokens(d)
    err = max_rel_err(out.float().cpu().numpy(), ref)
    assert err <= OUT_TOL, (name, err)


def test_nvfp4_every_pair_on_two_experts():
    # experts 0 and E-1 take every pair (six row tiles each, many column tiles and K steps in a
    # row through the same stages and scale slots); the other experts are empty
    T, D, F, E, K = 700, 512, 384, 8, 2
    ids = torch.zeros((T, K), dtype=torch.int32)
    ids[:, 1] = E - 1
    d = problem(T, D, F, E, K, seed=5, ids=ids)
    out, ws = run_nv(d)
    assert binding.moe_get_status(ws) == 0
    ref, _ = oracle_nv_tokens(d)
    err = max_rel_err(out.float().cpu().numpy(), ref)
    assert err <= OUT_TOL, err


@pytest.mark.parametrize("T", [300, 2100])  # 1024-column work items, and whole rows (T >= 2048)
def test_activation_rows_bit_exact_and_padding_scales_zero(T):
    D, F, E, K = 640, 256, 6, 3  # D leaves two padding scale groups per row
    d = problem(T, D, F, E, K, seed=4)
    out, ws = run_nv(d)
    lay = binding.moe_nvfp4_workspace_layout(T, D, F, E, K)
    R = T * K
    rp = 128 * (-(-R // 128) + min(E, R))
    tiles = ws[lay["tiles"]:lay["tiles"] + 4 * (E + 1)].view(torch.int32).cpu().numpy()
    xq = ws[lay["xq"]:lay["xq"] + rp * D // 2].cpu().numpy().reshape(rp, D // 2)
    xs_bytes = rp // 128 * groups(D) * 512
    xs = ws[lay["xs"]:lay["xs"] + xs_bytes].cpu().numpy()
    rt = oracle.routing(d["topk_ids"].cpu().numpy(), E)
    codes, sc = oracle.nvfp4_quantize_rows(bf16_bits(d["x"].cpu()), x_scale_of(d["x"]))
    valid_rows = []
    for e in range(E):
        n = int(rt["counts"][e])
        prows = 128 * int(tiles[e]) + np.arange(n)
        toks = rt["perm"][rt["offsets"][e]:rt["offsets"][e] + n] // K
        assert np.array_equal(unpack(xq[prows]), codes[toks]), e
        assert np.array_equal(untile_act_scales(xs, prows, D), sc[toks]), e
        valid_rows.append(prows)
    used = 128 * int(tiles[E])
    pad = np.setdiff1d(np.arange(used), np.concatenate(valid_rows))
    # padding rows: zero scales (their codes are not written: a zero scale makes them contribute 0)
    assert pad.size > 0 and not untile_act_scales(xs, pad, D).any()
    # the padding scale groups (K values D .. 768) of every used row tile are zero
    grid = xs[:used // 128 * groups(D) * 512].reshape(used // 128, groups(D), 512)
    assert not grid[:, D // 64:].any()


def test_nvfp4_deterministic_stages_and_reusable_workspace():
    T, D, F, E, K = 150, 256, 384, 5, 3
    d = problem(T, D, F, E, K, seed=9)
    nv = prepare(d)
    gx = x_scale_of(d["x"])
    a, ws = run_nv(d, nv)
    b, _ = run_nv(d, nv, workspace=ws)
    assert torch.equal(a, b)
    out = torch.empty_like(a)
    for s in range(binding.MX_STAGES):
        binding.moe_fwd_nvfp4_stages(d["x"], d["topk_ids"], d["topk_scores"], nv[0], nv[1], out, ws, (F, E), gx,
                                     H_SCALE, s, s + 1)
    assert torch.equal(out, a)
    small = problem(9, D, F, E, K, seed=6)
    run_nv(small, workspace=ws)
    c, _ = run_nv(d, nv, workspace=ws)
    assert torch.equal(a, c)


def test_nvfp4_invalid_ids_zero_and_bf16_scores():
    T, D, F, E, K = 64, 256, 128, 5, 3
    d = problem(T, D, F, E, K, seed=8)
    nv = prepare(d)
    ids = d["topk_ids"].clone()
    ids[::3, 1] = -1
    ids[1::7, 2] = E + 2
    dropped = dict(d, topk_ids=ids)
    out, ws = run_nv(dropped, nv)
    assert binding.moe_get_status(ws) & binding.MOE_DEV_BAD_EXPERT_ID
    ref, _ = oracle_nv_tokens(dropped)
    assert max_rel_err(out.float().cpu().numpy(), ref) <= OUT_TOL
    sc = d["topk_scores"].clone()
    sc[(ids < 0) | (ids >= E)] = 0.0
    zero, _ = run_nv(dict(d, topk_scores=sc), nv)
    assert torch.equal(zero, out)
    sb = d["topk_scores"].to(torch.bfloat16)
    outb, _ = run_nv(dict(d, topk_scores=sb), nv)
    refb, _ = oracle_nv_tokens(dict(d, topk_scores=sb))
    assert max_rel_err(outb.float().cpu().numpy(), refb) <= OUT_TOL


# sampled tokens beyond the first and last; the oracle quantizes every expert they touch
@pytest.mark.parametrize("name,ntok", [("medium", 10), ("decode", 1), ("skewed", 2), ("large", 0)])
def test_nvfp4_full_size_sampled_tokens(name, ntok):
    d = W.make_inputs(name, seed=0, device="cuda")
    T = d["workload"].T
    out, ws = run_nv(d)
    assert binding.moe_get_status(ws) == 0
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, ntok, replace=False)]))
    ref, tok = oracle_nv_tokens(d, tokens)
    err = max_rel_err(out.float().cpu().numpy()[tok], ref)
    assert err <= OUT_TOL, err
