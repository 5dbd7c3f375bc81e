"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and evaluate the oracle
on exactly the same inputs (copied to the host), whole or on a subset of tokens / pairs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from common import bf16_bits
from mixture_experts_routed_topk_gb300 import binding

OUT_TOL = 1e-2  # max|out - ref| / max|ref|, bf16 I/O with fp32 accumulation


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_fwd(d: dict, workspace=None, stream=None):
    """The whole forward pass through moe_routed_experts_fwd. Returns (out, workspace)."""
    x, ids, w13 = d["x"], d["topk_ids"], d["w13"]
    T, D = x.shape
    E, _, F, _ = w13.shape
    K = ids.shape[1]
    if workspace is None:
        workspace = binding.alloc_workspace(binding.moe_workspace_bytes(T, D, F, E, K), x.device)
    out = torch.empty((T, D), dtype=torch.bfloat16, device=x.device)
    binding.moe_routed_experts_fwd(x, ids, d["topk_scores"], w13, d["w2"], out, workspace, stream=stream)
    return out, workspace


def workspace_view(ws: torch.Tensor, dims, region: str, dtype, count: int) -> torch.Tensor:
    lay = binding.moe_workspace_layout(*dims)
    off = lay[region]
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def scores_host(scores: torch.Tensor) -> np.ndarray:
    s = scores.detach().cpu()
    if s.dtype == torch.bfloat16:
        return bf16_bits(s)
    return s.numpy().astype(np.float32)


def oracle_tokens(d: dict, tokens=None) -> tuple[np.ndarray, np.ndarray]:
    """Oracle out (fp32) for the given tokens (all when None). Only the experts those tokens touch
    are copied to the host; ids are renumbered into that compact set (ids outside [0, E) -> -1)."""
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
    w13 = bf16_bits(d["w13"].index_select(0, ex_t))
    w2 = bf16_bits(d["w2"].index_select(0, ex_t))
    x = bf16_bits(d["x"].index_select(0, tok_t))
    sc = scores_host(d["topk_scores"].index_select(0, tok_t))
    return oracle.routed_experts(x, ids_c, sc, w13, w2), tok


def oracle_pairs(d: dict, pairs) -> np.ndarray:
    """Oracle score * y for each flat pair p = t*K + k (K = 1 problems, one row per pair)."""
    ids_all = d["topk_ids"]
    K = ids_all.shape[1]
    pairs = np.asarray(pairs, dtype=np.int64)
    flat_ids = ids_all.reshape(-1).index_select(0, torch.from_numpy(pairs).to(ids_all.device)).cpu().numpy()
    flat_sc = d["topk_scores"].reshape(-1).index_select(0, torch.from_numpy(pairs).to(ids_all.device))
    sub = {
        "x": d["x"].index_select(0, torch.from_numpy(pairs // K).to(d["x"].device)),
        "topk_ids": torch.from_numpy(flat_ids.reshape(-1, 1).astype(np.int32)).to(ids_all.device),
        "topk_scores": flat_sc.reshape(-1, 1),
        "w13": d["w13"],
        "w2": d["w2"],
    }
    out, _ = oracle_tokens(sub)
    return out


def oracle_routing_of(d: dict) -> dict:
    return oracle.routing(d["topk_ids"].cpu().numpy(), d["w13"].shape[0])
