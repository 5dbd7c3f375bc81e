"""The forward passes inside a CUDA graph: no entry point allocates, synchronises or reads device
data on the host, so a whole forward call can be captured on a stream and replayed. Each replay
must give the bits an eager call gives, for inputs refreshed in place between replays."""

import pytest
import torch

from gpu_common import to_device
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def problem(T, D, F, E, K, seed):
    d = {"x": W.make_x(T, D, seed), "topk_ids": W.make_topk_ids(T, E, K, "uniform", seed),
         "topk_scores": W.make_scores(T, K, "softmax", seed)}
    d["w13"], d["w2"] = W.make_weights(E, D, F, seed)
    return to_device(d)


@pytest.mark.parametrize("precision", ["bf16", "mega", "mxfp8", "nvfp4"])
def test_forward_replays_from_a_cuda_graph(precision):
    T, D, F, E, K = 200, 256, 384, 6, 3
    d = problem(T, D, F, E, K, seed=11)
    other = to_device({"x": W.make_x(T, D, 12), "topk_ids": W.make_topk_ids(T, E, K, "uniform", 12),
                       "topk_scores": W.make_scores(T, K, "softmax", 12)})  # other tokens, same weights
    x, ids, sc = d["x"].clone(), d["topk_ids"].clone(), d["topk_scores"].clone()
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    if precision == "bf16":
        ws = binding.alloc_workspace(binding.moe_workspace_bytes(T, D, F, E, K))
        call = lambda s: binding.moe_routed_experts_fwd(x, ids, sc, d["w13"], d["w2"], out, ws, stream=s)
    elif precision == "mega":  # the fused forward: one dynamically scheduled grid for both GEMMs
        ws = binding.alloc_workspace(binding.moe_mega_workspace_bytes(T, D, F, E, K))
        call = lambda s: binding.moe_routed_experts_fwd_mega(x, ids, sc, d["w13"], d["w2"], out, ws, stream=s)
    elif precision == "mxfp8":
        w13 = binding.moe_mxfp8_prepare_weight(binding.MOE_WEIGHT_W13, d["w13"])
        w2 = binding.moe_mxfp8_prepare_weight(binding.MOE_WEIGHT_W2, d["w2"])
        ws = binding.alloc_workspace(binding.moe_mxfp8_workspace_bytes(T, D, F, E, K))
        call = lambda s: binding.moe_routed_experts_fwd_mxfp8(x, ids, sc, w13, w2, out, ws, (F, E), stream=s)
    else:
        w13 = binding.moe_nvfp4_prepare_weight(binding.MOE_WEIGHT_W13, d["w13"])
        w2 = binding.moe_nvfp4_prepare_weight(binding.MOE_WEIGHT_W2, d["w2"])
        ws = binding.alloc_workspace(binding.moe_nvfp4_workspace_bytes(T, D, F, E, K))
        call = lambda s: binding.moe_routed_experts_fwd_nvfp4(x, ids, sc, w13, w2, out, ws, (F, E), 2.0 ** -9,
                                                              2.0 ** -8, stream=s)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        call(stream)  # eager, once, outside the capture (per-device set-up happens here)
    stream.synchronize()
    eager_a = out.clone()
    x.copy_(other["x"]), ids.copy_(other["topk_ids"]), sc.copy_(other["topk_scores"])
    with torch.cuda.stream(stream):
        call(stream)
    stream.synchronize()
    eager_b = out.clone()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call(stream)
    for src, want in ((d, eager_a), (other, eager_b), (d, eager_a)):
        x.copy_(src["x"]), ids.copy_(src["topk_ids"]), sc.copy_(src["topk_scores"])
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert binding.moe_get_status(ws) == 0
