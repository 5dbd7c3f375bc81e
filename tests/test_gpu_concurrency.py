"""Two calls at once: one workspace serves one call in flight, but calls on different workspaces
share nothing, so they may run concurrently on different streams (and CPU threads). Each must give
the bits it gives alone."""

import threading

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


@pytest.mark.parametrize("entry", ["staged", "mega"])
def test_concurrent_calls_on_separate_workspaces(entry):
    # mega: two fused grids share the SMs; a grid's down tiles wait only for tiles its own running
    # CTAs claimed, so each finishes whatever the other holds
    T, D, F, E, K = (512, 512, 384, 8, 4) if entry == "staged" else (2048, 256, 1024, 32, 6)
    fwd = binding.moe_routed_experts_fwd if entry == "staged" else binding.moe_routed_experts_fwd_mega
    nbytes = (binding.moe_workspace_bytes if entry == "staged" else binding.moe_mega_workspace_bytes)(T, D, F, E, K)
    probs = [problem(T, D, F, E, K, seed) for seed in (21, 22)]
    wss = [binding.alloc_workspace(nbytes) for _ in probs]
    alone = []
    for d, ws in zip(probs, wss):
        out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
        fwd(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], d["w2"], out, ws)
        alone.append(out)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in probs]
    outs = [torch.empty_like(a) for a in alone]
    errors = []

    def run(i):
        try:
            d = probs[i]
            with torch.cuda.stream(streams[i]):
                for _ in range(5):
                    fwd(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], d["w2"], outs[i], wss[i],
                        stream=streams[i])
        except Exception as exc:  # surfaced below, on the main thread
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(probs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for out, want, ws in zip(outs, alone, wss):
        assert torch.equal(out, want)
        assert binding.moe_get_status(ws) == 0
