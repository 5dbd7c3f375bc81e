"""Failure detection on the GPU without a fault: a bounded wait that cannot be satisfied must end
with MOE_DEV_TIMEOUT in the status word, and the CUDA context must stay usable afterwards."""

import time

import pytest
import torch

from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    binding.moe_selftest_wait_timeout(50_000, status)  # 50 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == binding.MOE_DEV_TIMEOUT
    assert 0.04 < elapsed < 5.0
    # the context is still healthy: a normal forward pass runs and reports no error
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in W.make_inputs("tiny").items()}
    T, D = d["x"].shape
    E, _, F, _ = d["w13"].shape
    ws = binding.alloc_workspace(binding.moe_workspace_bytes(T, D, F, E, 2), "cuda")
    out = torch.empty_like(d["x"])
    binding.moe_routed_experts_fwd(d["x"], d["topk_ids"], d["topk_scores"], d["w13"], d["w2"], out, ws)
    assert binding.moe_get_status(ws) == 0
    assert torch.isfinite(out.float()).all()


def test_selftest_rejects_bad_arguments():
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MoeError):
        binding.moe_selftest_wait_timeout(0, status)
    with pytest.raises(binding.MoeError):
        binding.moe_selftest_wait_timeout(3_000_000, status)
