"""moe_routing_static_scratch: routing for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace -- their device memory is all owned by another
allocator, or they are plain host programs with no allocator at hand. This entry point keeps its
scratch in a fixed array inside the library instead. Its results must equal moe_routing's (the
workspace entry point) bit for bit, including when it is called twice in a row on the shared
array, which keeps the previous call's contents. This file sorts last so that a run stopping at
its first failure has already run every other test.
"""

import pytest
import torch

from mixture_experts_routed_topk_gb300 import binding

pytestmark = pytest.mark.gpu


def routing_outputs(T, E, K):
    dev = "cuda"
    return (torch.full((E,), -7, dtype=torch.int32, device=dev), torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((T * K,), -7, dtype=torch.int32, device=dev), torch.full((T * K,), -7, dtype=torch.int32, device=dev))


def with_workspace(ids, E):
    T, K = ids.shape
    out = routing_outputs(T, E, K)
    ws = binding.alloc_workspace(binding.moe_routing_workspace_bytes(T, E, K), "cuda")
    binding.moe_routing(ids, E, *out, ws)
    return out, binding.moe_get_status(ws)


def with_static_scratch(ids, E):
    T, K = ids.shape
    out = routing_outputs(T, E, K)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    binding.moe_routing_static_scratch(ids, E, *out, device_status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


@pytest.mark.parametrize("T,E,K,lo,hi", [(3000, 37, 5, 0, 37), (16384, 256, 8, -2, 258)])
def test_static_scratch_matches_workspace_routing_twice(T, E, K, lo, hi):
    for call in range(2):  # the second call runs on the array the first one left behind
        g = torch.Generator().manual_seed(100 * call + E)
        ids = torch.randint(lo, hi, (T, K), generator=g, dtype=torch.int32).cuda()
        ref, ref_bits = with_workspace(ids, E)
        got, got_bits = with_static_scratch(ids, E)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert got_bits == ref_bits


def test_static_scratch_rejects_sizes_beyond_its_capacity():
    E, K = 4096, 8
    T = 70_000  # (E + 1) * ceil(T*K / 2048) = 4097 * 274 > MOE_STATIC_SCRATCH_MAX_ENTRIES = 262144
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MoeError) as err:
        binding.moe_routing_static_scratch(ids, E, *routing_outputs(T, E, K))
    assert err.value.status == 2  # MOE_ERR_UNSUPPORTED_SHAPE
