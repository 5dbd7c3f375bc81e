"""moe_routing_static_scratch: routing for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace -- their device memory is all owned by another
allocator, or they are plain host programs with no allocator at hand. This entry point keeps its
scratch in a fixed array inside the library instead. Its results must equal the CPU oracle's
routing (counts, offsets and the stable permutation are unique, so bit for bit) and moe_routing's
(the workspace entry point), including when it is called twice in a row on the shared array, which
keeps the previous call's contents. This file sorts last so that a run stopping at its first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import oracle
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


def with_static_scratch(ids, E, pass_status=True):
    T, K = ids.shape
    out = routing_outputs(T, E, K)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda") if pass_status else None
    binding.moe_routing_static_scratch(ids, E, *out, device_status=status)
    torch.cuda.synchronize()
    return out, (int(status.item()) if pass_status else None)


def check_against_oracle(got, ids, E):
    ref = oracle.routing(ids.cpu().numpy(), E)
    for a, name in zip(got, ("counts", "offsets", "perm", "inv")):
        np.testing.assert_array_equal(a.cpu().numpy(), ref[name], err_msg=name)
    return ref["n_invalid"]


@pytest.mark.parametrize("T,E,K,lo,hi", [(3000, 37, 5, 0, 37), (16384, 256, 8, -2, 258)])
def test_static_scratch_matches_oracle_and_workspace_routing_twice(T, E, K, lo, hi):
    for call in range(2):  # the second call runs on the array the first one left behind
        g = torch.Generator().manual_seed(100 * call + E)
        ids = torch.randint(lo, hi, (T, K), generator=g, dtype=torch.int32).cuda()
        got, got_bits = with_static_scratch(ids, E)
        n_invalid = check_against_oracle(got, ids, E)
        assert got_bits == (binding.MOE_DEV_BAD_EXPERT_ID if n_invalid else 0)
        ref, ref_bits = with_workspace(ids, E)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert got_bits == ref_bits


def test_static_scratch_without_status_word_twice():
    # device_status = NULL: the status word lives in the library's array. A first call with ids out
    # of range leaves its bit there; the second call (valid ids) must clear it and still route right.
    T, E, K = 5000, 64, 6
    g = torch.Generator().manual_seed(7)
    bad = torch.randint(-3, E + 3, (T, K), generator=g, dtype=torch.int32).cuda()
    good = torch.randint(0, E, (T, K), generator=g, dtype=torch.int32).cuda()
    for ids in (bad, good):
        got, _ = with_static_scratch(ids, E, pass_status=False)
        check_against_oracle(got, ids, E)
        ref, _ = with_workspace(ids, E)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_static_scratch_rejects_sizes_beyond_its_capacity():
    E, K = 4096, 8
    T = 70_000  # (E + 1) * ceil(T*K / 2048) = 4097 * 274 > MOE_STATIC_SCRATCH_MAX_ENTRIES = 262144
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.MoeError) as err:
        binding.moe_routing_static_scratch(ids, E, *routing_outputs(T, E, K))
    assert err.value.status == 2  # MOE_ERR_UNSUPPORTED_SHAPE
