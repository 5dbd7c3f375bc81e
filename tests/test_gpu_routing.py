"""Routing on the GPU (histogram, scan, stable permutation) against the oracle: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routed_topk_gb300 import binding
from mixture_experts_routed_topk_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def gpu_routing(ids: torch.Tensor, E: int):
    T, K = ids.shape
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * K, dtype=torch.int32, device=dev)
    inv = torch.empty(T * K, dtype=torch.int32, device=dev)
    ws = binding.alloc_workspace(binding.moe_routing_workspace_bytes(T, E, K), dev)
    binding.moe_routing(ids, E, counts, offsets, perm, inv, ws)
    bits = binding.moe_get_status(ws)
    return {"counts": counts.cpu().numpy(), "offsets": offsets.cpu().numpy(), "perm": perm.cpu().numpy(),
            "inv": inv.cpu().numpy(), "bits": bits}


def assert_routing_equal(got, ref):
    for key in ("counts", "offsets", "perm", "inv"):
        assert np.array_equal(got[key], ref[key]), key


@pytest.mark.parametrize("name", ["tiny", "medium", "decode", "large", "skewed"])
def test_routing_workloads_bit_exact(name):
    wl = W.WORKLOADS[name]
    ids = W.make_topk_ids(wl.T, wl.E, wl.K, wl.routing, seed=0)
    got = gpu_routing(ids.cuda(), wl.E)
    ref = oracle.routing(ids.numpy(), wl.E)
    assert_routing_equal(got, ref)
    assert got["bits"] == 0
    if name == "tiny":
        assert np.all(got["counts"] == 4)


@pytest.mark.parametrize(
    "T,E,K,lo,hi",
    [
        (1, 1, 1, 0, 1),
        (1, 8, 4, 0, 8),
        (5000, 1, 3, 0, 1),  # one expert takes every pair
        (1023, 4096, 2, 0, 4096),  # E at its maximum, most experts empty
        (3000, 37, 9, 0, 37),  # duplicates within tokens, ragged block tail
        (2049, 16, 1, 0, 16),  # R one past a routing block
        (777, 12, 5, -3, 15),  # invalid ids on both sides
    ],
)
def test_routing_edge_cases_bit_exact(T, E, K, lo, hi):
    g = torch.Generator().manual_seed(T * 31 + E)
    ids = torch.randint(lo, hi, (T, K), generator=g, dtype=torch.int32)
    got = gpu_routing(ids.cuda(), E)
    ref = oracle.routing(ids.numpy(), E)
    assert_routing_equal(got, ref)
    assert (got["bits"] & binding.MOE_DEV_BAD_EXPERT_ID != 0) == (ref["n_invalid"] > 0)


def test_routing_empty_is_noop():
    ids = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(256, "cuda")
    z = torch.empty(0, dtype=torch.int32, device="cuda")
    binding.moe_routing(ids, 8, torch.empty(8, dtype=torch.int32, device="cuda"),
                        torch.empty(9, dtype=torch.int32, device="cuda"), z, z, ws)


@pytest.mark.parametrize("short", ["counts", "offsets", "perm", "inv"])
def test_binding_rejects_short_routing_outputs(short):
    # outputs too small for what the kernels write are refused before anything is enqueued
    T, E, K = 100, 16, 4
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    sizes = {"counts": E, "offsets": E + 1, "perm": T * K, "inv": T * K}
    sizes[short] -= 1
    outs = [torch.zeros(sizes[n], dtype=torch.int32, device="cuda") for n in ("counts", "offsets", "perm", "inv")]
    ws = binding.alloc_workspace(binding.moe_routing_workspace_bytes(T, E, K), "cuda")
    with pytest.raises(ValueError, match=short):
        binding.moe_routing(ids, E, *outs, ws)
    with pytest.raises(ValueError, match=short):
        binding.moe_routing_static_scratch(ids, E, *outs)


def test_binding_rejects_short_status_word():
    status = torch.zeros(3, dtype=torch.uint8, device="cuda")  # the library writes a whole uint32
    with pytest.raises(ValueError, match="device_status"):
        binding.moe_selftest_wait_timeout(10, status)
