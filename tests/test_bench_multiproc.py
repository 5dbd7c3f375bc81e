"""The benchmark's multi-rank host logic on CPU: two gloo ranks, barrier, max over ranks, seeds."""

import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, lr = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    got = bench.reduce_max(dist, float(10 + 5 * r))
    seed = bench.replica_seed(7, r)
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as fh:
        json.dump({"rank": r, "world": w, "local": lr, "max": got, "seed": seed}, fh)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["world"] == 2 for r in res)
    assert all(r["max"] == 15.0 for r in res)  # the max over ranks reaches every rank
    assert res[0]["seed"] != res[1]["seed"]  # each replica draws its own tokens


def test_single_process_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_init(1, "gloo") is None
    assert bench.reduce_max(None, 3.5) == 3.5
    args = bench.parse_args([])
    assert args.gpus == 1 and args.config == "large" and args.impl == "ours" and args.warmup >= 3
    assert bench.extra_workloads(args) == ["decode", "medium"]
    assert bench.extra_workloads(bench.parse_args(["--experts", "16", "--config", "decode"])) == []


def test_roofline_arithmetic():
    sys.path.insert(0, ROOT)
    import bench

    peaks = {"hbm_gbs": 6790.0, "bf16_tflops": 1926.5, "bf16_tflops_sustained": 1735.9}
    costs = bench.kernel_costs(4096, 2048, 1408, 64, 6, 64)
    # gemm1: 4 R D F flops; compute bound at this size
    r = bench.roofline_entry("gemm1_swiglu", costs, 1e-4, peaks, False, None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 4 * 4096 * 6 * 2048 * 1408 / 1e-4 / 1e12) < 0.1
    assert abs(r["frac"] - r["achieved"] / 1926.5) < 1e-3
    c = bench.roofline_entry("combine", costs, 1e-4, peaks, False, None)
    assert c["bound"] == "hbm" and c["unit"] == "GB/s"
    flops, nbytes = bench.path_costs(4096, 2048, 1408, 64, 6, 64)
    assert flops == 6 * 4096 * 6 * 2048 * 1408
    assert nbytes == 64 * 3 * 1408 * 2048 * 2 + 2 * 4096 * 2048 * 2 + 4096 * 6 * 8
    # the intermediates' round trips reported beside the result (large workload: 3.76 / 1.07 /
    # 3.76 GB for XP, H and Y)
    ov = bench.overhead_bytes(16384, 7168, 2048, 8)
    assert ov == {"xp": 2 * 131072 * 7168 * 2, "h": 2 * 131072 * 2048 * 2, "y": 2 * 131072 * 7168 * 2}
    assert abs(ov["xp"] / 1e9 - 3.76) < 0.01 and abs(ov["h"] / 1e9 - 1.07) < 0.01
    # fused GEMMs: 6 R D F flops, H stays inside the kernel
    fused = costs["fused_gemms"]
    assert fused["flops"] == costs["gemm1_swiglu"]["flops"] + costs["gemm2_score"]["flops"]


@pytest.mark.parametrize("precision", ["bf16", "mxfp8", "nvfp4"])
def test_reference_arm_line(precision):
    # the reference arm times the CPU oracle; on the tiny workload it needs no GPU and ends in seconds
    import subprocess

    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--precision", precision, "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "tiny" and line["config"]["precision"] == precision


def test_backward_stage_costs_add_up():
    sys.path.insert(0, ROOT)
    import bench

    T, D, F, E, K = 4096, 2048, 1408, 64, 6
    costs = bench.bwd_stage_costs(T, D, F, E, K, 64)
    R = T * K
    assert sum(c["flops"] for c in costs.values()) == 16 * R * D * F  # the whole call's flops
    assert [s for s in costs if costs[s]["flops"] == 0] == ["dispatch", "reduce"]
    # the weight-gradient GEMMs write every expert's gradient once
    assert costs["wgrad_down"]["bytes"] >= E * D * F * 2 and costs["wgrad_gate_up"]["bytes"] >= E * 2 * F * D * 2


def test_recorded_traffic_scales_a_cut_capture(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.md").write_text(
        "| config | kernel | source hash | traffic | read | write | experts touched | note |\n|---|---|---|---|---|---|---|---|\n"
        "| medium | gemm1_swiglu | 0123456789abcdef | 1000 | 900 | 100 | 64 | x |\n"
        "| decode (E=16) | gemm1_swiglu | 0123456789abcdef | 1600 | 1500 | 100 | 16 | y |\n"
        "| decode | gemm2_score | ffffffffffffffff | 5 | 4 | 1 | 16 | stale |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0123456789abcdef")
    assert bench.recorded_traffic("medium", "gemm1_swiglu", 64) == 1000.0
    assert bench.recorded_traffic("decode", "gemm1_swiglu", 222) == 1600 * 222 // 16  # scaled by touched experts
    assert bench.recorded_traffic("decode", "gemm2_score", 222) is None  # taken on other sources
