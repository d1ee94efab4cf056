"""Host-side logic of bench.py on CPU: the multi-rank timing reduction with a
gloo process group (world size 2), the kernel-source fingerprint that gates a
profiled traffic figure, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo")
    bench.barrier(world)
    slowest = bench.max_over_ranks(1.0 + rank, world, "cpu")
    out.put((rank, slowest))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.0), (1, 2.0)]


def test_traffic_gated_by_kernel_fingerprint(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_sources_sha("bf16")
    assert sha != bench.kernel_sources_sha("mxfp8")
    (prof / "fwd_bf16_w.md").write_text(f"workload: w\nkernel_kind: bf16\nkernel_sources_sha: {sha}\n"
                                        "dram_bytes_per_launch: 1.5e8\n")
    # a summary of another workload whose name ends the same way is not taken
    (prof / "bwd_bf16_bwd_w.md").write_text(f"workload: bwd_w\nkernel_kind: bf16\nkernel_sources_sha: {sha}\n"
                                            "dram_bytes_per_launch: 9.9e8\n")
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda kind="bf16": sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("w") == 1.5e8
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda kind="bf16": "abc")
    assert bench.profiled_traffic("w") is None  # taken on other kernel sources



def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_b1h2n256d64", "--steps", "1", "--warmup", "3", "--reference-seconds", "0.5"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_json_line_backward():
    # the backward workload's reference arm times the float64 backward oracle on one head
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--shape",
                        "1,1,512,64,1,0,1", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"].startswith("attention bwd") and line["value"] > 0
    assert line["config"]["pass"] == "bwd" and line["config"]["causal"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and "backward" in line["cpu_baseline"]["sample"]



def test_reference_arm_json_line_mxfp8_backward():
    # the MXFP8 backward's reference arm times the float64 MXFP8 backward oracle on one head
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--shape",
                        "1,1,256,128,0,1,1", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"].startswith("attention bwd") and line["value"] > 0
    assert line["config"]["pass"] == "bwd" and line["config"]["dtype"] == "mxfp8"
    assert line["cpu_baseline"]["kind"] == "oracle" and "MXFP8 backward" in line["cpu_baseline"]["sample"]
