"""The N > 1 host logic of bench.py on CPU: replicas timed as the slowest rank, whole-job
throughput, and the reference arm printing on rank 0 only.  Two gloo ranks, no GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 37.5 * rank                 # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, world, "cpu")
        q.put((rank, total, bench.job_throughput(world, 32768, 20, total)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_job_by_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [137.5, 137.5]                  # both ranks see the slowest time
    assert res[0][2] == pytest.approx(2 * 32768 * 20 / 0.1375)    # tokens of both replicas / job time


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_throughput(1, 100, 4, 2000.0) == pytest.approx(200.0)


def _reference_arm(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "0",
                           "--steps", "1", "--warmup", "0", "--gpus", "2"], capture_output=True, text=True,
                          env=env, timeout=600)


def test_reference_arm_prints_on_rank_zero_only():
    r1 = _reference_arm(1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _reference_arm(0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["n_gpus"] == 2


def test_layer_roofline_fraction_of_the_step():
    """The layer's fraction of roofline is the sum of the stages' roofline times over the sum of their measured
    times; stages measured at their roofline give 1, and the headline workload's roofline time is the sparse
    MLA's bf16 FLOPs plus the scoring's FP8 FLOPs plus three HBM-bound stages."""
    from pooled_key_dsa_gb300 import workloads
    wl = workloads.workload(3)
    work = bench._work(wl)
    peaks = {"hbm_gbs": 6000.0, "bf16": 1700.0, "bf16_sustained": 1500.0, "source": "test"}
    first = bench.layer_roofline(wl, work, {k: 1.0 for k in ("kpool_build", "hadamard_fp8", "score", "select",
                                                              "sparse_mla")}, peaks, 3400.0)
    r = first["t_roof_ms"]
    assert abs(r["sparse_mla"] - work["mla_flops"] / 1700e12 * 1e3) < 1e-12
    assert abs(r["score"] - work["score_flops"] / 3400e12 * 1e3) < 1e-12
    assert abs(r["select"] - 4.0 * wl.T * wl.W / 6000e9 * 1e3) < 1e-12
    at_roof = bench.layer_roofline(wl, work, dict(r), peaks, 3400.0)
    assert abs(at_roof["frac"] - 1.0) < 1e-12
    assert abs(first["frac"] - sum(r.values()) / 5.0) < 1e-12
