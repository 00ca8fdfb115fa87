"""The multi-rank path of bench.py on CPU: two gloo ranks, no GPU.

With N GPUs the bench runs N independent layer replicas (the layer forward
has no cross-GPU exchange); each rank draws its own inputs, the job time is
the slowest rank's and the throughput counts every rank's tokens.
"""
import os
import time
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import moe_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = moe_inputs.WORKLOADS["tiny_fp32"]
        rep = bench.replica_workload(wl, rank)
        inp = moe_inputs.make_inputs(rep, device="cpu")
        # per-rank times 3.0 and 5.0 ms: every rank sees the slowest
        t_max = bench.max_over_ranks(3.0 + 2.0 * rank, world, "cpu")
        out[rank] = (rep.seed, float(inp.x.sum()), t_max,
                     bench.job_tokens_per_s(wl.T, world, 10, t_max))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_slowest_rank_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    wl = moe_inputs.WORKLOADS["tiny_fp32"]
    (s0, x0, t0, v0), (s1, x1, t1, v1) = res[0], res[1]
    assert (s0, s1) == (wl.seed, wl.seed + 1000)
    assert x0 != x1  # independent replicas draw different inputs
    assert t0 == t1 == 5.0
    assert v0 == v1 == pytest.approx(2 * wl.T * 10 / 5.0e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25
    assert bench.job_tokens_per_s(4096, 1, 20, 4.0) == pytest.approx(4096 * 20 / 4.0e-3)


def test_reference_arm_prints_its_contract_line():
    # the oracle arm on the smallest workload: one JSON line with the keys the
    # benchmark contract names, and no copies in its e2e object
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    t0 = time.perf_counter()
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32", "--steps",
                          "2", "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=300)
    wall_s = time.perf_counter() - t0
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["higher_is_better"] is True and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"]
    # the measured wall time per step: the timed steps fit in the process's run
    assert 0 < line["steps"] * line["ms_per_step"] * 1e-3 < wall_s
    assert line["extrapolated_ms_per_layer"] > 0
    # the same config object as the GPU arm prints for this workload
    import bench
    wl = bench.moe_inputs.WORKLOADS["tiny_fp32"]
    import oracle
    C = oracle.capacity(wl.T, wl.k, wl.E, wl.D, wl.capacity_factor)[0]
    assert line["config"] == bench.workload_config(wl, C, line["config"]["kept"], line["config"]["dropped"], 1)
    assert line["config"]["kept"] + line["config"]["dropped"] == wl.T * wl.k
