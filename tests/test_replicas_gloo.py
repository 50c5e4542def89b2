"""The N > 1 host path of the bench, on CPU with two gloo ranks.

Rows are independent, so N GPUs run N replicas (each rank its own batch, no
collective on the data path); only the timing crosses ranks: a barrier around
the timed region and the maximum of the ranks' times.  This runs that host
logic with world_size 2 on CPU.
"""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import far_gen


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # each rank its own batch: seed = rank, as the bench does
        d = far_gen.make_inputs("c1", seed=rank)
        digest = float(d["x"].float().sum())
        # the slowest rank's time is the job's time
        t = bench.max_over_ranks(1.0 + rank * 0.5, dist, torch.device("cpu"))
        dist.barrier()
        results[rank] = (digest, t, bench.job_rate(100.0, world, t * 1e3))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    (d0, t0, v0), (d1, t1, v1) = res[0], res[1]
    assert d0 != d1                      # different batches on the two replicas
    assert t0 == t1 == 1.5               # both see the slower rank's time
    assert v0 == v1 == 100.0 * 2 / 1.5   # whole-job units per second


def test_single_process_path():
    assert bench.max_over_ranks(3.25, None, None) == 3.25
    assert bench.job_rate(10.0, 1, 2.0) == 5000.0


def test_traffic_record_matches_the_current_plans():
    """The DRAM bytes the bench reports as `traffic` come from committed ncu captures; each
    record names the kernel-source hash and the launch plan it was taken with. The record
    must match the sources and the plan the planner picks today on a 152-SM GB300, and the
    lookup must refuse another plan or token count."""
    import json

    import mixed_precision_residual_gb300 as far

    with open(bench.TRAFFIC_FILE) as f:
        d = json.load(f)
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}
    cases = {"c5": ("f16", 8192, far.plan_for_sms), "c5:layernorm": ("f16", 8192, far.plan_ln_for_sms),
             "c4": ("bf16", 5120, far.plan_for_sms)}
    for key, (act, hidden, planner) in cases.items():
        e = d[key]
        assert e["source_hash"] == bench.source_hash(), key
        p = planner(e["captured_tokens"], hidden, dt[act], dt[act], True, 152)
        assert e["launch_plan"] == [p[k] for k in bench.PLAN_KEYS], (key, p)
        assert e["dram_bytes_per_launch"] == e["captured_read_bytes"] + e["captured_write_bytes"]
        workload, _, op = key.partition(":")
        op = op or "rmsnorm"
        assert bench.traffic_from_profile(workload, op, p, e["captured_tokens"]) == e["dram_bytes_per_launch"]
        other = dict(p, groups=p["groups"] + 1)
        assert bench.traffic_from_profile(workload, op, other, e["captured_tokens"]) is None
        assert bench.traffic_from_profile(workload, op, p, e["captured_tokens"] // 2) is None
