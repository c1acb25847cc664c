"""Multi-rank bench logic on the CPU (gloo, world size 2): with N replicas the step
time reported is the max over ranks, so the slowest replica sets the number."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        bench.barrier(world)
        out[rank] = bench.max_over_ranks(1.5 + 2.0 * rank, world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    world = 2
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.25, 1) == 2.25
    bench.barrier(1)


def _replica_worker(rank, world, port, out):
    """Each rank decodes its own replica of the tiny workload (the float64 oracle on the
    host: the data path has no collective), then the ranks agree on the step time."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import time

    import numpy as np
    import torch
    import torch.distributed as dist

    import bench
    from oracle import gqa_paged_decode_oracle
    from paged_kv_gqa_split_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = wl.make_config("tiny")
        t0 = time.perf_counter()
        o, lse = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
        ms = (time.perf_counter() - t0) * 1e3 + 10.0 * rank  # the second rank is made the slower one
        digest = torch.tensor([float(np.nansum(o)), float(np.nansum(np.where(np.isfinite(lse), lse, 0.0)))],
                              dtype=torch.float64)
        got = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(got, digest)
        ms_max = bench.max_over_ranks(ms, world)
        out[rank] = (bool(all(torch.equal(g, got[0]) for g in got)), ms_max,
                     bench.replica_value(bench.counted_bytes(w.lens), ms_max, world), ms)
    finally:
        dist.destroy_process_group()


def test_replicas_gloo_two_ranks():
    """Replicas compute identical results; the job's value is all ranks' bytes over the slowest rank's time."""
    import bench
    from paged_kv_gqa_split_gb300 import workloads as wl
    ctx = mp.get_context("spawn")
    world = 2
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_replica_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                           join=True)
        res = dict(out)
    assert res[0][0] and res[1][0]
    assert res[0][1] == res[1][1] == max(res[0][3], res[1][3])
    b = bench.counted_bytes(wl.make_config("tiny").lens)
    assert res[0][2] == pytest.approx(2 * b / (res[0][1] * 1e-3) / 1e9)


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched under torch.distributed.run with N = 2: rank 0 alone prints
    one line (the oracle on the host's cores); the other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
