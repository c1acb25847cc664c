"""bench.py's CPU-baseline leg on the CPU: it times the oracle on all host cores
and, given the GPU run's outputs, reports their parity over every sequence.
Here the 'GPU outputs' are planted on the CPU."""
import numpy as np
import torch

import bench
from oracle import gqa_paged_decode_oracle
from paged_kv_gqa_split_gb300 import workloads as wl


def test_cpu_baseline_parity_accepts_match_and_flags_error(monkeypatch):
    monkeypatch.setattr(bench, "ORACLE_TARGET_CPU_S", 0.01)
    w = wl.make_config("tiny")
    o, l = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    out = torch.from_numpy(o).to(torch.bfloat16)
    lse = torch.from_numpy(l).to(torch.float32)
    base, par = bench.cpu_baseline(w, out, lse)
    assert base["kind"] == "oracle" and base["value"] > 0 and base["cores"] >= 1
    assert base["cores"] <= base["host_cores_available"]
    assert par["within_tolerance"] and par["sequences"] == w.batch
    bad = out.clone()
    first = next(b for b in range(w.batch) if w.lens[b] > 0)
    bad[first, 3, 7] += 1.0                       # an error far outside the tolerance
    _, par_bad = bench.cpu_baseline(w, bad, lse)
    assert not par_bad["within_tolerance"]
    assert np.isfinite(par_bad["max_abs_dO"])


def test_replica_value_counts_every_rank_over_the_slowest():
    assert bench.replica_value(10**9, 1.0, 1) == 1000.0
    assert bench.replica_value(10**9, 2.0, 4) == 2000.0
