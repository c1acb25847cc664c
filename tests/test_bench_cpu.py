"""bench.py's CPU-baseline leg on the CPU: it times the oracle on a bounded
sample and, given the GPU run's outputs, reports their parity on the same
sequences. Here the 'GPU outputs' are planted on the CPU."""
import numpy as np
import torch

import bench
from oracle import gqa_paged_decode_oracle
from paged_kv_gqa_split_gb300 import workloads as wl


def test_cpu_baseline_parity_accepts_match_and_flags_error():
    w = wl.make_config("tiny")
    o, l = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    out = torch.from_numpy(o).to(torch.bfloat16)
    lse = torch.from_numpy(l).to(torch.float32)
    base, par = bench.cpu_baseline(w, out, lse, budget_s=0.01)
    assert base["kind"] == "oracle" and base["value"] > 0 and base["cores"] >= 1
    assert par["within_tolerance"] and par["sequences"] >= 1
    bad = out.clone()
    first = next(b for b in range(w.batch) if w.lens[b] > 0)
    bad[first, 3, 7] += 1.0                       # an error far outside the tolerance
    _, par_bad = bench.cpu_baseline(w, bad, lse, budget_s=0.01)
    assert not par_bad["within_tolerance"]
    assert np.isfinite(par_bad["max_abs_dO"])
