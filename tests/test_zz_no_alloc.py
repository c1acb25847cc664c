"""gqa_paged_decode_noalloc against gqa_paged_decode, through the C ABI.

The no-allocation entry point serves callers that must not allocate device
memory: a serving runtime that has reserved all free HBM for its KV-cache pool,
code running under CUDA stream capture (cudaMalloc cannot be captured), or a
loop that cannot take cudaMalloc's device-wide synchronisation. It keeps the
split partials in a fixed device array instead of an allocated workspace, so
its results must match the default entry point's. This file sorts last so that
a failure here cannot stop a run before the rest of the suite has run.
"""
import numpy as np
import pytest
import torch

from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl
from paged_kv_gqa_split_gb300.build import build

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


def _args(g, out, lse, batch, stream):
    return (g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.kv_indptr.data_ptr(),
            g.kv_indices.data_ptr(), g.sm_scale, out.data_ptr(), lse.data_ptr(), batch, stream.cuda_stream)


def test_noalloc_matches_default_entry_point_on_two_calls(cuda_device):
    build()
    _lib.load()
    assert _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0) == 0
    stream = torch.cuda.current_stream()
    # two different batches in a row: long sequences cut across many CTAs (so
    # the partials in the fixed array are used), empty and one-token sequences
    cases = [wl.make_workload([5000, 0, 37, 1, 900, 2049], seed=77, pool_factor=1.2),
             wl.make_workload([3, 12000, 0, 0, 640, 1], seed=78, pool_factor=1.5)]
    for w in cases:
        g = w.to("cuda")
        out_ref = torch.empty_like(g.q)
        lse_ref = torch.empty((w.batch, 32), dtype=torch.float32, device="cuda")
        assert _lib.gqa_paged_decode(*_args(g, out_ref, lse_ref, w.batch, stream)) == 0
        out = torch.full_like(g.q, float("nan"))
        lse = torch.full((w.batch, 32), float("nan"), device="cuda")
        assert _lib.gqa_paged_decode_noalloc(*_args(g, out, lse, w.batch, stream)) == 0
        torch.cuda.synchronize()
        o, orf = out.float().cpu().double().numpy(), out_ref.float().cpu().double().numpy()
        l, lrf = lse.cpu().double().numpy(), lse_ref.cpu().double().numpy()
        assert np.all(np.abs(o - orf) <= O_ATOL + O_RTOL * np.abs(orf))
        assert np.array_equal(np.isneginf(l), np.isneginf(lrf))
        fin = np.isfinite(lrf)
        assert np.all(np.abs(l[fin] - lrf[fin]) <= LSE_ATOL)
