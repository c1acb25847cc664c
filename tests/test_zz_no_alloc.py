"""gqa_paged_decode_noalloc against gqa_paged_decode and the oracle, through the C ABI.

The no-allocation entry point serves callers that must not allocate device
memory: a serving runtime that has reserved all free HBM for its KV-cache pool,
code running under CUDA stream capture (cudaMalloc cannot be captured), or a
loop that cannot take cudaMalloc's device-wide synchronisation. It keeps the
split partials in a fixed device array instead of an allocated workspace, so
its results must match the default entry point's and the float64 oracle's.
This file sorts last so that a failure here cannot stop a run before the rest
of the suite has run.
"""
import numpy as np
import pytest
import torch

from oracle import gqa_paged_decode_oracle
from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl
from paged_kv_gqa_split_gb300.build import build

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


def _args(g, out, lse, batch, stream):
    return (g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.kv_indptr.data_ptr(),
            g.kv_indices.data_ptr(), g.sm_scale, out.data_ptr(), lse.data_ptr(), batch, stream.cuda_stream)


def _close(o, l, orf, lrf):
    assert np.all(np.abs(o - orf) <= O_ATOL + O_RTOL * np.abs(orf))
    assert np.array_equal(np.isneginf(l), np.isneginf(lrf))
    fin = np.isfinite(lrf)
    assert np.all(np.abs(l[fin] - lrf[fin]) <= LSE_ATOL)


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
        o, l = out.float().cpu().double().numpy(), lse.cpu().double().numpy()
        _close(o, l, out_ref.float().cpu().double().numpy(), lse_ref.cpu().double().numpy())
        # and against the float64 oracle directly
        o_or, l_or = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
        _close(o, l, o_or, l_or)


def test_noalloc_refuses_a_plan_whose_tier1_partials_do_not_fit(cuda_device):
    """1536 tier-1 CTAs need 1536 x 2 x 16.5 KB of partials, more than the 32 MiB
    array: the call must return GQA_ERR_WORKSPACE without launching anything."""
    build()
    _lib.load()
    w = wl.make_workload([300, 0, 40], seed=79)
    g = w.to("cuda")
    stream = torch.cuda.current_stream()
    assert _lib.gqa_paged_decode_set_tuning(1536, 0, 4, 16, 2, 0) == 0
    try:
        out = torch.full_like(g.q, 5.0)
        lse = torch.full((w.batch, 32), 5.0, device="cuda")
        rc = _lib.gqa_paged_decode_noalloc(*_args(g, out, lse, w.batch, stream))
        torch.cuda.synchronize()
        assert rc == _lib.GQA_ERR_WORKSPACE
        assert torch.all(out == 5.0) and torch.all(lse == 5.0)
    finally:
        assert _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0) == 0
    # the default plan fits again
    out = torch.empty_like(g.q)
    lse = torch.empty((w.batch, 32), dtype=torch.float32, device="cuda")
    assert _lib.gqa_paged_decode_noalloc(*_args(g, out, lse, w.batch, stream)) == 0
    torch.cuda.synchronize()
    o_or, l_or = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    _close(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_or, l_or)
