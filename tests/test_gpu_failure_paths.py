"""Failure paths of the library, exercised without faulting or hanging the GPU.

* A workspace allocation that fails: a test hook makes the next library-owned
  workspace allocation fail exactly where a failing cudaMalloc would. The call
  must return GQA_ERR_WORKSPACE without writing its outputs, and the next call
  must allocate and give the oracle's result.
* A bounded in-kernel merge wait that runs out (the one-wave decode), and a
  bounded pipeline wait that runs out: the TMA-gather decode variant bounds
  every mbarrier wait. With the give-up limit shortened to a few nanoseconds
  (valid inputs, nothing else changed) its waits give up before the first copies
  land; the CTAs drain their copies in flight (that drain keeps its normal
  limit) and return. The call must complete, the device error word must carry
  the timeout bit, and a following call with the normal limit must be correct.
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
ERR_TIMEOUT_FULL, ERR_TIMEOUT_EMPTY, ERR_MERGE_WAIT = 1, 2, 32


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    _lib.load()
    yield
    _lib.gqa_paged_decode_test_fail_allocs(0)
    _lib.gqa_paged_decode_test_wait_limit_ns(0)
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)


def _matches_oracle(w, out, lse):
    o_ref, l_ref = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    assert np.array_equal(np.isneginf(l), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(l[fin] - l_ref[fin]).max() <= LSE_ATOL


def test_injected_workspace_allocation_failure_then_recovery():
    w = wl.make_workload([700, 0, 33, 2500, 1], seed=61, pool_factor=1.3)
    g = w.to("cuda")
    assert _lib.gqa_paged_decode_device_error() == 0
    _lib.gqa_paged_decode_release()  # the next call has to allocate
    assert _lib.gqa_paged_decode_test_fail_allocs(1) == 0
    out = torch.full_like(g.q, 3.0)
    lse = torch.full((w.batch, 32), 3.0, device="cuda")
    stream = torch.cuda.current_stream()
    rc = _lib.gqa_paged_decode(g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(), g.kv_indptr.data_ptr(),
                               g.kv_indices.data_ptr(), w.sm_scale, out.data_ptr(), lse.data_ptr(), w.batch,
                               stream.cuda_stream)
    torch.cuda.synchronize()
    assert rc == _lib.GQA_ERR_WORKSPACE
    assert torch.all(out == 3.0) and torch.all(lse == 3.0)  # nothing was launched
    # the hook fired once; the next call allocates and computes normally
    out2, lse2 = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
    torch.cuda.synchronize()
    _matches_oracle(w, out2, lse2)
    assert _lib.gqa_paged_decode_device_error() == 0


def test_injected_failure_count_and_reset():
    assert _lib.gqa_paged_decode_test_fail_allocs(-1) == _lib.GQA_ERR_INVALID_ARGUMENT
    w = wl.make_workload([40, 9], seed=62)
    g = w.to("cuda")
    _lib.gqa_paged_decode_release()
    assert _lib.gqa_paged_decode_test_fail_allocs(2) == 0
    for _ in range(2):
        with pytest.raises(_lib.GqaError) as e:
            _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
        assert e.value.code == _lib.GQA_ERR_WORKSPACE
    out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
    torch.cuda.synchronize()
    _matches_oracle(w, out, lse)
    # turned off again (0) before it fires: the allocation succeeds
    _lib.gqa_paged_decode_release()
    assert _lib.gqa_paged_decode_test_fail_allocs(1) == 0
    assert _lib.gqa_paged_decode_test_fail_allocs(0) == 0
    out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
    torch.cuda.synchronize()
    _matches_oracle(w, out, lse)


def test_in_kernel_merge_wait_gives_up_and_call_completes():
    """The one-wave decode (an opt-in mode) merges a split sequence once all of its pieces have
    arrived, waiting at most the give-up limit. With that limit at a few
    nanoseconds, a merge of a sequence cut into hundreds of pieces gives up: the
    call completes, bit 32 of the device error word is set, and a following call
    with the normal limit is correct."""
    w = wl.make_workload([60000, 0, 900, 40000], seed=64, pool_factor=1.1)
    g = w.to("cuda")
    assert _lib.gqa_paged_decode_device_error() == 0
    assert _lib.gqa_paged_decode_set_merge_mode(_lib.MERGE_ONE_WAVE) == 0
    try:
        assert _lib.gqa_paged_decode_test_wait_limit_ns(5) == 0
        _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
        torch.cuda.synchronize()
        flags = _lib.gqa_paged_decode_device_error()
        assert flags & ERR_MERGE_WAIT, flags
        assert flags & ~ERR_MERGE_WAIT == 0, flags
        assert _lib.gqa_paged_decode_test_wait_limit_ns(0) == 0
        out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
        torch.cuda.synchronize()
        _matches_oracle(w, out, lse)
        assert _lib.gqa_paged_decode_device_error() == 0
    finally:
        _lib.gqa_paged_decode_test_wait_limit_ns(0)
        _lib.gqa_paged_decode_set_merge_mode(_lib.MERGE_KERNEL)


@pytest.mark.parametrize("variant", [(0, 0, 4, 16, 5, 1), (0, 0, 4, 32, 3, 1), (0, 0, 1, 16, 4, 1)])
def test_bounded_wait_gives_up_and_call_completes(variant):
    w = wl.make_workload([3000, 0, 129, 17, 1500], seed=63, pool_factor=1.2)
    g = w.to("cuda")
    assert _lib.gqa_paged_decode_device_error() == 0
    assert _lib.gqa_paged_decode_set_tuning(*variant) == 0
    try:
        assert _lib.gqa_paged_decode_test_wait_limit_ns(5) == 0
        _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)  # returns 0: it launched
        torch.cuda.synchronize()  # and it completes: every CTA returned
        flags = _lib.gqa_paged_decode_device_error()
        assert flags & (ERR_TIMEOUT_FULL | ERR_TIMEOUT_EMPTY), flags
        assert flags & ~(ERR_TIMEOUT_FULL | ERR_TIMEOUT_EMPTY) == 0, flags
        # the normal limit again: the same variant is correct and raises nothing
        assert _lib.gqa_paged_decode_test_wait_limit_ns(0) == 0
        out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
        torch.cuda.synchronize()
        _matches_oracle(w, out, lse)
        assert _lib.gqa_paged_decode_device_error() == 0
    finally:
        _lib.gqa_paged_decode_test_wait_limit_ns(0)
        _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
