"""The multi-process oracle runner returns exactly the single-process oracle's
rows: each worker evaluates the same function on its sequences, with their pages
copied out and renumbered, which the oracle's page-relabelling pin shows leaves
every float64 result unchanged."""
import numpy as np

from oracle import gqa_paged_decode_oracle
from oracle.pool import OraclePool, _share_plan, gqa_paged_decode_oracle_parallel, host_cores
from paged_kv_gqa_split_gb300 import workloads as wl


def test_parallel_rows_are_bit_identical_to_single_process():
    w = wl.make_workload([0, 37, 1, 300, 0, 129, 64, 2, 0], seed=91, pool_factor=1.7)
    o1, l1 = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    o2, l2 = gqa_paged_decode_oracle_parallel(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale,
                                              workers=3)
    assert np.array_equal(o1, o2)
    assert np.array_equal(l1, l2)  # -inf rows of empty sequences included


def test_selected_sequences_leave_other_rows_nan():
    w = wl.make_workload([5, 0, 40, 7], seed=92)
    o, l = gqa_paged_decode_oracle_parallel(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale,
                                            seqs=[1, 3], workers=2)
    o1, l1 = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale,
                                     seqs=[1, 3])
    assert np.isnan(o[[0, 2]]).all() and np.isnan(l[[0, 2]]).all()
    assert np.array_equal(o[[1, 3]], o1[[1, 3]]) and np.array_equal(l[[1, 3]], l1[[1, 3]])


def test_all_empty_share_and_repeated_rounds():
    w = wl.make_workload([0, 0, 0, 9], seed=93)
    with OraclePool(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale, workers=4) as pool:
        a = pool.run()
        b = pool.run()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.all(a[0][:3] == 0.0) and np.all(np.isneginf(a[1][:3]))
    assert a[2] > 0 and b[2] > 0


def test_shares_balance_tokens_and_cover_every_sequence():
    lens = [5000, 10, 10, 10, 4000, 0, 3000, 20]
    shares = _share_plan(lens, list(range(len(lens))), 3)
    assert sorted(b for s in shares for b in s) == list(range(len(lens)))
    loads = [sum(max(1, lens[b]) for b in s) for s in shares]
    assert max(loads) <= 5000 + 30
    assert host_cores() >= 1
