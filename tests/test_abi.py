"""C-ABI checks that need no GPU: the library builds, loads, exports every
declared entry point, and rejects bad arguments before touching the device."""
import os
import re

import pytest

from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_paged_decode.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_\w+)\s*\(", text)))


def test_header_declares_the_problem_entry_point():
    names = declared_functions()
    assert "gqa_paged_decode" in names
    assert len(names) >= 8


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib._SIGNATURES, f"{name} has no binding"


def test_binding_names_match_header():
    assert sorted(_lib._SIGNATURES) == declared_functions()


def test_strerror(lib):
    assert _lib.strerror(0) == "success"
    for code in (-1, -2, -3, -4):
        assert len(_lib.strerror(code)) > 10
    assert _lib.strerror(-99) == "unknown error code"


def test_batch_zero_is_a_noop(lib):
    assert _lib.gqa_paged_decode(None, None, None, None, None, 0.1, None, None, 0, None) == 0


def test_negative_batch_rejected(lib):
    assert _lib.gqa_paged_decode(16, 16, 16, 16, 16, 0.1, 16, 16, -1, None) == _lib.GQA_ERR_INVALID_ARGUMENT


def test_null_pointers_rejected(lib):
    a = 1 << 20  # a 256-aligned dummy address; never dereferenced on this path
    args = [a, a, a, a, a, 0.1, a, a, 3, None]
    for i in (0, 3, 6, 7):
        bad = list(args)
        bad[i] = None
        assert _lib.gqa_paged_decode(*bad) == _lib.GQA_ERR_INVALID_ARGUMENT, i


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), float("-inf")])
def test_non_finite_scale_rejected(lib, scale):
    a = 1 << 20
    assert _lib.gqa_paged_decode(a, a, a, a, a, scale, a, a, 3, None) == _lib.GQA_ERR_INVALID_ARGUMENT


def test_misaligned_pointers_rejected(lib):
    a = 1 << 20
    for i, off in ((0, 8), (1, 2), (2, 4), (6, 8), (7, 4), (3, 2), (4, 1)):
        args = [a, a, a, a, a, 0.1, a, a, 3, None]
        args[i] = a + off
        assert _lib.gqa_paged_decode(*args) == _lib.GQA_ERR_INVALID_ARGUMENT, (i, off)


def test_checked_needs_pages_and_flag(lib):
    a = 1 << 20
    assert _lib.gqa_paged_decode_checked(a, a, a, a, a, 0.1, a, a, 2, None, 0, a) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_decode_checked(a, a, a, a, a, 0.1, a, a, 2, None, 5, None) == _lib.GQA_ERR_INVALID_ARGUMENT


def test_ws_variant_needs_workspace(lib):
    a = 1 << 20
    assert _lib.gqa_paged_decode_ws(a, a, a, a, a, 0.1, a, a, 2, None, None, 0) == _lib.GQA_ERR_WORKSPACE


@pytest.mark.parametrize("tuning", [(0, 0, 3, 0, 0, 0), (0, 0, 4, 24, 0, 0), (0, 0, 4, 16, 9, 0), (-1, 0, 0, 0, 0, 0),
                                    (0, 0, 4, 32, 3, 0), (0, 0, 4, 32, 3, 2), (0, 0, 2, 16, 5, 1), (2000, 0, 0, 0, 0, 0),
                                    (0, 0, 0, 0, 0, 0, -2), (0, 0, 0, 0, 0, 0, 0, -2), (0, 0, 0, 0, 0, 0, 0, 70000),
                                    (0, 0, 0, 0, 0, 0, 0, 0, 901), (0, 0, 0, 0, 0, 0, 0, 0, -1),
                                    (0, 0, 0, 0, 0, 0, 0, 0, 0, -1), (0, 0, 4, 16, 3, 3), (0, 0, 2, 16, 2, 3),
                                    (0, 0, 0, 0, 0, 4), (0, 0, 2, 16, 2, 2), (0, 0, 4, 24, 2, 2), (0, 0, 4, 16, 5, 2)])
def test_unsupported_tuning_rejected(lib, tuning):
    assert _lib.gqa_paged_decode_set_tuning(*tuning) == _lib.GQA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("tuning", [(0, 0, 0, 0, 0, 0), (0, 0, 4, 16, 3, 0), (0, 0, 1, 16, 6, 0),
                                    (0, 0, 4, 32, 3, 1), (0, 0, 4, 16, 5, 1), (64, 32, 2, 16, 5, 0),
                                    (0, 0, 0, 0, 0, 0, -1), (0, 0, 0, 0, 0, 0, 64), (0, 0, 0, 0, 0, 0, 0, -1),
                                    (0, 0, 0, 0, 0, 0, 0, 5000, 900, 1), (0, 0, 0, 0, 0, 0, 0, 0, 50, 128),
                                    (0, 0, 4, 16, 2, 3), (0, 0, 0, 0, 0, 3), (0, 0, 4, 16, 3, 2), (0, 0, 4, 32, 2, 2),
                                    (0, 0, 0, 0, 0, 2)])
def test_supported_tuning_accepted(lib, tuning):
    assert _lib.gqa_paged_decode_set_tuning(*tuning) == 0
    assert _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0) == 0


def test_cpu_tensors_raise():
    import torch
    from paged_kv_gqa_split_gb300 import workloads as wl
    w = wl.make_workload([3, 4], seed=1)
    with pytest.raises(ValueError, match="no CPU path"):
        _lib.run(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices)
    assert torch.is_tensor(w.q)


def test_append_argument_checks(lib):
    a = 1 << 20
    assert _lib.gqa_paged_kv_append(None, None, None, None, None, 0, 0, None) == 0
    assert _lib.gqa_paged_kv_append(a, a, a, a, a, -1, 4, None) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_kv_append(a, a, a, a, a, 3, 0, None) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_kv_append(a, None, a, a, a, 3, 4, None) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_kv_append(a + 8, a, a, a, a, 3, 4, None) == _lib.GQA_ERR_INVALID_ARGUMENT


def _sparse_args(**kw):
    a = 1 << 20  # 16-byte aligned dummy device address; no call below reaches the device
    args = dict(q=a, k_cache=a, v_cache=a, logical_indices=a, block_table=a, token_to_req=a, sm_scale=0.1, out=a,
                lse=a, rows=2, topk=8, page_size=16, num_cache_blocks=10, num_requests=2, page_table_width=4,
                stream=None)
    args.update(kw)
    return list(args.values())


def test_sparse_rows_zero_is_a_noop(lib):
    assert _lib.gqa_sparse_paged_decode(*_sparse_args(rows=0, q=None, k_cache=None)) == 0


@pytest.mark.parametrize("bad", [dict(rows=-1), dict(topk=0), dict(page_size=0), dict(num_cache_blocks=0),
                                 dict(num_requests=0), dict(page_table_width=0), dict(q=None), dict(out=None),
                                 dict(block_table=None), dict(token_to_req=None), dict(logical_indices=None),
                                 dict(sm_scale=float("nan")), dict(q=(1 << 20) + 8), dict(lse=(1 << 20) + 4),
                                 dict(logical_indices=(1 << 20) + 2), dict(num_cache_blocks=1 << 26, page_size=64),
                                 dict(rows=1 << 20, topk=1 << 12)])
def test_sparse_bad_arguments_rejected(lib, bad):
    assert _lib.gqa_sparse_paged_decode(*_sparse_args(**bad)) == _lib.GQA_ERR_INVALID_ARGUMENT


def test_sparse_cpu_tensors_raise():
    import torch
    from paged_kv_gqa_split_gb300 import workloads as wl
    w = wl.make_sparse_workload([5, 9], 4, 4, seed=1)
    with pytest.raises(ValueError, match="no CPU path"):
        _lib.sparse_run(w.q, w.k_cache, w.v_cache, w.logical_indices, w.block_table, w.token_to_req)


def test_fp8_argument_checks(lib):
    a = 1 << 20
    assert _lib.gqa_paged_decode_fp8(None, None, None, None, None, 0.1, None, None, 0, None) == 0
    assert _lib.gqa_paged_decode_fp8(a, a, a, a, a, 0.1, a, a, -1, None) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_decode_fp8(a, a, a, None, a, 0.1, a, a, 2, None) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_decode_fp8(a, a + 8, a, a, a, 0.1, a, a, 2, None) == _lib.GQA_ERR_INVALID_ARGUMENT
    assert _lib.gqa_paged_decode_fp8(a, a, a, a, a, float("nan"), a, a, 2, None) == _lib.GQA_ERR_INVALID_ARGUMENT


def test_fp8_wrapper_checks():
    import torch
    from paged_kv_gqa_split_gb300 import workloads as wl
    w = wl.make_fp8_workload([3, 4], seed=1)
    with pytest.raises(ValueError, match="no CPU path"):
        _lib.run_fp8(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices)
    assert w.k_cache.shape[1] == _lib.FP8_ROW_BYTES and w.k_cache.dtype == torch.uint8


def test_mla_argument_checks(lib):
    a = 1 << 20
    ok = [a, a, a, a, 0.07, a, a, 2, 1, 16, 64, 10, 4, None]
    assert _lib.gqa_mla_decode(*ok[:7], 0, *ok[8:]) == 0
    for i, bad in ((7, -1), (8, 0), (9, 12), (10, 0), (11, 0), (12, 0), (0, None), (5, None), (2, None),
                   (0, a + 8), (6, a + 2), (4, float("nan"))):
        args = list(ok)
        args[i] = bad
        assert _lib.gqa_mla_decode(*args) == _lib.GQA_ERR_INVALID_ARGUMENT, (i, bad)


def test_mla_set_tuning_checks(lib):
    for bad in (-1, 2, 5, 8):
        assert _lib.gqa_mla_set_tuning(bad) == _lib.GQA_ERR_INVALID_ARGUMENT
    for ok in (1, 3, 4, 0):
        assert _lib.gqa_mla_set_tuning(ok) == 0


def test_mla_cpu_tensors_raise():
    from paged_kv_gqa_split_gb300 import workloads as wl
    w = wl.make_mla_workload([5, 9], 16, 1, 4, seed=1)
    with pytest.raises(ValueError, match="no CPU path"):
        _lib.mla_run(w.q, w.kv_cache, w.block_table, w.cache_seqlens)
