"""Selected-token (sparse) paged decode on the GPU against the float64 oracle.

The sparse path of the sigit.si vLLM "qsa.py" page: each query row selects
TOPK logical positions of its request, resolved through a block table of any
page size; invalid columns drop out of the softmax. Tolerances are those of
the dense path: |dO| <= 2e-2 + 2e-2 |O_ref| and |dlse| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle.sparse as sp
from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


@pytest.fixture(autouse=True)
def _defaults(cuda_device):
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
    yield
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)


def gpu_sparse(w, with_lse=True):
    g = w.to("cuda")
    out, lse = _lib.sparse_run(g.q, g.k_cache, g.v_cache, g.logical_indices, g.block_table, g.token_to_req,
                               w.sm_scale, with_lse=with_lse)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy(), (lse.cpu().double().numpy() if lse is not None else None)


def check(w, out, lse, rows=None):
    o_ref, l_ref = sp.sparse_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.logical_indices, w.block_table,
                                                 w.token_to_req, w.sm_scale, rows)
    sel = list(range(w.rows)) if rows is None else list(rows)
    o, orf = out[sel], o_ref[sel]
    bad = np.abs(o - orf) > O_ATOL + O_RTOL * np.abs(orf)
    assert not bad.any(), f"{bad.sum()} O elements out of tolerance, max |dO| {np.abs(o - orf).max():.3g}"
    if lse is not None:
        l, lrf = lse[sel], l_ref[sel]
        assert np.array_equal(np.isneginf(l), np.isneginf(lrf))
        fin = np.isfinite(lrf)
        assert np.all(np.abs(l[fin] - lrf[fin]) <= LSE_ATOL), np.abs(l[fin] - lrf[fin]).max()
    empty = np.isneginf(l_ref[sel]).all(axis=1)
    assert np.all(o[empty] == 0)                                  # rows with no valid column: exact zeros
    return o_ref, l_ref


@pytest.mark.parametrize("lens,topk,page_size,seed", [
    ([40, 300, 17, 1000], 37, 16, 1),        # topk not a multiple of 16, short rows padded with -1
    ([2048, 5000, 3000], 2048, 64, 2),       # decode-sized rows, full selections
    ([100] * 9, 100, 1, 3),                  # page size 1 (the dense layout)
    ([700, 1, 129, 4096, 33], 256, 128, 4),  # large pages, a one-token request
    ([5000, 6000], 4096, 32, 5),             # rows long enough to be cut across CTAs
])
def test_sparse_matches_oracle(lens, topk, page_size, seed):
    w = wl.make_sparse_workload(lens, topk, page_size, seed)
    out, lse = gpu_sparse(w)
    check(w, out, lse)


def test_invalid_columns_repeats_and_unknown_requests():
    w = wl.make_sparse_workload([300, 90, 500, 64, 200], 96, 16, seed=11)
    idx = w.logical_indices
    width = w.block_table.shape[1]
    idx[0, 5] = -3                              # negative position
    idx[0, 6] = width * 16 + 7                  # logical page past the table
    idx[1, 0:10] = idx[1, 20]                   # one column repeated ten times
    nb1 = (w.lens[1] + 15) // 16
    idx[1, 40] = nb1 * 16 + 2 if nb1 < width else -1   # a logical page whose table entry is -1
    w.block_table[2, 3] = w.num_blocks + 9      # physical page past the pool
    w.token_to_req[3] = -1                      # unknown request: the whole row is invalid
    idx[4, :] = -1                              # nothing selected
    out, lse = gpu_sparse(w)
    o_ref, l_ref = check(w, out, lse)
    assert np.all(np.isneginf(l_ref[3])) and np.all(np.isneginf(l_ref[4]))


def test_permuted_requests_and_shared_request():
    w = wl.make_sparse_workload([400, 50, 900, 300], 128, 32, seed=12)
    w.token_to_req.copy_(torch.tensor([2, 0, 3, 2], dtype=torch.int32))   # rows 0 and 3 read request 2
    w.logical_indices.clamp_(max=min(w.lens) - 1)                          # positions valid in every request
    out, lse = gpu_sparse(w)
    check(w, out, lse)


@pytest.mark.parametrize("tuning", [(40, 8, 0, 0, 0, 0, 0, 0, 500, 16), (7, 1, 0, 0, 0, 0, 0, 13, 400, 4),
                                    (300, 1, 0, 0, 0, 0, 0, -1), (60, 8, 0, 0, 0, 0, 4, 0, 300, 8)])
def test_sparse_split_across_ctas(tuning):
    """Rows cut into many pieces: small CTA counts, tier 2, both merge placements."""
    assert _lib.gqa_paged_decode_set_tuning(*tuning) == 0
    w = wl.make_sparse_workload([3000, 40, 1200, 2500, 7], 1024, 16, seed=13)
    w.logical_indices[2, 100:400] = -1          # a run of masked columns inside a row
    w.logical_indices[3, :] = -1                # a row with nothing: all its pieces are masked
    out, lse = gpu_sparse(w)
    check(w, out, lse)


def test_without_lse_buffer():
    w = wl.make_sparse_workload([500, 800], 256, 64, seed=14)
    out, lse = gpu_sparse(w, with_lse=False)
    assert lse is None
    check(w, out, None)


def test_sparse_config_every_row():
    """The bench's selected-token workload at full size, every row against the oracle."""
    w = wl.make_sparse_config()
    out, lse = gpu_sparse(w)
    check(w, out, lse)


def test_sparse_rows_past_grid():
    """3000 rows, more than the decode and merge grids: rows of empty requests (every column -1) are
    written as O = 0, LSE = -inf over outputs that start as garbage; the rest match the oracle."""
    lens = torch.randint(0, 40, (3000,), generator=torch.Generator().manual_seed(71)).tolist()
    w = wl.make_sparse_workload(lens, 16, 16, 72)
    g = w.to("cuda")
    out = torch.full_like(g.q, 7.0)
    lse = torch.full((w.rows, 32), 7.0, dtype=torch.float32, device="cuda")
    _lib.sparse_run(g.q, g.k_cache, g.v_cache, g.logical_indices, g.block_table, g.token_to_req, w.sm_scale,
                    out=out, lse=lse)
    torch.cuda.synchronize()
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    empty = [r for r, n in enumerate(lens) if n == 0]
    assert empty and np.all(o[empty] == 0.0) and np.all(np.isneginf(l[empty]))
    check(w, o, l)
