"""Pins of the selected-token (sparse) decode oracle, on the CPU.

The oracle follows the sparse split-K GQA path of the sigit.si vLLM "qsa.py"
page. These tests tie it to things other than itself:

* a sparse problem built by scattering a dense page-size-1 problem into
  blocks through a random block table must give the dense oracle's result
  over the selected pages (the dense oracle is pinned in test_oracle.py);
* every kind of invalid column leaves the result unchanged, a row with no
  valid column gives zeros and -inf, a duplicated column counts twice;
* a scalar brute force on a tiny case, and the one-column closed form;
* mistakes planted in the resolution rule fail one of the pins.
"""
import math

import numpy as np
import pytest
import torch

import oracle.sparse as sp
from oracle import gqa_paged_decode_oracle
from paged_kv_gqa_split_gb300 import workloads as wl

SCALE = 1.0 / math.sqrt(128)


def scatter_dense_into_blocks(dense, page_size, seed, topk, dup=True):
    """Sparse inputs equivalent, by construction, to a dense page-size-1 problem.

    Request order is a permutation of the rows; each request's logical token t
    is stored at block_table[req, t // ps], offset t % ps, holding the dense
    page kv_indices[indptr[b] + t]. Returns (sparse inputs, dense reference
    inputs over the selected columns).
    """
    g = torch.Generator().manual_seed(seed)
    lens = dense.lens
    rows = len(lens)
    ip = dense.kv_indptr.tolist()
    req_of_row = torch.randperm(rows, generator=g)          # row r belongs to request req_of_row[r]
    nblk = [max(1, -(-n // page_size)) for n in lens]
    width = max(nblk) + 1
    num_blocks = sum(nblk) + 3
    perm = torch.randperm(num_blocks, generator=g)
    table = torch.full((rows, width), -1, dtype=torch.int32)
    kc = torch.zeros((num_blocks, page_size, 4, 128), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    off = 0
    for r in range(rows):
        q_req = int(req_of_row[r])
        b = r                                                 # row r carries dense sequence r
        for j in range(nblk[b]):
            blk = int(perm[off + j])
            table[q_req, j] = blk
            for o in range(page_size):
                t = j * page_size + o
                if t < lens[b]:
                    page = int(dense.kv_indices[ip[b] + t])
                    kc[blk, o] = dense.k_cache[page, 0]
                    vc[blk, o] = dense.v_cache[page, 0]
        off += nblk[b]
    idx = torch.full((rows, topk), -1, dtype=torch.int32)
    sel_pages, sel_ptr = [], [0]
    for r in range(rows):
        n = lens[r]
        if n:
            if dup:
                cols = torch.randint(0, n, (min(topk, n + 2),), generator=g)   # repeats allowed
            else:
                cols = torch.randperm(n, generator=g)[:min(topk, n)]
            idx[r, :cols.numel()] = cols.to(torch.int32)
            sel_pages += [int(dense.kv_indices[ip[r] + int(t)]) for t in cols]
        sel_ptr.append(len(sel_pages))
    sparse = wl.SparseWorkload("scatter", dense.q, kc, vc, idx, table, req_of_row.to(torch.int32), SCALE, list(lens))
    ref = (torch.tensor(sel_ptr, dtype=torch.int32), torch.tensor(sel_pages, dtype=torch.int32))
    return sparse, ref


def run_sparse(w, rows=None):
    return sp.sparse_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.logical_indices, w.block_table,
                                         w.token_to_req, w.sm_scale, rows)


@pytest.mark.parametrize("page_size,topk,dup", [(16, 40, True), (1, 7, False), (5, 64, True), (64, 3, False)])
def test_equals_dense_oracle_on_scattered_problem(page_size, topk, dup):
    dense = wl.make_workload([13, 0, 70, 1, 33], seed=61, pool_factor=1.5)
    sparse, (ptr, pages) = scatter_dense_into_blocks(dense, page_size, seed=62, topk=topk, dup=dup)
    o, l = run_sparse(sparse)
    od, ld = gqa_paged_decode_oracle(dense.q, dense.k_cache, dense.v_cache, ptr, pages, SCALE)
    assert np.allclose(o, od, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(ld)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.allclose(l[fin], ld[fin], rtol=0, atol=1e-12)
    assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))   # the empty request selects nothing


def _with_columns(w, extra):
    """Copy of w whose rows get the extra columns appended (one list per row)."""
    width = max(len(e) for e in extra)
    add = torch.full((w.rows, width), -1, dtype=torch.int32)
    for r, e in enumerate(extra):
        add[r, :len(e)] = torch.tensor(e, dtype=torch.int32)
    idx = torch.cat([w.logical_indices, add], dim=1)
    return wl.SparseWorkload(w.name, w.q, w.k_cache, w.v_cache, idx, w.block_table.clone(), w.token_to_req.clone(),
                             w.sm_scale, list(w.lens))


def test_invalid_columns_are_ignored():
    w = wl.make_sparse_workload([20, 9, 33], 12, 8, seed=71)
    o0, l0 = run_sparse(w)
    width = w.block_table.shape[1]
    # row 1 owns 2 of the 5 block-table entries: logical page 3 maps to -1
    assert int(w.block_table[1, 3]) == -1
    extra = [[-1, -7, width * 8 + 2], [3 * 8 + 1, -1], [width * 8 + 100, -1]]
    w2 = _with_columns(w, extra)
    o, l = run_sparse(w2)
    assert np.array_equal(o, o0) and np.array_equal(l, l0)
    # a physical page past the pool is invalid too
    w3 = _with_columns(w, [[17], [], []])
    w3.block_table[0, 17 // 8] = w.num_blocks + 5
    o3, l3 = run_sparse(w3)
    base = _with_columns(w, [[], [], []])
    base.block_table[0, 17 // 8] = w.num_blocks + 5   # the same table, no extra column
    ob, lb = run_sparse(base)
    assert np.array_equal(o3, ob) and np.array_equal(l3, lb)


@pytest.mark.parametrize("req", [-1, 3, 1000])
def test_row_of_unknown_request_gives_zeros(req):
    w = wl.make_sparse_workload([20, 9, 33], 12, 8, seed=72)
    w.token_to_req[2] = req
    o, l = run_sparse(w)
    assert np.all(o[2] == 0) and np.all(np.isneginf(l[2]))
    assert np.all(np.isfinite(l[:2]))


def test_row_with_only_invalid_columns():
    w = wl.make_sparse_workload([20, 9], 6, 4, seed=73)
    w.logical_indices[1] = -1
    o, l = run_sparse(w)
    assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))


def test_single_column_closed_form():
    w = wl.make_sparse_workload([30], 4, 8, seed=74)
    w.logical_indices[0] = torch.tensor([-1, 21, -1, -1], dtype=torch.int32)
    o, l = run_sparse(w)
    blk = int(w.block_table[0, 21 // 8])
    k = w.k_cache[blk, 21 % 8].double().numpy()
    v = w.v_cache[blk, 21 % 8].double().numpy()
    q = w.q[0].double().numpy()
    for h in range(32):
        g = h // 8
        assert np.array_equal(o[0, h], v[g])                     # one token: O is its value row
        assert abs(l[0, h] - SCALE * float(q[h] @ k[g]) / math.log(2.0)) < 1e-12


def test_scalar_brute_force():
    """Loops over columns with math.exp and math.fsum, no max subtraction."""
    w = wl.make_sparse_workload([7, 11], 9, 3, seed=75)
    w.logical_indices[0, 2] = w.logical_indices[0, 0]            # a repeated column
    w.logical_indices[1, 4] = 50                                  # past the table width
    o, l = run_sparse(w)
    nb, ps = w.num_blocks, w.page_size
    for r in range(2):
        req = int(w.token_to_req[r])
        for h in range(32):
            g = h // 8
            qv = [float(x) for x in w.q[r, h].float()]
            ws, rows_v = [], []
            for c in range(w.topk):
                t = int(w.logical_indices[r, c])
                if t < 0 or t // ps >= w.block_table.shape[1]:
                    continue
                blk = int(w.block_table[req, t // ps])
                if not 0 <= blk < nb:
                    continue
                kv = [float(x) for x in w.k_cache[blk, t % ps, g].float()]
                s = SCALE * math.fsum(a * b for a, b in zip(qv, kv))
                ws.append(math.exp(s))
                rows_v.append([float(x) for x in w.v_cache[blk, t % ps, g].float()])
            den = math.fsum(ws)
            for d in range(0, 128, 17):
                num = math.fsum(wi * rv[d] for wi, rv in zip(ws, rows_v))
                assert abs(o[r, h, d] - num / den) < 1e-12 * max(1.0, abs(num / den))
            assert abs(l[r, h] - math.log2(den)) < 1e-12


@pytest.mark.parametrize("slip", ["offset_from_page", "row_as_request", "no_page_range_check", "page_floor_plus_one"])
def test_pins_catch_planted_mistakes(monkeypatch, slip):
    """Each slip in the resolution rule must fail a pin."""
    good = sp.resolve_slots

    def bad(logical_indices, block_table, token_to_req, page_size, num_cache_blocks):
        idx = np.asarray(logical_indices, dtype=np.int64)
        table = np.asarray(block_table, dtype=np.int64)
        req = np.asarray(token_to_req, dtype=np.int64)
        if slip == "row_as_request":
            req = np.arange(idx.shape[0])
        out = np.full(idx.shape, -1, dtype=np.int64)
        for r in range(idx.shape[0]):
            for c in range(idx.shape[1]):
                t = int(idx[r, c])
                if t < 0 or t // page_size >= table.shape[1] or not 0 <= req[r] < table.shape[0]:
                    continue
                lp = t // page_size + (1 if slip == "page_floor_plus_one" and t % page_size == page_size - 1 else 0)
                lp = min(lp, table.shape[1] - 1)
                page = int(table[req[r], lp])
                if slip != "no_page_range_check" and not 0 <= page < num_cache_blocks:
                    continue
                if page < 0:
                    continue
                offs = (t // page_size) % page_size if slip == "offset_from_page" else t % page_size
                out[r, c] = page * page_size + offs
        return out

    monkeypatch.setattr(sp, "resolve_slots", bad)
    failed = False
    try:
        test_equals_dense_oracle_on_scattered_problem(16, 40, True)
        test_invalid_columns_are_ignored()
    except AssertionError:
        failed = True
    except IndexError:
        failed = True
    finally:
        monkeypatch.setattr(sp, "resolve_slots", good)
    assert failed, slip
