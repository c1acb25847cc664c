"""Pins of the dense MLA decode oracle (oracle/mla.py), on the CPU.

* a scalar brute force on a tiny case (math.exp / math.fsum, no max shift);
* the result does not depend on which blocks hold the tokens;
* one token: O is its 512 NoPE values and lse its score; q = 0: O is the
  mean NoPE row and lse = ln n; every token twice: O unchanged, lse + ln 2;
* the rows (query token i, head h) and the [B, h_q, s_q] lse layout;
* an empty sequence gives zeros and -inf;
* slips planted in the oracle (value slice, dropped RoPE term, block/offset
  swap, base-2 lse) each fail one of these pins.
"""
import math

import numpy as np
import pytest
import torch

import oracle.mla as ml
from paged_kv_gqa_split_gb300 import workloads as wl


def run(w, seqs=None):
    return ml.mla_decode_oracle(w.q, w.kv_cache, w.block_table, w.cache_seqlens, w.softmax_scale, seqs)


def _tokens(w, b):
    """KV rows of sequence b in token order, read through the block table by hand."""
    rows = []
    for t in range(w.lens[b]):
        blk = int(w.block_table[b, t // w.page_size])
        rows.append(w.kv_cache[blk, t % w.page_size, 0].double().numpy())
    return np.array(rows).reshape(-1, 576)


def test_scalar_brute_force():
    w = wl.make_mla_workload([5, 3], h_q=16, s_q=2, page_size=4, seed=91)
    o, l = run(w)
    for b in range(2):
        kv = _tokens(w, b)
        for i in range(2):
            for h in (0, 7, 15):
                qv = w.q[b, i, h].double().numpy()
                ws = [math.exp(w.softmax_scale * math.fsum(qv * kv[t])) for t in range(len(kv))]
                den = math.fsum(ws)
                for d in (0, 100, 511):
                    num = math.fsum(ws[t] * kv[t, d] for t in range(len(kv)))
                    assert abs(o[b, i, h, d] - num / den) < 1e-12 * max(1.0, abs(num / den))
                assert abs(l[b, h, i] - math.log(den)) < 1e-12


def test_block_placement_does_not_matter():
    w = wl.make_mla_workload([70, 5, 130], h_q=16, s_q=1, page_size=16, seed=92)
    o, l = run(w)
    # move every block to a new place in a bigger pool
    nb = w.kv_cache.shape[0]
    g = torch.Generator().manual_seed(93)
    new_of = torch.randperm(2 * nb, generator=g)[:nb]
    kv2 = torch.zeros((2 * nb,) + tuple(w.kv_cache.shape[1:]), dtype=w.kv_cache.dtype)
    kv2[new_of] = w.kv_cache
    t2 = torch.where(w.block_table >= 0, new_of[w.block_table.clamp(min=0).long()].to(torch.int32), w.block_table)
    w2 = wl.MlaWorkload("moved", w.q, kv2, t2, w.cache_seqlens, w.softmax_scale, w.lens)
    o2, l2 = run(w2)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_one_token_closed_form():
    w = wl.make_mla_workload([1], h_q=16, s_q=1, page_size=64, seed=94)
    o, l = run(w)
    kv = _tokens(w, 0)[0]
    q = w.q[0, 0].double().numpy()
    assert np.array_equal(o[0, 0], np.broadcast_to(kv[:512], (16, 512)))
    assert np.allclose(l[0, :, 0], w.softmax_scale * (q @ kv), rtol=0, atol=1e-12)


def test_zero_query_and_duplicated_tokens():
    w = wl.make_mla_workload([9, 40], h_q=16, s_q=1, page_size=8, seed=95)
    w.q.zero_()
    o, l = run(w)
    for b in range(2):
        kv = _tokens(w, b)
        assert np.allclose(o[b, 0], kv[:, :512].mean(axis=0), rtol=0, atol=1e-12)
        assert np.allclose(l[b, :, 0], math.log(w.lens[b]), rtol=0, atol=1e-12)
    # every token twice: same softmax, log-sum-exp up by ln 2
    w = wl.make_mla_workload([9, 40], h_q=16, s_q=1, page_size=8, seed=96)
    o, l = run(w)
    n0 = w.lens
    nb = w.kv_cache.shape[0]
    kv2 = torch.cat([w.kv_cache, w.kv_cache])
    width = w.block_table.shape[1]
    t2 = torch.full((2, 2 * width), -1, dtype=torch.int32)
    lens2 = []
    for b in range(2):
        toks = [(int(w.block_table[b, t // 8]), t % 8) for t in range(n0[b])]
        toks = toks + [(blk + nb, off) for blk, off in toks]           # the copy lives in the second half
        # lay the 2n tokens out in fresh blocks of the doubled pool, keeping order within pages
        flat = []
        for blk, off in toks:
            flat.append(kv2[blk, off, 0])
        blocks = (len(flat) + 7) // 8
        base = b * 2 * width
        for j in range(blocks):
            t2[b, j] = base + j
        lens2.append(len(flat))
        if b == 0:
            kv3 = torch.zeros((4 * width * 2, 8, 1, 576), dtype=torch.bfloat16)
        for t, row in enumerate(flat):
            kv3[base + t // 8, t % 8, 0] = row
    w2 = wl.MlaWorkload("twice", w.q, kv3, t2, torch.tensor(lens2, dtype=torch.int32), w.softmax_scale, lens2)
    o2, l2 = run(w2)
    assert np.allclose(o2, o, rtol=1e-12, atol=1e-12)
    assert np.allclose(l2, l + math.log(2.0), rtol=0, atol=1e-12)


def test_row_layout_and_lse_transpose():
    w = wl.make_mla_workload([30, 11], h_q=16, s_q=3, page_size=8, seed=97)
    o, l = run(w)
    w.q = w.q[:, [2, 0, 1]].contiguous()            # permute the query tokens
    o2, l2 = run(w)
    assert np.array_equal(o2, o[:, [2, 0, 1]])
    assert np.array_equal(l2, l[:, :, [2, 0, 1]])
    w.q = w.q[:, :, torch.arange(15, -1, -1)].contiguous()   # and the heads
    o3, l3 = run(w)
    assert np.array_equal(o3, o2[:, :, ::-1])
    assert np.array_equal(l3, l2[:, ::-1, :])


def test_empty_sequence():
    w = wl.make_mla_workload([0, 5, 0], h_q=16, s_q=1, page_size=4, seed=98)
    o, l = run(w)
    for b in (0, 2):
        assert np.all(o[b] == 0) and np.all(np.isneginf(l[b]))
    assert np.all(np.isfinite(l[1]))


@pytest.mark.parametrize("slip", ["value_slice", "no_rope", "block_offset_swap", "lse_base2"])
def test_pins_catch_planted_mistakes(monkeypatch, slip):
    good_attend, good_slots = ml.attend_rows, ml.mla_slots

    def bad_attend(qg, k, v, scale):
        if slip == "value_slice":
            v = k[:, 64:]
        if slip == "no_rope":
            qg, k = qg[:, :512], k[:, :512]
        o, lse2 = good_attend(qg, k, v, scale)
        if slip == "lse_base2":
            lse2 = lse2 / math.log(2.0)           # the caller's ln 2 factor then yields log2
        return o, lse2

    def bad_slots(block_table, cache_seqlens, page_size, num_blocks=None):
        table = np.asarray(block_table, dtype=np.int64)
        out = []
        for b, n in enumerate(np.asarray(cache_seqlens)):
            t = np.arange(int(n))
            out.append(table[b, t % page_size % table.shape[1]] * page_size + t // page_size % page_size)
        return out

    if slip == "block_offset_swap":
        monkeypatch.setattr(ml, "mla_slots", bad_slots)
    else:
        monkeypatch.setattr(ml, "attend_rows", bad_attend)
    failed = False
    try:
        test_scalar_brute_force()
        test_one_token_closed_form()
        test_zero_query_and_duplicated_tokens()
    except (AssertionError, IndexError):
        failed = True
    finally:
        monkeypatch.setattr(ml, "attend_rows", good_attend)
        monkeypatch.setattr(ml, "mla_slots", good_slots)
    assert failed, slip
