"""Pins for the float64 oracle: brute force, closed forms and invariants.

None of these compares the oracle with itself. Each check is chosen so that a
plausible slip in the oracle (natural-log LSE, wrong KV-head mapping, dropped
sm_scale, swapped K/V, a missing max shift that overflows, wrong empty-sequence
value) fails at least one of them; ``test_pins_catch_planted_mistakes`` plants
several such slips and confirms it.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_gqa_split_gb300 import workloads as wl

H, G, D = 32, 4, 128


def _brute(w):
    """Pure-Python scalar attention: math.fsum sums, no max subtraction."""
    q = w.q.to(torch.float64).tolist()
    k = w.k_cache.to(torch.float64).tolist()
    v = w.v_cache.to(torch.float64).tolist()
    indptr = w.kv_indptr.tolist()
    idx = w.kv_indices.tolist()
    outs, lses = [], []
    for b in range(len(indptr) - 1):
        pages = idx[indptr[b]:indptr[b + 1]]
        ob, lb = [], []
        for h in range(H):
            g = h // 8
            if not pages:
                ob.append([0.0] * D)
                lb.append(-math.inf)
                continue
            s = [w.sm_scale * math.fsum(q[b][h][d] * k[p][0][g][d] for d in range(D)) for p in pages]
            e = [math.exp(x) for x in s]
            z = math.fsum(e)
            ob.append([math.fsum(e[j] * v[p][0][g][d] for j, p in enumerate(pages)) / z
                       for d in range(D)])
            lb.append(math.log2(z))
        outs.append(ob)
        lses.append(lb)
    return np.array(outs), np.array(lses)


def _run(w, **kw):
    return orc.gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices,
                                       w.sm_scale, **kw)


def _score(w, b, h, j):
    """sm_scale * q.k for token j of sequence b, head h, by math.fsum."""
    g = h // 8
    p = int(w.kv_indices[int(w.kv_indptr[b]) + j])
    qv = w.q[b, h].to(torch.float64).tolist()
    kv = w.k_cache[p, 0, g].to(torch.float64).tolist()
    return w.sm_scale * math.fsum(a * c for a, c in zip(qv, kv))


def test_brute_force_tiny():
    w = wl.make_workload([1, 3, 0, 7, 20, 2], seed=11, pool_factor=1.5)
    o, l = _run(w)
    ob, lb = _brute(w)
    assert np.allclose(o, ob, rtol=1e-12, atol=1e-13)
    fin = np.isfinite(lb)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.allclose(l[fin], lb[fin], rtol=0, atol=1e-12)


def test_single_token_gives_v_and_scaled_score():
    w = wl.make_workload([1, 1, 1], seed=5, pool_factor=3.0)
    o, l = _run(w)
    for b in range(3):
        p = int(w.kv_indices[b])
        for h in range(H):
            g = h // 8
            assert np.array_equal(o[b, h], w.v_cache[p, 0, g].to(torch.float64).numpy())
            assert abs(l[b, h] - _score(w, b, h, 0) / math.log(2.0)) < 1e-12


def test_constant_v_gives_constant():
    w = wl.make_workload([9, 40, 3], seed=6)
    consts = [0.75, -1.5, 3.0, 0.125]
    for g, c in enumerate(consts):
        w.v_cache[:, :, g, :] = c
    o, _ = _run(w)
    for h in range(H):
        assert np.allclose(o[:, h, :], consts[h // 8], rtol=0, atol=1e-13)


def test_empty_sequence_zero_and_minus_inf():
    w = wl.make_workload([0, 5, 0, 0], seed=7)
    o, l = _run(w)
    for b in (0, 2, 3):
        assert np.all(o[b] == 0.0)
        assert np.all(np.isneginf(l[b]))
    assert np.all(np.isfinite(l[1]))


def test_all_empty_batch():
    w = wl.make_workload([0, 0], seed=8)
    o, l = _run(w)
    assert np.all(o == 0.0) and np.all(np.isneginf(l))


def test_page_relabelling_is_bit_identical():
    w = wl.make_workload([17, 5, 33], seed=9, pool_factor=2.0)
    o, l = _run(w)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(w.num_pages, generator=g)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    idx2 = perm[w.kv_indices.long()].to(torch.int32)
    o2, l2 = orc.gqa_paged_decode_oracle(w.q, k2, v2, w.kv_indptr, idx2, w.sm_scale)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_token_order_permutation():
    w = wl.make_workload([29, 64], seed=10)
    o, l = _run(w)
    idx = w.kv_indices.clone()
    g = torch.Generator().manual_seed(3)
    for b in range(2):
        lo, hi = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        idx[lo:hi] = idx[lo:hi][torch.randperm(hi - lo, generator=g)]
    o2, l2 = orc.gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, idx, w.sm_scale)
    assert np.allclose(o, o2, rtol=1e-12, atol=1e-13)
    assert np.allclose(l, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", ["q_zero", "scale_zero"])
def test_uniform_scores_give_mean_and_log2_n(mode):
    lens = [1, 6, 31]
    w = wl.make_workload(lens, seed=12)
    if mode == "q_zero":
        w.q.zero_()
    else:
        w.sm_scale = 0.0
    o, l = _run(w)
    for b, n in enumerate(lens):
        lo = int(w.kv_indptr[b])
        pages = w.kv_indices[lo:lo + n].long()
        for g in range(G):
            mean = w.v_cache[pages, 0, g].to(torch.float64).numpy().mean(axis=0)
            for h in range(8 * g, 8 * g + 8):
                assert np.allclose(o[b, h], mean, rtol=1e-12, atol=1e-13)
                assert abs(l[b, h] - math.log2(n)) < 1e-12


def test_duplicating_tokens_adds_one_to_lse():
    w = wl.make_workload([5, 12], seed=13)
    o, l = _run(w)
    idx, ptr = [], [0]
    for b in range(2):
        lo, hi = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        seg = w.kv_indices[lo:hi].tolist()
        idx += seg + seg
        ptr.append(len(idx))
    o2, l2 = orc.gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, torch.tensor(ptr, dtype=torch.int32),
                                         torch.tensor(idx, dtype=torch.int32), w.sm_scale)
    assert np.allclose(o2, o, rtol=1e-12, atol=1e-13)
    assert np.allclose(l2, l + 1.0, rtol=0, atol=1e-12)


def test_two_token_closed_form():
    w = wl.make_workload([2], seed=14)
    o, l = _run(w)
    p0, p1 = (int(x) for x in w.kv_indices)
    for h in range(H):
        g = h // 8
        s0, s1 = _score(w, 0, h, 0), _score(w, 0, h, 1)
        assert abs(l[0, h] - math.log2(math.exp(s0) + math.exp(s1))) < 1e-12
        a = 1.0 / (1.0 + math.exp(s1 - s0))
        want = a * w.v_cache[p0, 0, g].double().numpy() + (1 - a) * w.v_cache[p1, 0, g].double().numpy()
        assert np.allclose(o[0, h], want, rtol=1e-12, atol=1e-13)


def test_lse_is_base_two_of_natural_sum():
    """Scores fixed by construction: s = [0, 1, 1, 2] gives lse = log2(1 + 2e + e^2)."""
    lens = [4]
    w = wl.make_workload(lens, seed=15)
    w.sm_scale = 1.0
    w.q.zero_()
    w.q[0, :, 0] = 1.0
    for j, s in enumerate([0.0, 1.0, 1.0, 2.0]):
        p = int(w.kv_indices[j])
        w.k_cache[p, 0, :, :] = 0.0
        w.k_cache[p, 0, :, 0] = s
    _, l = _run(w)
    want = math.log2(1.0 + 2.0 * math.e + math.e ** 2)
    assert np.allclose(l[0], want, rtol=0, atol=1e-13)


def test_gqa_head_mapping_is_contiguous_groups():
    """q head h reads KV head h // 8: give each KV head its own constant V."""
    w = wl.make_workload([7, 19], seed=16)
    for g in range(G):
        w.v_cache[:, :, g, :] = float(g + 1)
    o, _ = _run(w)
    for h in range(H):
        assert np.allclose(o[:, h, :], h // 8 + 1, atol=1e-13)


def test_large_scores_do_not_overflow():
    """q ~ 3 N(0,1) at sm_scale 1 gives scores of hundreds: two-pass softmax stays finite."""
    w = wl.make_workload([50], seed=17, q_std=30.0)
    w.sm_scale = 1.0
    o, l = _run(w)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    assert l.max() > 100.0


def test_sampled_rows_match_full():
    w = wl.make_workload([3, 9, 0, 4], seed=18)
    o, l = _run(w)
    os_, ls = _run(w, seqs=[1, 2])
    assert np.array_equal(os_[[1, 2]], o[[1, 2]]) and np.array_equal(ls[[1, 2]], l[[1, 2]])
    assert np.all(np.isnan(os_[[0, 3]]))


@pytest.mark.parametrize("pieces", [[10], [1, 9], [3, 3, 4], [0, 5, 0, 5], [1] * 10])
def test_split_merge_equals_whole(pieces):
    """Merging oracle partials over a partition of the tokens reproduces the whole."""
    n = sum(pieces)
    w = wl.make_workload([n], seed=19)
    o, l = _run(w)
    parts = []
    lo = 0
    for c in pieces:
        sub_idx = w.kv_indices[lo:lo + c]
        po, pl = orc.gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache,
                                             torch.tensor([0, c], dtype=torch.int32), sub_idx, w.sm_scale)
        parts.append((po[0], pl[0]))
        lo += c
    mo, ml = orc.merge_partials(parts)
    assert np.allclose(mo, o[0], rtol=1e-12, atol=1e-13)
    assert np.allclose(ml, l[0], rtol=0, atol=1e-12)


def test_merge_of_only_empty_parts():
    z = (np.zeros((H, D)), np.full(H, -np.inf))
    mo, ml = orc.merge_partials([z, z])
    assert np.all(mo == 0.0) and np.all(np.isneginf(ml))


def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant slips in the oracle and confirm the pins above detect each one."""
    # 1) natural-log LSE instead of base 2
    monkeypatch.setattr(orc, "LN2", 1.0)
    with pytest.raises(AssertionError):
        test_lse_is_base_two_of_natural_sum()
    monkeypatch.undo()

    # 2) K and V swapped
    real_oracle = orc.gqa_paged_decode_oracle

    def swapped_oracle(q, k, v, ip, ix, sc, seqs=None):
        return real_oracle(q, v, k, ip, ix, sc, seqs)

    monkeypatch.setattr(orc, "gqa_paged_decode_oracle", swapped_oracle)
    with pytest.raises(AssertionError):
        test_constant_v_gives_constant()
    monkeypatch.undo()

    # 3) interleaved head mapping (h % 4) instead of contiguous groups (h // 8)
    real_attend = orc.attend_rows

    def interleaved_oracle(q, k, v, ip, ix, sc, seqs=None):
        qp = q[:, [((h % 4) * 8 + h // 4) for h in range(H)], :]
        return real_oracle(qp, k, v, ip, ix, sc, seqs)

    monkeypatch.setattr(orc, "gqa_paged_decode_oracle", interleaved_oracle)
    with pytest.raises(AssertionError):
        test_brute_force_tiny()
    monkeypatch.undo()

    # 4) sm_scale dropped
    def unscaled(qg, k, v, sm_scale):
        return real_attend(qg, k, v, 1.0)

    monkeypatch.setattr(orc, "attend_rows", unscaled)
    with pytest.raises(AssertionError):
        test_single_token_gives_v_and_scaled_score()
    monkeypatch.undo()

    # 5) no max shift: exp overflows on large scores
    def unshifted(qg, k, v, sm_scale):
        if k.shape[0] == 0:
            return real_attend(qg, k, v, sm_scale)
        s = sm_scale * (qg @ k.T)
        with np.errstate(over="ignore", invalid="ignore"):
            e = np.exp(s)
            lsum = e.sum(axis=1, keepdims=True)
            return (e @ v) / lsum, np.log(lsum[:, 0]) / orc.LN2

    monkeypatch.setattr(orc, "attend_rows", unshifted)
    with pytest.raises(AssertionError):
        test_large_scores_do_not_overflow()
    monkeypatch.undo()

    # 6) empty sequence giving +inf instead of -inf
    def plus_inf(qg, k, v, sm_scale):
        o, l = real_attend(qg, k, v, sm_scale)
        return o, (np.full_like(l, np.inf) if k.shape[0] == 0 else l)

    monkeypatch.setattr(orc, "attend_rows", plus_inf)
    with pytest.raises(AssertionError):
        test_empty_sequence_zero_and_minus_inf()
    monkeypatch.undo()


def test_pattern_fixture_regression():
    """The oracle reproduces the stored values for the formula-defined workload."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "pattern_oracle.json")
    with open(path) as f:
        doc = json.load(f)
    w = wl.make_pattern_workload()
    o, l = _run(w)
    want_l = np.array(doc["lse"], dtype=np.float64)
    assert np.array_equal(np.isneginf(want_l), np.isneginf(l))
    fin = np.isfinite(want_l)
    assert np.allclose(l[fin], want_l[fin], rtol=0, atol=1e-12)
    assert np.allclose([[o[b, h].sum() for h in range(H)] for b in range(w.batch)],
                       doc["o_row_sums"], rtol=1e-12, atol=1e-12)
    for key, row in doc["o_rows"].items():
        b, h = (int(x) for x in key.split(","))
        assert np.allclose(o[b, h], row, rtol=1e-12, atol=1e-13)
    # the empty middle sequence is stored as zeros / -inf
    assert np.all(np.isneginf(want_l[1]))
