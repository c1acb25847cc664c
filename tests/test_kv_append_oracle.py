"""Pins for the KV-append oracle (no GPU): what a row store must and must not touch."""
import pytest
import torch

import oracle.kv_append as ka


def _pool(p, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(p, 1, 4, 128, generator=g).to(torch.bfloat16),
            torch.randn(p, 1, 4, 128, generator=g).to(torch.bfloat16))


def _rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, 4, 128, generator=g).to(torch.bfloat16),
            torch.randn(n, 4, 128, generator=g).to(torch.bfloat16))


def test_valid_rows_land_and_nothing_else_changes():
    k, v = _pool(50, 1)
    kn, vn = _rows(6, 2)
    slots = torch.tensor([7, 0, 49, 13, 21, 30], dtype=torch.int32)
    k2, v2 = ka.kv_append_oracle(kn, vn, slots, k, v)
    for r, s in enumerate(slots.tolist()):
        assert torch.equal(k2[s, 0], kn[r]) and torch.equal(v2[s, 0], vn[r])
    untouched = [p for p in range(50) if p not in slots.tolist()]
    assert torch.equal(k2[untouched], k[untouched]) and torch.equal(v2[untouched], v[untouched])
    # inputs are not modified in place
    k0, v0 = _pool(50, 1)
    assert torch.equal(k, k0) and torch.equal(v, v0)


def test_invalid_slots_store_nothing():
    k, v = _pool(10, 3)
    kn, vn = _rows(4, 4)
    k2, v2 = ka.kv_append_oracle(kn, vn, torch.tensor([-1, 10, 11, -7], dtype=torch.int32), k, v)
    assert torch.equal(k2, k) and torch.equal(v2, v)


def test_order_of_distinct_rows_does_not_matter_and_repeat_is_idempotent():
    k, v = _pool(40, 5)
    kn, vn = _rows(8, 6)
    slots = torch.tensor([3, 9, 1, 38, 22, 15, 7, 30], dtype=torch.int32)
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(7))
    a = ka.kv_append_oracle(kn, vn, slots, k, v)
    b = ka.kv_append_oracle(kn[perm], vn[perm], slots[perm], k, v)
    c = ka.kv_append_oracle(kn, vn, slots, *a)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_empty_append():
    k, v = _pool(5, 8)
    kn = torch.empty(0, 4, 128, dtype=torch.bfloat16)
    k2, v2 = ka.kv_append_oracle(kn, kn, torch.empty(0, dtype=torch.int32), k, v)
    assert torch.equal(k2, k) and torch.equal(v2, v)


def test_append_then_decode_sees_the_new_token():
    """A token appended into a free page and referenced by kv_indices is attended to
    exactly like a token that was in the pool from the start."""
    from oracle import gqa_paged_decode_oracle
    k, v = _pool(20, 9)
    kn, vn = _rows(1, 10)
    q = torch.randn(1, 32, 128, generator=torch.Generator().manual_seed(11)).to(torch.bfloat16)
    k2, v2 = ka.kv_append_oracle(kn, vn, torch.tensor([17], dtype=torch.int32), k, v)
    indptr = torch.tensor([0, 4], dtype=torch.int32)
    o_a, l_a = gqa_paged_decode_oracle(q, k2, v2, indptr, torch.tensor([2, 5, 11, 17], dtype=torch.int32), 0.0884)
    kd, vd = k.clone(), v.clone()
    kd[17, 0] = kn[0]
    vd[17, 0] = vn[0]
    o_b, l_b = gqa_paged_decode_oracle(q, kd, vd, indptr, torch.tensor([2, 5, 11, 17], dtype=torch.int32), 0.0884)
    assert (o_a == o_b).all() and (l_a == l_b).all()


@pytest.mark.parametrize("slip", ["swap_kv", "slot_off_by_one", "negative_wraps", "upper_bound_inclusive",
                                  "stores_in_place"])
def test_pins_catch_planted_mistakes(monkeypatch, slip):
    """Each plausible slip in the row store fails at least one pin above."""
    good = ka.kv_append_oracle

    def bad(k_new, v_new, slots, k_cache, v_cache):
        k_out = k_cache if slip == "stores_in_place" else k_cache.clone()
        v_out = v_cache if slip == "stores_in_place" else v_cache.clone()
        num_pages = k_cache.shape[0]
        for r, slot in enumerate(slots.tolist()):
            if slip == "slot_off_by_one":
                slot += 1
            ok = (slot < num_pages if slip == "negative_wraps" else
                  0 <= slot <= num_pages if slip == "upper_bound_inclusive" else 0 <= slot < num_pages)
            if ok:
                k_out[slot, 0] = v_new[r] if slip == "swap_kv" else k_new[r]
                v_out[slot, 0] = k_new[r] if slip == "swap_kv" else v_new[r]
        return k_out, v_out

    monkeypatch.setattr(ka, "kv_append_oracle", bad)
    failed = False
    try:
        test_valid_rows_land_and_nothing_else_changes()
        test_invalid_slots_store_nothing()
        test_order_of_distinct_rows_does_not_matter_and_repeat_is_idempotent()
        test_empty_append()
    except (AssertionError, IndexError):
        failed = True
    finally:
        monkeypatch.setattr(ka, "kv_append_oracle", good)
    assert failed, slip
