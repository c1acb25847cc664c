"""GPU parity of the KV-cache append (byte copies: bit-exact against the oracle)."""
import numpy as np
import pytest
import torch

from oracle import gqa_paged_decode_oracle
from oracle.kv_append import kv_append_oracle
from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    _lib.load()


def _make(num_pages, n, seed, n_invalid=0):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(num_pages, 1, 4, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(num_pages, 1, 4, 128, generator=g).to(torch.bfloat16)
    kn = torch.randn(n, 4, 128, generator=g).to(torch.bfloat16)
    vn = torch.randn(n, 4, 128, generator=g).to(torch.bfloat16)
    slots = torch.randperm(num_pages, generator=g)[:n].to(torch.int32)
    if n_invalid:
        where = torch.randperm(n, generator=g)[:n_invalid]
        bad = torch.tensor([-1, num_pages, num_pages + 7, -100], dtype=torch.int32)
        slots[where] = bad[torch.arange(n_invalid) % 4]
    return k, v, kn, vn, slots


@pytest.mark.parametrize("num_pages,n,n_invalid", [(10, 1, 0), (64, 64, 0), (1000, 333, 40), (5000, 4096, 0),
                                                   (200000, 150001, 1000)])
def test_append_bit_exact(num_pages, n, n_invalid):
    k, v, kn, vn, slots = _make(num_pages, n, seed=num_pages + n, n_invalid=n_invalid)
    kd, vd = k.cuda(), v.cuda()
    _lib.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), kd, vd)
    torch.cuda.synchronize()
    ko, vo = kv_append_oracle(kn, vn, slots, k, v)
    assert torch.equal(kd.cpu(), ko) and torch.equal(vd.cpu(), vo)


def test_append_nothing_and_non_default_stream():
    k, v, kn, vn, slots = _make(32, 8, seed=3)
    kd, vd = k.cuda(), v.cuda()
    _lib.kv_append(kn[:0].cuda(), vn[:0].cuda(), slots[:0].cuda(), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _lib.kv_append(kn.cuda(), vn.cuda(), slots.cuda(), kd, vd)
    s.synchronize()
    ko, vo = kv_append_oracle(kn, vn, slots, k, v)
    assert torch.equal(kd.cpu(), ko) and torch.equal(vd.cpu(), vo)


def test_append_then_decode_step():
    """One decode step of a serving loop: append one new token per sequence into free
    pages, extend the page table by those pages, decode; compare with the oracle."""
    g = torch.Generator().manual_seed(12)
    lens = [5, 0, 300, 1024, 77]
    total, pool = sum(lens), sum(lens) + 64
    k = torch.randn(pool, 1, 4, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(pool, 1, 4, 128, generator=g).to(torch.bfloat16)
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    used, free = perm[:total], perm[total:]
    q = torch.randn(len(lens), 32, 128, generator=g).to(torch.bfloat16)
    kn = torch.randn(len(lens), 4, 128, generator=g).to(torch.bfloat16)
    vn = torch.randn(len(lens), 4, 128, generator=g).to(torch.bfloat16)
    new_slots = free[: len(lens)].clone()
    idx, ptr, off = [], [0], 0
    for b, n in enumerate(lens):
        idx += used[off:off + n].tolist() + [int(new_slots[b])]
        off += n
        ptr.append(len(idx))
    indptr = torch.tensor(ptr, dtype=torch.int32)
    indices = torch.tensor(idx, dtype=torch.int32)
    kd, vd = k.cuda(), v.cuda()
    _lib.kv_append(kn.cuda(), vn.cuda(), new_slots.cuda(), kd, vd)
    out, lse = _lib.run(q.cuda(), kd, vd, indptr.cuda(), indices.cuda())
    torch.cuda.synchronize()
    ko, vo = kv_append_oracle(kn, vn, new_slots, k, v)
    o_ref, l_ref = gqa_paged_decode_oracle(q, ko, vo, indptr, indices, 1.0 / np.sqrt(128))
    o = out.float().cpu().double().numpy()
    assert np.all(np.abs(o - o_ref) <= 2e-2 + 2e-2 * np.abs(o_ref))
    assert np.abs(lse.cpu().double().numpy() - l_ref).max() <= 1e-3
