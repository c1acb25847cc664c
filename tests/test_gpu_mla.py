"""Dense MLA paged decode on the GPU against the float64 oracle (oracle/mla.py).

The flash_mla_with_kvcache page's dense path: one latent KV head of 576 values
(512 of them also V), blocks through a block table, natural-log LSE in the
page's [B, h_q, s_q] layout. Tolerances are the dense path's: |dO| <= 2e-2 +
2e-2 |O_ref|, |dlse| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle.mla as ml
from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


@pytest.fixture(autouse=True)
def _defaults(cuda_device):
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
    _lib.gqa_mla_set_tuning(0)
    yield
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
    _lib.gqa_mla_set_tuning(0)


def gpu_mla(w, with_lse=True):
    g = w.to("cuda")
    out, lse = _lib.mla_run(g.q, g.kv_cache, g.block_table, g.cache_seqlens, w.softmax_scale, with_lse=with_lse)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy(), (lse.cpu().double().numpy() if lse is not None else None)


def check(w, out, lse, seqs=None):
    o_ref, l_ref = ml.mla_decode_oracle(w.q, w.kv_cache, w.block_table, w.cache_seqlens, w.softmax_scale, seqs)
    sel = list(range(w.batch)) if seqs is None else list(seqs)
    o, orf = out[sel], o_ref[sel]
    bad = np.abs(o - orf) > O_ATOL + O_RTOL * np.abs(orf)
    assert not bad.any(), f"{bad.sum()} O elements out of tolerance, max |dO| {np.abs(o - orf).max():.3g}"
    if lse is not None:
        l, lrf = lse[sel], l_ref[sel]
        assert np.array_equal(np.isneginf(l), np.isneginf(lrf))
        fin = np.isfinite(lrf)
        assert np.all(np.abs(l[fin] - lrf[fin]) <= LSE_ATOL), np.abs(l[fin] - lrf[fin]).max()
    empty = np.isneginf(l_ref[sel]).all(axis=(1, 2))
    assert np.all(o[empty] == 0)


CASES = [
    ([1, 0, 17, 64, 65, 300], 16, 1, 64, 1),
    ([2000, 5, 700], 32, 1, 64, 2),             # two row groups
    ([900, 33, 0, 128], 16, 2, 16, 3),          # two query tokens per sequence
    ([500, 77], 8, 2, 1, 4),                    # page size 1, 8 heads x 2 tokens = 16 rows
    ([4000, 3, 1500], 16, 1, 128, 5),
    ([6000, 6000], 64, 1, 64, 6),               # rows cut across CTAs in 4 row groups
    ([31, 32, 33, 95, 96, 97], 16, 1, 32, 7),   # tiles of exactly one block
]


# kernel 1: the tensor-memory kernel (blocks of 32, 64, 128; mma.sync otherwise); 0: the default (mma.sync)
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("lens,h_q,s_q,ps,seed", CASES)
def test_mla_matches_oracle(lens, h_q, s_q, ps, seed, kernel):
    assert _lib.gqa_mla_set_tuning(kernel) == 0
    w = wl.make_mla_workload(lens, h_q, s_q, ps, seed)
    out, lse = gpu_mla(w)
    check(w, out, lse)


def test_mla_kernels_agree():
    """The tensor-memory and mma.sync kernels on the same inputs: both within tolerance of
    the oracle above; here, within twice that of each other on every element."""
    w = wl.make_mla_workload([3000, 64, 0, 1, 777], 32, 1, 64, seed=21)
    outs = []
    for kernel in (1, 3):
        assert _lib.gqa_mla_set_tuning(kernel) == 0
        outs.append(gpu_mla(w))
    (o1, l1), (o3, l3) = outs
    assert np.all(np.abs(o1 - o3) <= 2 * (O_ATOL + O_RTOL * np.abs(o3)))
    fin = np.isfinite(l3)
    assert np.array_equal(np.isneginf(l1), np.isneginf(l3))
    assert np.all(np.abs(l1[fin] - l3[fin]) <= 2 * LSE_ATOL)


def test_mla_invalid_blocks_and_long_lengths():
    w = wl.make_mla_workload([700, 300, 129], 16, 1, 64, seed=11)
    w.block_table[0, 3] = -1                    # a hole: tokens 192..255 of sequence 0 are left out
    w.block_table[1, 1] = w.kv_cache.shape[0] + 7
    w.cache_seqlens[2] = 10 ** 6                # past the table: counts as width * page_size
    w.lens[2] = 10 ** 6
    out, lse = gpu_mla(w)
    check(w, out, lse)


@pytest.mark.parametrize("tuning", [(40, 8, 0, 0, 0, 0, 0, 0, 500, 16), (7, 1, 0, 0, 0, 0, 0, 13, 400, 4),
                                    (300, 1, 0, 0, 0, 0, 0, -1), (1, 0, 0, 0, 0, 0, 0, -1)])
def test_mla_split_plans(tuning):
    assert _lib.gqa_paged_decode_set_tuning(*tuning) == 0
    w = wl.make_mla_workload([3000, 40, 1200, 0, 7], 16, 1, 64, seed=12)
    out, lse = gpu_mla(w)
    check(w, out, lse)


@pytest.mark.parametrize("kernel", [1, 3, 4])
@pytest.mark.parametrize("tuning", [(0, 0, 0, 0, 0, 0), (50, 4, 0, 0, 0, 0, 0, 40, 300, 8)])
def test_mla_kernel_choices(kernel, tuning):
    assert _lib.gqa_mla_set_tuning(kernel) == 0
    assert _lib.gqa_paged_decode_set_tuning(*tuning) == 0
    w = wl.make_mla_workload([2500, 1, 0, 640, 17, 900], 16, 2, 64, seed=14)
    out, lse = gpu_mla(w)
    check(w, out, lse)


def test_mla_without_lse():
    w = wl.make_mla_workload([800, 90], 16, 1, 64, seed=13)
    out, lse = gpu_mla(w, with_lse=False)
    assert lse is None
    check(w, out, None)


@pytest.mark.parametrize("wide", [False, True])
def test_mla_config_every_sequence(wide):
    """The bench's MLA workloads (16 and 64 query heads) at full size, every
    sequence against the oracle."""
    w = wl.make_mla_config(wide)
    out, lse = gpu_mla(w)
    check(w, out, lse)


@pytest.mark.parametrize("kernel", [0, 1])
def test_mla_int64_slot_addressing(kernel):
    """Blocks past 2^31 / (64 * 1152) sit more than 2^31 bytes into the latent pool."""
    assert _lib.gqa_mla_set_tuning(kernel) == 0
    ps = 64
    base = (1 << 31) // (ps * 1152) + 1
    num_blocks = base + 64
    small = wl.make_mla_workload([700, 0, 130], 16, 1, ps, seed=15)
    g = torch.Generator().manual_seed(7)
    used = (small.block_table >= 0)
    high = torch.randperm(num_blocks - base, generator=g)[: int(used.sum())] + base
    table = small.block_table.clone()
    table[used] = high.to(torch.int32)
    kv = torch.zeros((num_blocks, ps, 1, 576), dtype=torch.bfloat16, device="cuda")
    kv[table[used].long().cuda()] = small.kv_cache[small.block_table[used].long()].cuda()
    out, lse = _lib.mla_run(small.q.cuda(), kv, table.cuda(), small.cache_seqlens.cuda(), small.softmax_scale)
    torch.cuda.synchronize()
    check(small, out.float().cpu().double().numpy(), lse.cpu().double().numpy())
    del kv


@pytest.mark.parametrize("lens,h_q,s_q,ps,seed,ctas", [
    ([129, 1, 0, 255, 256, 257], 48, 1, 64, 31, 0),       # three row groups per sequence
    ([600, 2, 130], 16, 3, 128, 32, 0),                   # three query tokens: 48 rows
    ([128] * 9 + [0, 1, 127], 16, 1, 32, 33, 5),          # tiles of exactly one 128-token window, few CTAs
    ([5000, 17, 4100], 16, 1, 64, 34, 77),                # pieces cut inside 128-token tiles
    (list(range(1, 200, 7)), 16, 1, 64, 35, 0),           # many short sequences
])
def test_mla_tensor_memory_shapes(lens, h_q, s_q, ps, seed, ctas):
    """Tile edges of the tensor-memory kernel (128-token windows, 32- or 64-row copies, row groups),
    against the oracle, and against the mma.sync kernel on the same inputs."""
    w = wl.make_mla_workload(lens, h_q, s_q, ps, seed)
    assert _lib.gqa_paged_decode_set_tuning(ctas, 0, 0, 0, 0, 0) == 0
    outs = []
    for kernel in (1, 3):
        assert _lib.gqa_mla_set_tuning(kernel) == 0
        outs.append(gpu_mla(w))
    check(w, *outs[0])
    (o1, l1), (o3, l3) = outs
    assert np.all(np.abs(o1 - o3) <= 2 * (O_ATOL + O_RTOL * np.abs(o3)))


@pytest.mark.parametrize("lens,h_q,s_q,ps,seed,ctas,kernel", [
    ([900, 1, 0, 130], 64, 1, 64, 41, 0, 0),              # one 64-row piece per sequence (default kernel)
    ([700, 257], 128, 1, 64, 42, 0, 1),                   # two 64-row groups
    ([600, 33, 128], 32, 2, 32, 43, 0, 1),                # 2 query tokens x 32 heads, 32-row copies
    ([3000, 5, 2000], 64, 1, 128, 44, 9, 1),              # few CTAs: several pieces and Q reloads per CTA
    ([4096, 4096, 4095], 64, 1, 64, 45, 300, 1),          # many pieces per sequence: the merge's long chains
    ([900, 1, 0, 130], 32, 1, 64, 47, 0, 1),              # 32-row pieces
    ([700, 257, 33], 16, 2, 64, 48, 0, 1),                # 2 query tokens x 16 heads: 32-row pieces
    ([600, 129], 96, 1, 32, 49, 0, 1),                    # three 32-row groups, 32-row copies
    ([3000, 5, 2000], 32, 1, 128, 50, 9, 1),              # 32-row pieces, few CTAs: Q reloads per CTA
    ([4096, 4095], 32, 1, 64, 51, 300, 1),                # 32-row pieces, many pieces per sequence
])
def test_mla_wide_pieces(lens, h_q, s_q, ps, seed, ctas, kernel):
    """64- and 32-row pieces of the tensor-memory kernel (a sequence's rows in multiples of 64 or 32),
    against the oracle and against the mma.sync kernel (16-row pieces) on the same inputs."""
    w = wl.make_mla_workload(lens, h_q, s_q, ps, seed)
    assert _lib.gqa_paged_decode_set_tuning(ctas, 0, 0, 0, 0, 0) == 0
    assert _lib.gqa_mla_set_tuning(kernel) == 0
    o1, l1 = gpu_mla(w)
    check(w, o1, l1)
    assert _lib.gqa_mla_set_tuning(3) == 0
    o3, l3 = gpu_mla(w)
    assert np.all(np.abs(o1 - o3) <= 2 * (O_ATOL + O_RTOL * np.abs(o3)))


def test_mla_wide_holes_and_long_lengths():
    w = wl.make_mla_workload([700, 300, 129], 64, 1, 64, seed=46)
    w.block_table[0, 3] = -1                    # a hole: tokens 192..255 of sequence 0 are left out
    w.block_table[1, 1] = w.kv_cache.shape[0] + 7
    w.cache_seqlens[2] = 10 ** 6                # past the table: counts as width * page_size
    w.lens[2] = 10 ** 6
    assert _lib.gqa_mla_set_tuning(1) == 0
    out, lse = gpu_mla(w)
    check(w, out, lse)


@pytest.mark.parametrize("kernel,h_q", [(0, 16), (1, 16), (0, 64), (1, 64)])
def test_mla_batch_past_grid(kernel, h_q):
    """2000 sequences of 0-69 tokens, more than either kernel has CTAs: every empty sequence is written
    (O = 0, LSE = -inf) over outputs that start as garbage, and each CTA range walks many sequences."""
    assert _lib.gqa_mla_set_tuning(kernel) == 0
    lens = torch.randint(0, 70, (2000,), generator=torch.Generator().manual_seed(61)).tolist()
    lens[:3] = [0, 0, 0]
    w = wl.make_mla_workload(lens, h_q, 1, 64, 62)
    g = w.to("cuda")
    out = torch.full((w.batch, 1, h_q, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.batch, h_q, 1), 7.0, dtype=torch.float32, device="cuda")
    _lib.mla_run(g.q, g.kv_cache, g.block_table, g.cache_seqlens, w.softmax_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    empty = [b for b, n in enumerate(lens) if n == 0]
    assert np.all(o[empty] == 0.0) and np.all(np.isneginf(l[empty]))
    check(w, o, l)
