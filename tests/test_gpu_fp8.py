"""Paged GQA decode over an FP8 (e4m3, per-128 fp32 scale) cache, on the GPU,
against the float64 oracle over the same FP8 rows (oracle/fp8.py).

The tolerances are the dense path's: |dO| <= 2e-2 + 2e-2 |O_ref|, |dlse| <= 1e-3.
The oracle dequantizes the very bytes the kernel reads, so the comparison
measures the kernel's arithmetic, not the quantization of the inputs.
"""
import numpy as np
import pytest
import torch

import oracle.fp8 as f8
from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


@pytest.fixture(autouse=True)
def _defaults(cuda_device):
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
    yield
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)


@pytest.fixture(params=[16, 32], ids=["stage16", "stage32"])
def f8_stage(request):
    """Both FP8 stage sizes (16 or 32 tokens per pipeline stage, 2-deep ring)."""
    assert _lib.gqa_paged_decode_set_tuning(0, 0, 4, request.param, 2, _lib.GATHER_LSU_F8) == 0
    return request.param


def gpu_fp8(w):
    g = w.to("cuda")
    out, lse = _lib.run_fp8(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy()


def check(w, out, lse, seqs=None):
    o_ref, l_ref = f8.gqa_paged_decode_fp8_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale,
                                                  seqs)
    sel = list(range(w.batch)) if seqs is None else list(seqs)
    o, orf, l, lrf = out[sel], o_ref[sel], lse[sel], l_ref[sel]
    bad = np.abs(o - orf) > O_ATOL + O_RTOL * np.abs(orf)
    assert not bad.any(), f"{bad.sum()} O elements out of tolerance, max |dO| {np.abs(o - orf).max():.3g}"
    assert np.array_equal(np.isneginf(l), np.isneginf(lrf))
    fin = np.isfinite(lrf)
    assert np.all(np.abs(l[fin] - lrf[fin]) <= LSE_ATOL), np.abs(l[fin] - lrf[fin]).max()
    assert np.all(o[~fin.any(axis=1)] == 0)


@pytest.mark.parametrize("lens", [[1], [0], [0, 0, 3], [15, 16, 17], [255, 256, 257, 0, 129],
                                  [3, 1000, 0, 77, 2049, 1, 16, 600], list(range(1, 41))])
def test_fp8_edge_and_ragged(lens, f8_stage):
    w = wl.make_fp8_workload(lens, seed=len(lens) + 300, pool_factor=1.5)
    out, lse = gpu_fp8(w)
    check(w, out, lse)


@pytest.mark.parametrize("tuning", [(0, 0, 4, 16, 2, 0), (0, 0, 4, 16, 3, 0), (0, 0, 4, 16, 4, 0),
                                    (40, 8, 4, 16, 2, 0, 0, 0, 500, 16), (7, 1, 4, 16, 3, 0, 0, 13, 400, 4),
                                    (300, 1, 4, 16, 2, 0, 4), (60, 8, 4, 16, 4, 0, -1, -1),
                                    (0, 0, 4, 32, 2, 2), (0, 0, 4, 16, 3, 2), (40, 8, 4, 32, 2, 2, 0, 0, 500, 16),
                                    (7, 1, 4, 32, 2, 2, 0, 13, 400, 4), (300, 1, 4, 32, 2, 2, 4),
                                    (60, 8, 4, 32, 2, 2, -1, -1), (5, 40, 4, 32, 2, 2, 0, 3, 300, 33)])
def test_fp8_variants_and_splits(tuning):
    assert _lib.gqa_paged_decode_set_tuning(*tuning) == 0
    w = wl.make_fp8_workload([5000, 3, 17, 0, 900, 1, 64], seed=301, pool_factor=1.1)
    out, lse = gpu_fp8(w)
    check(w, out, lse)


def test_fp8_large_queries(f8_stage):
    """|q| near 1e4: the f16 form of Q needs its power-of-two rescale."""
    w = wl.make_fp8_workload([700, 64, 3], seed=302, q_std=1.0)
    w.q.mul_(8192.0)                                   # exact in bf16 (a power of two)
    w.sm_scale = w.sm_scale / 8192.0 / 4.0             # keep the logits in a sane range
    out, lse = gpu_fp8(w)
    check(w, out, lse)


def _scale_rows(cache, up, down):
    sc = cache[:, 512:].clone().view(torch.float32)          # [P, 4]
    sc[0::7] *= up
    sc[3::11] *= down
    cache[:, 512:] = sc.view(torch.uint8)


def test_fp8_extreme_and_zero_scales(f8_stage):
    """K scales 2^4 up and down on some tokens (sharp softmax), V scales 2^5 up
    and down on others (the P operand's running normaliser), all-zero rows
    elsewhere. Much larger spreads leave the test's absolute tolerances, not
    the kernel: logits near 10^6 have an fp32 ulp far above 1e-3 in the LSE,
    and V scales 2^20 apart within one sequence push the small-scale tokens'
    probabilities into f16's subnormal range, an error that grows with the
    largest V value as it does for any 16-bit P operand."""
    w = wl.make_fp8_workload([900, 300, 40], seed=303)
    _scale_rows(w.k_cache, 2.0 ** 4, 2.0 ** -4)
    _scale_rows(w.v_cache, 2.0 ** 5, 2.0 ** -5)
    w.v_cache[5::13, :512] = 0                                   # zero codes: value 0 whatever the scale
    w.k_cache[9::17, :] = 0                                      # zero codes and zero scales
    out, lse = gpu_fp8(w)
    check(w, out, lse)


@pytest.mark.parametrize("name", ["mid", "skewed"])
def test_fp8_named_workloads_every_sequence(name, f8_stage):
    """The mid and skewed batches over an FP8 copy of their caches, every
    sequence against the FP8 oracle."""
    w = wl.make_fp8_config(name)
    out, lse = gpu_fp8(w)
    check(w, out, lse)


def test_fp8_int64_page_addressing(f8_stage):
    """Pages above 2^31 / 528 sit more than 2^31 bytes into each 528-byte-per-page pool."""
    base = (1 << 31) // _lib.FP8_ROW_BYTES + 1
    num_pages = base + 4096
    small = wl.make_fp8_workload([40, 0, 300], seed=61)
    g = torch.Generator().manual_seed(6)
    high = torch.randperm(num_pages - base, generator=g)[: small.total_tokens] + base
    high[0] = num_pages - 1
    k = torch.zeros((num_pages, _lib.FP8_ROW_BYTES), dtype=torch.uint8, device="cuda")
    v = torch.zeros_like(k)
    k[high.cuda()] = small.k_cache[small.kv_indices.long()].cuda()
    v[high.cuda()] = small.v_cache[small.kv_indices.long()].cuda()
    out, lse = _lib.run_fp8(small.q.cuda(), k, v, small.kv_indptr.cuda(), high.to(torch.int32).cuda(), small.sm_scale)
    torch.cuda.synchronize()
    check(small, out.float().cpu().double().numpy(), lse.cpu().double().numpy())
    del k, v


def test_bf16_call_under_fp8_tuning():
    """An FP8 tuning leaves bf16-cache calls on the default bf16 kernel."""
    import oracle
    assert _lib.gqa_paged_decode_set_tuning(0, 0, 4, 32, 2, _lib.GATHER_LSU_F8) == 0
    w = wl.make_workload([300, 0, 17, 2000], seed=304)
    g = w.to("cuda")
    out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    o = out.float().cpu().double().numpy()
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    l = lse.cpu().double().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isneginf(l), np.isneginf(l_ref))
    assert np.all(np.abs(l[fin] - l_ref[fin]) <= LSE_ATOL)


def test_fp8_batch_past_merge_grid(f8_stage):
    """5000 sequences of 0-8 tokens over outputs that start as garbage: every empty sequence is written
    (O = 0, LSE = -inf) and the rest match the oracle."""
    lens = torch.randint(0, 9, (5000,), generator=torch.Generator().manual_seed(81)).tolist()
    w = wl.make_fp8_workload(lens, seed=82, pool_factor=1.25)
    g = w.to("cuda")
    out = torch.full_like(g.q, 7.0)
    lse = torch.full((w.batch, 32), 7.0, dtype=torch.float32, device="cuda")
    _lib.run_fp8(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    empty = [b for b, n in enumerate(lens) if n == 0]
    assert empty and np.all(o[empty] == 0.0) and np.all(np.isneginf(l[empty]))
    check(w, o, l)
