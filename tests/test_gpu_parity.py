"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Tolerance (stated for this path): |dO| <= 2e-2 + 2e-2 * |O_ref| elementwise and
|dlse| <= 1e-3 absolute, with -inf == -inf for empty sequences.
"""
import json
import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import gqa_paged_decode_oracle
from oracle.pool import gqa_paged_decode_oracle_parallel
from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl
from paged_kv_gqa_split_gb300.build import build

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    _lib.load()
    yield
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)


@pytest.fixture
def tuning():
    """Apply a tuning for one test and restore the defaults afterwards."""
    def apply(*args):
        assert _lib.gqa_paged_decode_set_tuning(*args) == 0
    yield apply
    assert _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0) == 0


@pytest.fixture(params=[_lib.MERGE_KERNEL, _lib.MERGE_ONE_WAVE], ids=["merge_kernel", "one_wave"])
def merge_mode(request):
    """Run a test with the static grid followed by the merge kernel (the default)
    and with the one-wave decode (merge inside the kernel)."""
    assert _lib.gqa_paged_decode_set_merge_mode(request.param) == 0
    yield request.param
    assert _lib.gqa_paged_decode_set_merge_mode(_lib.MERGE_KERNEL) == 0


def gpu_run(w, dev="cuda"):
    g = w.to(dev)
    out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale)
    torch.cuda.synchronize()
    assert _lib.gqa_paged_decode_last_launch_count() in (1, 2)
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy()


def check(w, out, lse, seqs=None, ref=None):
    if ref is None:
        ref = gqa_paged_decode_oracle(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale, seqs=seqs)
    o_ref, l_ref = ref
    rows = list(range(w.batch)) if seqs is None else list(seqs)
    o, l, orf, lrf = out[rows], lse[rows], o_ref[rows], l_ref[rows]
    err = np.abs(o - orf)
    bad = err > O_ATOL + O_RTOL * np.abs(orf)
    assert not bad.any(), f"O mismatch at {np.argwhere(bad)[:5].tolist()}: max err {err.max():.3e}"
    assert np.array_equal(np.isneginf(l), np.isneginf(lrf)), "empty-sequence LSE mismatch"
    fin = np.isfinite(lrf)
    assert np.all(np.isfinite(l[fin]))
    lerr = np.abs(l[fin] - lrf[fin]) if fin.any() else np.zeros(1)
    assert lerr.max() <= LSE_ATOL, f"LSE max err {lerr.max():.3e}"
    for b in rows:
        if w.lens and w.lens[b] == 0:
            assert np.all(out[b] == 0.0)
    return float(err.max()), float(lerr.max())


# ------------------------------------------------------------ small fixed cases
def test_pattern_workload_matches_golden():
    w = wl.make_pattern_workload()
    out, lse = gpu_run(w)
    path = os.path.join(os.path.dirname(__file__), "golden", "pattern_oracle.json")
    doc = json.load(open(path))
    want_l = np.array(doc["lse"], dtype=np.float64)
    assert np.array_equal(np.isneginf(lse), np.isneginf(want_l))
    fin = np.isfinite(want_l)
    assert np.abs(lse[fin] - want_l[fin]).max() <= LSE_ATOL
    for key, row in doc["o_rows"].items():
        b, h = (int(x) for x in key.split(","))
        row = np.array(row)
        assert np.all(np.abs(out[b, h] - row) <= O_ATOL + O_RTOL * np.abs(row))
    assert np.all(out[1] == 0.0)


EDGE_LENS = {
    "single_token": [1],
    "one_empty": [0],
    "all_empty": [0, 0, 0],
    "ones": [1] * 7,
    "around_16": [15, 16, 17],
    "around_32": [31, 32, 33],
    "ramp_1_40": list(range(1, 41)),
    "leading_trailing_empty": [0, 0, 5, 0, 300, 0, 0],
    "around_256": [255, 256, 257, 0, 129],
    "ragged_mix": [3, 1000, 0, 77, 2049, 1, 16, 600],
}


@pytest.mark.parametrize("name", sorted(EDGE_LENS))
def test_edge_cases_default(name, merge_mode):
    w = wl.make_workload(EDGE_LENS[name], seed=100 + len(name), pool_factor=1.5)
    out, lse = gpu_run(w)
    check(w, out, lse)


@pytest.mark.parametrize("case", ["5000_short", "3000_empty"])
def test_batch_past_merge_grid(case, merge_mode):
    """More sequences than merge CTAs (and than one-wave warps x 32): every empty sequence is still
    written (O = 0, LSE = -inf) over outputs that start as garbage, and a CTA range walks hundreds of
    sequences."""
    if case == "5000_short":
        lens = torch.randint(0, 9, (5000,), generator=torch.Generator().manual_seed(5)).tolist()
    else:
        lens = [0] * 3000
    w = wl.make_workload(lens, seed=6, pool_factor=1.25)
    g = w.to("cuda")
    out = torch.full_like(g.q, 7.0)
    lse = torch.full((w.batch, 32), 7.0, dtype=torch.float32, device="cuda")
    _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    empty = [b for b, n in enumerate(lens) if n == 0]
    assert len(empty) > 1367 or case == "5000_short"
    assert np.all(o[empty] == 0.0) and np.all(np.isneginf(l[empty]))
    if sum(lens):
        check(w, o, l)


# (num_ctas, min_units_per_cta, heads_per_cta, tile, stages, gather[, fused_merge_max_splits, tier2_ctas,
#  tier2_permille, tier2_min_units]): gather 0 = cp.async, 1 = TMA bulk; tier2_ctas -1 = one tier
VARIANTS = {
    "lsu_ng4_s3": (0, 0, 4, 16, 3, 0),
    "lsu_ng4_s4": (0, 0, 4, 16, 4, 0),
    "lsu_ng4_s2": (0, 0, 4, 16, 2, 0),
    "lsu_ng2_s3": (0, 0, 2, 16, 3, 0),
    "lsu_ng2_s5": (0, 0, 2, 16, 5, 0),
    "lsu_ng2_s2": (0, 0, 2, 16, 2, 0),
    "lsu_ng1_s2": (0, 0, 1, 16, 2, 0),
    "lsu_ng1_s4": (0, 0, 1, 16, 4, 0),
    "lsu_ng1_s3": (0, 0, 1, 16, 3, 0),
    "lsu_ng1_s6": (0, 0, 1, 16, 6, 0),
    "lsu_few_ctas": (7, 0, 4, 16, 3, 0),
    "lsu_small_units": (0, 16, 4, 16, 3, 0),
    "lsu_ng1_small_units": (0, 16, 1, 16, 3, 0),
    "lsu_one_cta": (1, 0, 4, 16, 3, 0),
    "tma_ng4_t16": (0, 0, 4, 16, 5, 1),
    "tma_ng4_t32": (0, 0, 4, 32, 3, 1),
    "tma_ng1_t16": (0, 0, 1, 16, 4, 1),
    "tma_small_units": (0, 16, 4, 32, 3, 1),
    # tier 2 takes units only once the tier-1 CTAs are full, hence few tier-1 CTAs here
    "lsu_one_tier": (0, 0, 4, 16, 2, 0, 0, -1),
    "lsu_tier2_half_fine": (40, 8, 4, 16, 2, 0, 0, 0, 500, 16),
    "lsu_ng1_tier2": (40, 8, 1, 16, 2, 0, 0, 0, 300, 8),
    "lsu_few_ctas_tier2": (7, 0, 4, 16, 2, 0, 0, 13, 400, 4),
    "lsu_tier2_unfused": (40, 8, 4, 16, 2, 0, -1, 0, 600, 8),
    "tma_tier2": (40, 8, 4, 16, 5, 1, 0, 0, 300, 16),
    # the contractions on the CUDA cores (comparison variant)
    "cuda_cores": (0, 0, 4, 16, 2, 3),
    "cuda_cores_split": (40, 8, 4, 16, 2, 3, 0, 0, 300, 16),
}


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("case", ["ragged_mix", "leading_trailing_empty", "ramp_1_40"])
def test_kernel_variants(tuning, variant, case, merge_mode):
    tuning(*VARIANTS[variant])
    w = wl.make_workload(EDGE_LENS[case], seed=7, pool_factor=1.25)
    out, lse = gpu_run(w)
    check(w, out, lse)


@pytest.mark.parametrize("ng,stages", [(4, 3), (4, 2), (1, 2)])
@pytest.mark.parametrize("fuse", [0, -1, 64, 2, 5])
@pytest.mark.parametrize("num_ctas,min_units", [(152, 16), (40, 16), (300, 1), (3, 1), (90, 1), (1200, 1)])
def test_split_and_merge_paths(tuning, num_ctas, min_units, fuse, ng, stages, merge_mode):
    """One long and several short sequences cut into 2 to ~300 pieces, with the merge
    done in the decode kernel (up to `fuse` pieces; 0 = default 16, -1 = never; the
    warp stages 4 partials per round trip, so 5 and 16 take several batches) or by
    the merge kernel (warp path up to 16 pieces; above that the block path, whose
    block width runs from 32 dims at 17 pieces down to 1 dim past 256 pieces)."""
    tuning(num_ctas, min_units, ng, 16, stages, 0, fuse)
    w = wl.make_workload([5000, 3, 17, 0, 900, 1, 64], seed=21, pool_factor=1.1)
    out, lse = gpu_run(w)
    check(w, out, lse)


@pytest.mark.parametrize("variant", [(200, 8, 4, 16, 3, 0), (600, 8, 1, 16, 3, 0), (120, 8, 2, 16, 5, 0),
                                     (90, 8, 4, 32, 3, 1), (300, 8, 4, 16, 5, 1), (200, 8, 4, 16, 3, 0, -1),
                                     (600, 8, 1, 16, 3, 0, 64), (300, 8, 4, 16, 5, 1, -1),
                                     (100, 8, 4, 16, 2, 0, 0, 700, 500, 4), (100, 8, 4, 16, 2, 0, -1, 700, 500, 4)])
def test_token_count_exact_with_uniform_scores(tuning, variant, merge_mode):
    """q = 0 makes every score 0: lse must be log2(n) to fp32 precision, which a
    dropped or doubled token would break (1.44/n >> 2e-5 for n <= 9000), and O
    must be the mean of the sequence's V rows."""
    tuning(*variant)
    lens = [9000, 1, 2, 3, 4000, 0, 17, 1023, 1024, 1025, 5]
    w = wl.make_workload(lens, seed=33, pool_factor=1.0)
    w.q.zero_()
    out, lse = gpu_run(w)
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(np.isneginf(lse[b]))
        else:
            assert np.abs(lse[b] - math.log2(n)).max() < 2e-5, (b, n, lse[b][:4])
    check(w, out, lse)


@pytest.mark.parametrize("ng", [4, 2, 1])
@pytest.mark.parametrize("pieces", [17, 32, 33, 34, 64, 65, 97, 150, 300])
def test_block_merge_piece_counts(tuning, ng, pieces):
    """Sequences cut into more than 16 pieces go to the merge kernel's block path, whose block width
    halves as the piece count doubles (32 dims at 17 pieces, 16 past 32, ..., 1 past 256) and whose
    rows walk the pieces in batches. One tier of pieces x (4 / ng) CTAs cuts the long sequence into
    about `pieces` pieces per head group (around those edges, checked on the host plan), for every
    head-group shape; then the same with q = 0, where lse must be log2(n) exactly (a piece dropped or
    folded twice shows) and O the mean of the V rows."""
    lens = [4160, 3, 0, 1]
    ctas = pieces * (4 // ng)
    plan = _lib.gqa_paged_decode_plan([0] + list(itertools.accumulate(lens)), ctas, 1, ng, 0, 0, 0)
    cut = max(sum(1 for x in plan if x[1] == 0 and x[2] == hg) for hg in range(4 // ng))
    assert abs(cut - pieces) <= 1 + pieces // 16, cut
    tuning(ctas, 1, ng, 16, 2, 0, 0, -1)
    w = wl.make_workload(lens, seed=90 + pieces, pool_factor=1.1)
    out, lse = gpu_run(w)
    check(w, out, lse)
    w.q.zero_()
    out, lse = gpu_run(w)
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(np.isneginf(lse[b]))
        else:
            assert np.abs(lse[b] - math.log2(n)).max() < 2e-5, (b, n, lse[b][:4])
    check(w, out, lse)


def test_peaky_softmax_large_scores(merge_mode):
    w = wl.make_workload([700, 64, 3], seed=44, q_std=30.0)
    out, lse = gpu_run(w)
    check(w, out, lse)


def test_deterministic_bitwise(merge_mode):
    w = wl.make_workload([1000, 0, 333, 4096], seed=45)
    g = w.to("cuda")
    o1, l1 = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices)
    o2, l2 = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_int64_page_addressing(merge_mode):
    """Pages above 2^21 sit more than 2^31 bytes into each 1 KB-per-page pool."""
    num_pages = (1 << 21) + 4096
    small = wl.make_workload([40, 0, 300], seed=46, pool_factor=1.0)
    g = torch.Generator().manual_seed(5)
    high = torch.randperm(num_pages - (1 << 21), generator=g)[: small.total_tokens] + (1 << 21)
    high[0] = num_pages - 1
    k = torch.zeros((num_pages, 1, 4, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    k[high.cuda()] = small.k_cache[small.kv_indices.long()].cuda()
    v[high.cuda()] = small.v_cache[small.kv_indices.long()].cuda()
    q = small.q.cuda()
    out, lse = _lib.run(q, k, v, small.kv_indptr.cuda(), high.to(torch.int32).cuda(), small.sm_scale)
    torch.cuda.synchronize()
    check(small, out.float().cpu().double().numpy(), lse.cpu().double().numpy())
    del k, v


# ----------------------------------------------------------- entry variants
def test_workspace_variant_matches_and_rejects_small(merge_mode):
    w = wl.make_workload([2000, 5, 0, 700], seed=47)
    g = w.to("cuda")
    need = _lib.gqa_paged_decode_ws_size(w.batch, w.total_tokens)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o1, l1 = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices)
    o2, l2 = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    small = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.GqaError) as e:
        _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, workspace=small)
    assert e.value.code == _lib.GQA_ERR_WORKSPACE


def test_checked_valid_matches_unchecked(merge_mode):
    w = wl.make_workload([129, 0, 64, 1000], seed=48, pool_factor=1.3)
    g = w.to("cuda")
    o1, l1 = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices)
    o2, l2, err = _lib.run_checked(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_checked_rejects_bad_page_before_reading(merge_mode):
    w = wl.make_workload([50, 20], seed=49)
    g = w.to("cuda")
    bad_idx = g.kv_indices.clone()
    bad_idx[7] = w.num_pages  # one past the pool
    out = torch.full_like(g.q, 7.0)
    lse = torch.full((w.batch, 32), 7.0, device="cuda")
    _, _, err = _lib.run_checked(g.q, g.k_cache, g.v_cache, g.kv_indptr, bad_idx, out=out, lse=lse)
    torch.cuda.synchronize()
    assert int(err.item()) & 4
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)  # nothing was written


def test_checked_rejects_decreasing_indptr():
    w = wl.make_workload([10, 10, 10], seed=50)
    g = w.to("cuda")
    bad = g.kv_indptr.clone()
    bad[1] = 25
    bad[2] = 12  # decreasing; the last entry still equals len(kv_indices)
    _, _, err = _lib.run_checked(g.q, g.k_cache, g.v_cache, bad, g.kv_indices)
    torch.cuda.synchronize()
    assert int(err.item()) & 8


def test_non_default_stream():
    w = wl.make_workload([300, 7], seed=51)
    g = w.to("cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse = _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices)
    s.synchronize()
    check(w, out.float().cpu().double().numpy(), lse.cpu().double().numpy())


# ------------------------------------------------------ the five workloads
@pytest.mark.parametrize("name", ["tiny", "mid", "long", "large", "skewed"])
def test_workload_parity(name, merge_mode):
    """Every sequence of every workload, element by element, against the float64
    oracle (evaluated across the host's cores; the rows are the single-process
    oracle's, bit for bit)."""
    w = wl.make_config(name)
    out, lse = gpu_run(w)
    ref = gqa_paged_decode_oracle_parallel(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    o_err, l_err = check(w, out, lse, ref=ref)
    print(f"{name}: max |dO| {o_err:.3e}, max |dlse| {l_err:.3e}, all {w.batch} sequences checked")
    assert np.all(np.isfinite(out))
    assert np.all(np.isfinite(lse) | np.isneginf(lse))


@pytest.fixture
def one_wave():
    assert _lib.gqa_paged_decode_set_merge_mode(_lib.MERGE_ONE_WAVE) == 0
    yield
    assert _lib.gqa_paged_decode_set_merge_mode(_lib.MERGE_KERNEL) == 0


@pytest.mark.parametrize("name", ["mid", "skewed"])
def test_cuda_core_variant_full_workload(tuning, name):
    """The CUDA-core comparison variant on full workloads, every sequence."""
    tuning(0, 0, 4, 16, 2, 3)
    w = wl.make_config(name)
    out, lse = gpu_run(w)
    ref = gqa_paged_decode_oracle_parallel(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale)
    check(w, out, lse, ref=ref)


@pytest.mark.parametrize("tier2", [(0, 0, 0), (-1, 0, 0), (4000, 900, 1), (912, 500, 8), (6840, 100, 0),
                                   (8000, 500, 1)])
def test_one_wave_tier2_shapes(tuning, tier2, one_wave):
    """One-wave mode with the default tiers, one tier, 90% of the line in 4000
    small tier-2 ranges (about 9 per warp), half the line in tier 2, and 15
    tier-2 ranges per tier-1 CTA (the most a warp takes on a 152-SM part); 8000
    tier-2 CTAs are more than the warps may take, so that call falls back to the
    merge kernel. A long sequence, short ones and empties, against the oracle."""
    t2, permille, min_units = tier2
    tuning(0, 0, 4, 16, 2, 0, 0, t2, permille, min_units)
    w = wl.make_workload([70000, 0, 3, 1, 5000, 0, 129, 16, 17, 2049], seed=52, pool_factor=1.3)
    out, lse = gpu_run(w)
    assert _lib.gqa_paged_decode_last_launch_count() == (2 if t2 == 8000 else 1)
    check(w, out, lse)


def test_no_device_error_flagged():
    assert _lib.gqa_paged_decode_device_error() == 0
