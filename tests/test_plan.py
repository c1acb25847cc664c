"""Split plan on the host (no GPU): the arithmetic shared by the decode and merge
kernels (units per CTA in each of the two tiers, where sequences are cut, which
partial slot each piece uses, and how the merge finds them) must tile every batch
exactly once and agree between the decode side and the merge side."""
import numpy as np
import pytest

from paged_kv_gqa_split_gb300 import _lib
from paged_kv_gqa_split_gb300 import workloads as wl
from paged_kv_gqa_split_gb300.build import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    _lib.load()


def indptr_of(lens):
    ip = np.zeros(len(lens) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lens)
    return ip


def tier_shape(W, p1, p2, min_units, permille, min2):
    """Units per CTA in each tier, restated from the plan's definition: tier 2 sets
    aside floor(W * permille / 1000) units, tier 1 splits the rest evenly (at least
    min_units per CTA), tier 2 splits what tier 1 leaves (at least min2 per CTA)."""
    w2t = W * permille // 1000 if p2 > 0 else 0
    q1 = max(min_units, -(-(W - w2t) // p1), 1)
    w1 = min(W, q1 * p1)
    q2 = max(min2, -(-(W - w1) // p2) if p2 > 0 else 1, 1)
    return q1, w1, q2


def check_plan(lens, num_ctas, min_units, ng, tier2=0, permille=0, min2=0):
    ip = indptr_of(lens)
    T = int(ip[-1])
    hg_count = 4 // ng
    pieces = _lib.gqa_paged_decode_plan(ip, num_ctas, min_units, ng, tier2, permille, min2)
    W = T * hg_count
    mu = min_units if min_units > 0 else 32
    q1, w1, q2 = tier_shape(W, num_ctas, tier2, mu, permille if permille > 0 else 100, min2 if min2 > 0 else 64)
    # 1) every (head group, sequence) is covered exactly once by contiguous pieces
    cover = {}
    for (cta, b, hg, lo, hi, slot, f, l, fs) in pieces:
        assert 0 <= b < len(lens) and 0 <= hg < hg_count and lo < hi
        assert ip[b] <= lo and hi <= ip[b + 1]
        cover.setdefault((hg, b), []).append((lo, hi, cta, slot, f, l, fs))
    for hg in range(hg_count):
        for b, n in enumerate(lens):
            segs = sorted(cover.get((hg, b), []))
            if n == 0:
                assert not segs
                continue
            assert segs[0][0] == ip[b] and segs[-1][1] == ip[b + 1]
            for a, c in zip(segs, segs[1:]):
                assert a[1] == c[0]
            # 2) decode view and merge view agree
            first, last, first_slot = segs[0][4], segs[0][5], segs[0][6]
            ctas = [s[2] for s in segs]
            assert ctas == list(range(first, last + 1))
            if first == last:
                assert len(segs) == 1 and segs[0][3] == -1
            else:
                assert segs[0][3] == first_slot
                assert all(s[3] == 0 for s in segs[1:])
                assert all(s[3] in (0, 1) for s in segs)
    # 3) partial slots are unique per CTA
    used = [(p[0], p[5]) for p in pieces if p[5] >= 0]
    assert len(used) == len(set(used))
    # 4) balance: within each tier every CTA holds that tier's share, except the
    #    last active CTA of the tier; tier 1 covers units [0, w1), tier 2 the rest
    per_cta = {}
    for (cta, b, hg, lo, hi, slot, *_rest) in pieces:
        per_cta[cta] = per_cta.get(cta, 0) + hi - lo
    assert sum(per_cta.values()) == W
    assert all(0 <= c < num_ctas + tier2 for c in per_cta)
    t1 = sorted(c for c in per_cta if c < num_ctas)
    t2 = sorted(c for c in per_cta if c >= num_ctas)
    assert t1 == list(range(len(t1)))
    assert t2 == list(range(num_ctas, num_ctas + len(t2)))
    assert sum(per_cta[c] for c in t1) == w1
    for tier, q in ((t1, q1), (t2, q2)):
        for c in tier[:-1]:
            assert per_cta[c] == q
        if tier:
            assert 0 < per_cta[tier[-1]] <= q
    assert not t2 or len(t1) == num_ctas  # tier 2 starts only once tier 1 is full
    return pieces


@pytest.mark.parametrize("ng", [4, 2, 1])
@pytest.mark.parametrize("num_ctas,min_units", [(1, 0), (3, 1), (7, 16), (152, 0), (304, 128), (1000, 1)])
def test_random_ragged_batches(ng, num_ctas, min_units):
    rng = np.random.default_rng(num_ctas * 31 + ng)
    for _ in range(5):
        lens = rng.integers(0, 3000, size=int(rng.integers(1, 60))).tolist()
        lens[int(rng.integers(0, len(lens)))] = 0
        check_plan(lens, num_ctas, min_units, ng)


@pytest.mark.parametrize("ng", [4, 2, 1])
@pytest.mark.parametrize("num_ctas,tier2,permille,min2", [(152, 608, 0, 0), (456, 1824, 100, 64), (7, 3, 900, 1),
                                                          (304, 50, 300, 16), (1, 4, 500, 8), (300, 1, 1, 1)])
def test_two_tier_ragged_batches(ng, num_ctas, tier2, permille, min2):
    rng = np.random.default_rng(num_ctas * 7 + tier2 + ng)
    for _ in range(5):
        lens = rng.integers(0, 5000, size=int(rng.integers(1, 80))).tolist()
        lens[int(rng.integers(0, len(lens)))] = 0
        check_plan(lens, num_ctas, 1, ng, tier2, permille, min2)


@pytest.mark.parametrize("lens", [[0], [0, 0, 0], [1], [5, 0, 0, 7], [0, 0, 131072], [16] * 40])
def test_edge_batches(lens):
    for num_ctas in (1, 2, 304):
        for ng in (1, 4):
            check_plan(lens, num_ctas, 1, ng)
            check_plan(lens, num_ctas, 1, ng, 4 * num_ctas, 100, 64)
            check_plan(lens, num_ctas, 1, ng, 3, 900, 1)


@pytest.mark.parametrize("name", ["tiny", "mid", "long", "large", "skewed"])
def test_workload_plans(name):
    lens = wl.config_lens(name)
    check_plan(lens, 456, 0, 4, 1824)  # the default shape on 152 SMs
    pieces = check_plan(lens, 304, 0, 4)
    splits = {}
    for p in pieces:
        splits[p[1]] = splits.get(p[1], 0) + 1
    # a long sequence is cut once per CTA boundary it spans
    longest = int(np.argmax(lens))
    q = max(32, -(-sum(lens) // 304))
    assert splits[longest] >= lens[longest] // q


def test_empty_batch_and_bad_tables():
    assert _lib.gqa_paged_decode_plan(np.zeros(1, dtype=np.int32), 4) == []
    with pytest.raises(_lib.GqaError):
        _lib.gqa_paged_decode_plan(np.array([0, 5, 3, 8], dtype=np.int32), 4, 1, 4)
    with pytest.raises(_lib.GqaError):
        _lib.gqa_paged_decode_plan(indptr_of([3, 4]), 4, 1, 3)
    with pytest.raises(_lib.GqaError):
        _lib.gqa_paged_decode_plan(indptr_of([3, 4]), 4, 1, 4, -1)
    with pytest.raises(_lib.GqaError):
        _lib.gqa_paged_decode_plan(indptr_of([3, 4]), 4, 1, 4, 8, 901)
