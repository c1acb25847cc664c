"""Seeded synthetic inputs for paged GQA decode (h32 / kv4 / d128 / page size 1, bf16).

This module only draws inputs. It holds none of the attention arithmetic, so the
float64 oracle and the CUDA path can both consume what it produces without
sharing any of the method.

Problem shape, as fixed by the FlashInfer-style problem statement on the
kernelindex.com page "gqa_paged_decode_h32_kv4_d128_ps1" (its ``run()`` docstring):

* ``q``          [batch, 32, 128] bf16
* ``k_cache``    [num_pages, 1, 4, 128] bf16
* ``v_cache``    [num_pages, 1, 4, 128] bf16
* ``kv_indptr``  [batch + 1] int32, CSR offsets into ``kv_indices``
* ``kv_indices`` [kv_indptr[-1]] int32, page ids in token order
* ``sm_scale``   1/sqrt(128)

Draw order for every workload (one ``torch.Generator`` seeded with the
workload's seed): sequence lengths (and, for the skewed mix, the positions of
the long sequences), the page permutation, then q, k, v. q, k and v are drawn
as float32 standard normals and rounded to bf16 (round-to-nearest-even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import torch

NUM_QO_HEADS = 32
NUM_KV_HEADS = 4
HEAD_DIM = 128
PAGE_SIZE = 1
DEFAULT_SM_SCALE = 1.0 / math.sqrt(HEAD_DIM)

# Elements drawn per randn call when filling the page pools; fixed so that the
# stream of draws (and therefore every value) depends on the seed alone.
_CHUNK = 1 << 22


@dataclass
class Workload:
    """One batch of decode inputs, all on the CPU."""

    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    sm_scale: float
    lens: List[int] = field(default_factory=list)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.kv_indices.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    def to(self, device, non_blocking: bool = False) -> "Workload":
        return Workload(
            self.name,
            self.q.to(device, non_blocking=non_blocking),
            self.k_cache.to(device, non_blocking=non_blocking),
            self.v_cache.to(device, non_blocking=non_blocking),
            self.kv_indptr.to(device, non_blocking=non_blocking),
            self.kv_indices.to(device, non_blocking=non_blocking),
            self.sm_scale,
            list(self.lens),
        )


def _randn_bf16(shape: Sequence[int], g: torch.Generator, std: float = 1.0) -> torch.Tensor:
    """float32 N(0, std^2) draws rounded to bf16, produced in fixed-size chunks."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        x = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[lo:hi] = x.to(torch.bfloat16)
    return out.view(*shape)


def make_workload(
    lens: Sequence[int],
    seed: int,
    *,
    pool_factor: float = 1.0,
    q_std: float = 1.0,
    name: str = "custom",
    sm_scale: float = DEFAULT_SM_SCALE,
    g: Optional[torch.Generator] = None,
) -> Workload:
    """Build a workload from explicit sequence lengths.

    ``num_pages = ceil(pool_factor * sum(lens))`` (at least 1, so the pools are
    never zero-sized); ``kv_indices`` is the first ``sum(lens)`` entries of a
    seeded random permutation of the pool, i.e. pages sampled without
    replacement and scattered at random through the pool.
    """
    if g is None:
        g = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in lens]
    if any(x < 0 for x in lens):
        raise ValueError("sequence lengths must be non-negative")
    batch = len(lens)
    total = sum(lens)
    num_pages = max(1, int(math.ceil(pool_factor * total)))
    indptr = torch.zeros(batch + 1, dtype=torch.int64)
    if batch:
        indptr[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)
    perm = torch.randperm(num_pages, generator=g)
    kv_indices = perm[:total].to(torch.int32).contiguous()
    q = _randn_bf16((batch, NUM_QO_HEADS, HEAD_DIM), g, q_std)
    k = _randn_bf16((num_pages, PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM), g)
    v = _randn_bf16((num_pages, PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM), g)
    return Workload(name, q, k, v, indptr.to(torch.int32), kv_indices, float(sm_scale), lens)


def _tiny(g: torch.Generator) -> List[int]:
    lens = torch.randint(1, 257, (5,), generator=g).tolist()
    lens[2] = 0  # the third sequence (0-based index 2) is forced empty
    return lens


def _mid(g: torch.Generator) -> List[int]:
    return torch.randint(512, 4097, (64,), generator=g).tolist()


def _long(g: torch.Generator) -> List[int]:
    return [131072]


def _large(g: torch.Generator) -> List[int]:
    return torch.randint(1024, 8193, (256,), generator=g).tolist()


def _skewed(g: torch.Generator) -> List[int]:
    batch = 128
    n_long = int(round(0.1 * batch))  # 13 long sequences, 115 short ones
    where = torch.randperm(batch, generator=g)[:n_long]
    lens = torch.randint(64, 513, (batch,), generator=g)
    lens[where] = torch.randint(32768, 65537, (n_long,), generator=g)
    return lens.tolist()


@dataclass(frozen=True)
class Config:
    name: str
    seed: int
    lens_fn: object
    pool_factor: float
    q_std: float
    description: str


CONFIGS: Dict[str, Config] = {
    "tiny": Config("tiny", 0, _tiny, 1.0, 1.0,
                   "batch 5, lens U{1..256}, sequence 2 empty, pool = sum(lens), kv_indices = randperm"),
    "mid": Config("mid", 1, _mid, 1.0, 1.0,
                  "batch 64, lens U{512..4096}, pool = sum(lens), kv_indices = randperm"),
    "long": Config("long", 2, _long, 1.0, 1.0,
                   "batch 1, one sequence of 131072 tokens, kv_indices = randperm(131072)"),
    "large": Config("large", 3, _large, 1.25, 1.0,
                    "batch 256, lens U{1024..8192}, pool = ceil(1.25 sum(lens)), indices sampled without replacement"),
    "skewed": Config("skewed", 4, _skewed, 2.0, 3.0,
                     "batch 128, 115 lens U{64..512} + 13 lens U{32768..65536}, pool = 2 sum(lens), q ~ 3 N(0,1)"),
}


def config_lens(name: str) -> List[int]:
    """Sequence lengths of a named workload, without drawing the tensors."""
    cfg = CONFIGS[name]
    g = torch.Generator().manual_seed(cfg.seed)
    return list(cfg.lens_fn(g))


def make_config(name: str) -> Workload:
    """Draw the named workload (tiny, mid, long, large, skewed) on the CPU."""
    cfg = CONFIGS[name]
    g = torch.Generator().manual_seed(cfg.seed)
    lens = cfg.lens_fn(g)
    return make_workload(lens, cfg.seed, pool_factor=cfg.pool_factor, q_std=cfg.q_std,
                         name=cfg.name, g=g)


def make_pattern_workload() -> Workload:
    """A small fixed workload with formula-defined values (no random draws).

    Three sequences of lengths 3, 0 and 5 over a pool of 10 pages; page ids are
    ``(7 * j + 3) % 10`` for token j of the batch. Every q/k/v entry is a
    multiple of 1/8 in [-1, 1], exactly representable in bf16, given by
    ``((a * i + e) % 17 - 8) / 8`` over the flattened index i of the tensor
    (a, e fixed per tensor). Identical on every machine.
    """
    lens = [3, 0, 5]
    total = sum(lens)
    indptr = torch.tensor([0, 3, 3, 8], dtype=torch.int32)
    indices = torch.tensor([(7 * j + 3) % 10 for j in range(total)], dtype=torch.int32)

    def pattern(shape, a, e):
        n = 1
        for s in shape:
            n *= s
        i = torch.arange(n, dtype=torch.int64)
        vals = ((a * i + e) % 17 - 8).to(torch.float32) / 8.0
        return vals.to(torch.bfloat16).view(*shape)

    q = pattern((3, NUM_QO_HEADS, HEAD_DIM), 5, 1)
    k = pattern((10, PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM), 3, 2)
    v = pattern((10, PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM), 11, 4)
    return Workload("pattern", q, k, v, indptr, indices, DEFAULT_SM_SCALE, lens)


# ------------------------------------------------------------------ sparse
@dataclass
class SparseWorkload:
    """Inputs of a selected-token (sparse) paged decode, all on the CPU.

    Shapes follow the sparse split-K GQA path of the sigit.si vLLM "qsa.py" page
    (``qsa_sparse_paged_attention``): q [rows, 32, 128] bf16; k_cache, v_cache
    [num_blocks, page_size, 4, 128] bf16; logical_indices [rows, topk] int32
    (logical token positions of the row's request, -1 = no selection);
    block_table [num_requests, width] int32 (-1 = no page); token_to_req [rows]
    int32.
    """

    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    logical_indices: torch.Tensor
    block_table: torch.Tensor
    token_to_req: torch.Tensor
    sm_scale: float
    lens: List[int] = field(default_factory=list)

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def topk(self) -> int:
        return int(self.logical_indices.shape[1])

    @property
    def page_size(self) -> int:
        return int(self.k_cache.shape[1])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    def to(self, device, non_blocking: bool = False) -> "SparseWorkload":
        t = lambda x: x.to(device, non_blocking=non_blocking)  # noqa: E731
        return SparseWorkload(self.name, t(self.q), t(self.k_cache), t(self.v_cache), t(self.logical_indices),
                              t(self.block_table), t(self.token_to_req), self.sm_scale, list(self.lens))


def make_sparse_workload(
    lens: Sequence[int],
    topk: int,
    page_size: int,
    seed: int,
    *,
    pool_factor: float = 1.25,
    q_std: float = 1.0,
    name: str = "sparse",
    sm_scale: float = DEFAULT_SM_SCALE,
) -> SparseWorkload:
    """One query row per request, request r holding lens[r] cached tokens.

    Draw order (one ``torch.Generator`` seeded with ``seed``): the physical
    block permutation, then each row's selection, then q, k, v. Request r
    owns ceil(lens[r] / page_size) blocks, taken in order from a seeded
    random permutation of ``ceil(pool_factor * total blocks)`` blocks; the
    rest of its block-table row is -1. Row r selects min(topk, lens[r])
    distinct positions below lens[r] (a seeded random subset, in increasing
    order, as a top-k selection would give) and pads with -1.
    """
    g = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in lens]
    rows = len(lens)
    if rows == 0 or topk <= 0 or page_size <= 0:
        raise ValueError("need rows, a positive topk and a positive page size")
    nblk = [(n + page_size - 1) // page_size for n in lens]
    width = max(1, max(nblk))
    total_blocks = sum(nblk)
    num_blocks = max(1, int(math.ceil(pool_factor * total_blocks)))
    perm = torch.randperm(num_blocks, generator=g)
    table = torch.full((rows, width), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(nblk):
        table[r, :n] = perm[off:off + n].to(torch.int32)
        off += n
    idx = torch.full((rows, topk), -1, dtype=torch.int32)
    for r, n in enumerate(lens):
        k = min(topk, n)
        if k > 0:
            sel = torch.randperm(n, generator=g)[:k].sort().values
            idx[r, :k] = sel.to(torch.int32)
    q = _randn_bf16((rows, NUM_QO_HEADS, HEAD_DIM), g, q_std)
    kc = _randn_bf16((num_blocks, page_size, NUM_KV_HEADS, HEAD_DIM), g)
    vc = _randn_bf16((num_blocks, page_size, NUM_KV_HEADS, HEAD_DIM), g)
    return SparseWorkload(name, q, kc, vc, idx, table.contiguous(), torch.arange(rows, dtype=torch.int32),
                          float(sm_scale), lens)


# Selected-token decode workload timed by bench.py: the pages fix no sizes for
# this path, so it takes decode-sized rows of the same head shape: 128
# requests with 2k-8k cached tokens in blocks of 64, 2048 selected positions
# per row (512 MB of K/V rows read per call).
SPARSE_CONFIG = dict(rows=128, topk=2048, page_size=64, len_lo=2048, len_hi=8192, seed=5, pool_factor=1.25)


def make_sparse_config() -> SparseWorkload:
    c = SPARSE_CONFIG
    g = torch.Generator().manual_seed(c["seed"])
    lens = torch.randint(c["len_lo"], c["len_hi"] + 1, (c["rows"],), generator=g).tolist()
    return make_sparse_workload(lens, c["topk"], c["page_size"], c["seed"] + 1000, pool_factor=c["pool_factor"],
                                name="sparse")


# --------------------------------------------------------------------- fp8
FP8_ROW_BYTES = NUM_KV_HEADS * HEAD_DIM + 4 * NUM_KV_HEADS  # 512 e4m3 values + 4 fp32 scales per token


def quantize_fp8_rows(x: torch.Tensor) -> torch.Tensor:
    """[P, 1, 4, 128] bf16 -> [P, 528] uint8 FP8 cache rows.

    Each (token, KV head) row of 128 values gets the scale amax / 448 (1 for an
    all-zero row) and is stored as e4m3 codes of x / scale (torch's
    round-to-nearest cast), followed by the 4 heads' float32 scales. This is
    input encoding only: the decode reads the rows as given.
    """
    xf = x.reshape(-1, NUM_KV_HEADS, HEAD_DIM).to(torch.float32)
    amax = xf.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (xf / scale[:, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    rows = torch.empty((xf.shape[0], FP8_ROW_BYTES), dtype=torch.uint8, device=x.device)
    rows[:, :NUM_KV_HEADS * HEAD_DIM] = codes.reshape(-1, NUM_KV_HEADS * HEAD_DIM)
    rows[:, NUM_KV_HEADS * HEAD_DIM:] = scale.contiguous().view(torch.uint8).reshape(-1, 4 * NUM_KV_HEADS)
    return rows


def make_fp8_workload(lens: Sequence[int], seed: int, *, pool_factor: float = 1.0, q_std: float = 1.0,
                      name: str = "custom_fp8") -> Workload:
    """The bf16 workload of the same lengths and seed, with K and V quantized to
    [P, 528]-byte FP8 rows (quantize_fp8_rows). q, kv_indptr and kv_indices are
    unchanged."""
    w = make_workload(lens, seed, pool_factor=pool_factor, q_std=q_std, name=name)
    return Workload(name, w.q, quantize_fp8_rows(w.k_cache), quantize_fp8_rows(w.v_cache), w.kv_indptr,
                    w.kv_indices, w.sm_scale, list(w.lens))


def make_fp8_config(name: str) -> Workload:
    """A named workload (same lengths, seed and pool as the bf16 one) over an FP8 cache."""
    cfg = CONFIGS[name]
    g = torch.Generator().manual_seed(cfg.seed)
    lens = cfg.lens_fn(g)
    return make_fp8_workload(lens, cfg.seed, pool_factor=cfg.pool_factor, q_std=cfg.q_std, name=name + "_fp8")


# --------------------------------------------------------------------- mla
MLA_D_QK = 576
MLA_D_V = 512


@dataclass
class MlaWorkload:
    """Inputs of a dense MLA paged decode (one latent KV head), all on the CPU.

    Shapes follow the flash_mla_with_kvcache page: q [B, s_q, h_q, 576] bf16;
    kv_cache [num_blocks, page_size, 1, 576] bf16 (the first 512 values of a
    row are also its value vector); block_table [B, width] int32;
    cache_seqlens [B] int32.
    """

    name: str
    q: torch.Tensor
    kv_cache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    softmax_scale: float
    lens: List[int] = field(default_factory=list)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def page_size(self) -> int:
        return int(self.kv_cache.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lens))

    def to(self, device, non_blocking: bool = False) -> "MlaWorkload":
        t = lambda x: x.to(device, non_blocking=non_blocking)  # noqa: E731
        return MlaWorkload(self.name, t(self.q), t(self.kv_cache), t(self.block_table), t(self.cache_seqlens),
                           self.softmax_scale, list(self.lens))


def make_mla_workload(lens: Sequence[int], h_q: int, s_q: int, page_size: int, seed: int, *,
                      pool_factor: float = 1.25, q_std: float = 1.0, name: str = "mla") -> MlaWorkload:
    """Sequence b holds lens[b] cached tokens in ceil(lens[b] / page_size)
    blocks, taken in order from a seeded random permutation of
    ceil(pool_factor * blocks in use) blocks (the rest of its block-table row
    is -1). Draw order: the block permutation, then q, then the cache."""
    g = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in lens]
    bsz = len(lens)
    nblk = [(n + page_size - 1) // page_size for n in lens]
    width = max(1, max(nblk) if nblk else 1)
    num_blocks = max(1, int(math.ceil(pool_factor * sum(nblk))))
    perm = torch.randperm(num_blocks, generator=g)
    table = torch.full((bsz, width), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = _randn_bf16((bsz, s_q, h_q, MLA_D_QK), g, q_std)
    kv = _randn_bf16((num_blocks, page_size, 1, MLA_D_QK), g)
    return MlaWorkload(name, q, kv, table.contiguous(), torch.tensor(lens, dtype=torch.int32),
                       MLA_D_QK ** -0.5, lens)


# Dense MLA decode workload timed by bench.py: the pages fix the latent shape
# (576 / 512, one KV head) and show blocks of 64; the batch takes decode-sized
# sequences with 16 query heads per sequence (a DeepSeek-style model split 8
# ways by heads): 128 sequences of U[1024, 8192] cached tokens (about 680 MB of
# latent rows per call).
MLA_CONFIG = dict(batch=128, h_q=16, s_q=1, page_size=64, len_lo=1024, len_hi=8192, seed=6, pool_factor=1.25)


# The same batch with 64 query heads sharing each latent row (h_q = 64, as in a
# 128-head model split over two GPUs): one pass over the cache serves 64 rows.
MLA_WIDE_CONFIG = dict(MLA_CONFIG, h_q=64)


def make_mla_config(wide: bool = False, h_q: Optional[int] = None) -> MlaWorkload:
    """The MLA batch (16 query heads), its 64-head form (`wide`), or the same lengths and
    cache with `h_q` query heads."""
    c = MLA_WIDE_CONFIG if wide else MLA_CONFIG
    heads = c["h_q"] if h_q is None else int(h_q)
    g = torch.Generator().manual_seed(c["seed"])
    lens = torch.randint(c["len_lo"], c["len_hi"] + 1, (c["batch"],), generator=g).tolist()
    name = "mla_wide" if wide else "mla"
    return make_mla_workload(lens, heads, c["s_q"], c["page_size"], c["seed"] + 1000,
                             pool_factor=c["pool_factor"], name=name if h_q is None else f"mla_h{heads}")
