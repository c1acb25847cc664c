"""Float64 CPU oracle for dense MLA paged decode (one latent KV head).

TEST INFRASTRUCTURE. Only the test suite and ``bench.py``'s CPU-baseline leg may
import or run this module. The CUDA library never calls it, and it imports
nothing from the CUDA package.

What it computes follows the dense decode kernel of the flash_mla_with_kvcache
page (docs.flagos.io, FlagGems; ``flash_mla_with_kvcache`` with
``_dense_decode_dispatch``). The cache holds one latent row of d_qk = 576
values per token (512 "NoPE" values followed by 64 "RoPE" values), in blocks
of page_size tokens: request b's token t lives at block
block_table[b, t // page_size], offset t % page_size. For every query row
(query token i of s_q, query head h of h_q) of sequence b:

    s_t   = softmax_scale * q[b, i, h, :] . kv_t[:]      (all 576 values)
    O     = sum_t softmax(s)_t * kv_t[:512]               (the NoPE part is V)
    lse   = log sum_t exp(s_t)                            (natural log)

over t < cache_seqlens[b] (the page's dense kernel is not causal within the
rows of one call). O is [B, s_q, h_q, 512]; lse is [B, h_q, s_q], the page's
layout. A sequence with no cached token gives O = 0 and lse = -inf. Tokens
the page leaves undefined (past the block table, or in a block outside the
pool) are left out (``mla_slots``).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np
import torch

from .oracle import _as_np_int, _f64, attend_rows

D_QK = 576
D_V = 512


def mla_slots(block_table, cache_seqlens, page_size: int, num_blocks: Optional[int] = None) -> list:
    """Per sequence, the flat slot (block * page_size + offset) of every cached
    token. Where the page leaves the result undefined (its kernel would read
    outside the table or the pool), this reading leaves the token out: tokens
    past the table's width * page_size, and tokens whose block lies outside
    [0, num_blocks)."""
    table = np.asarray(_as_np_int(block_table), dtype=np.int64)
    lens = np.asarray(_as_np_int(cache_seqlens), dtype=np.int64)
    cap = table.shape[1] * page_size
    out = []
    for b in range(lens.shape[0]):
        t = np.arange(min(max(int(lens[b]), 0), cap), dtype=np.int64)
        blk = table[b, t // page_size]
        keep = blk >= 0 if num_blocks is None else (blk >= 0) & (blk < num_blocks)
        out.append((blk * page_size + t % page_size)[keep])
    return out


def mla_decode_oracle(q, kv_cache, block_table, cache_seqlens, softmax_scale: float,
                      seqs: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Float64 (O [B, s_q, h_q, 512], lse [B, h_q, s_q]) for the sequences in ``seqs``.

    q: [B, s_q, h_q, 576] bf16; kv_cache: [num_blocks, page_size, 1, 576] bf16.
    Sequences not listed are left as NaN.
    """
    bsz, s_q, h_q, d = (int(x) for x in q.shape)
    num_blocks, page_size = int(kv_cache.shape[0]), int(kv_cache.shape[1])
    flat = kv_cache.reshape(num_blocks * page_size, D_QK)
    out = np.full((bsz, s_q, h_q, D_V), np.nan)
    lse = np.full((bsz, h_q, s_q), np.nan)
    slots = mla_slots(block_table, cache_seqlens, page_size, num_blocks)
    todo = range(bsz) if seqs is None else seqs
    for b in todo:
        if len(slots[b]) == 0:                                   # nothing cached: O = 0, lse = -inf
            out[b] = 0.0
            lse[b] = -np.inf
            continue
        idx = torch.as_tensor(slots[b])
        kv = _f64(flat.index_select(0, idx) if isinstance(flat, torch.Tensor) else np.asarray(flat)[slots[b]])
        qb = _f64(q[b]).reshape(s_q * h_q, D_QK)               # rows (i, h)
        o, lse2 = attend_rows(qb, kv, kv[:, :D_V], softmax_scale)
        out[b] = o.reshape(s_q, h_q, D_V)
        lse[b] = (lse2 * math.log(2.0)).reshape(s_q, h_q).T     # natural log, [h_q, s_q]
    return out, lse
