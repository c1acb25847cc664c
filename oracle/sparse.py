"""Float64 CPU oracle for selected-token (sparse) paged GQA decode.

TEST INFRASTRUCTURE. Only the test suite and ``bench.py``'s CPU-baseline leg may
import or run this module. The CUDA library never calls it, and it imports
nothing from the CUDA package.

What it computes follows the sparse split-K GQA path of the sigit.si vLLM
"qsa.py" page (``qsa_sparse_paged_attention`` and its
``_qsa_sparse_paged_gqa_splitk_kernel``). Every query row r belongs to request
``req = token_to_req[r]`` and selects TOPK logical token positions
``t = logical_indices[r, c]`` of that request. Column c is valid when

    0 <= req < num_requests,   t >= 0,   t // page_size < page_table_width,
    page = block_table[req, t // page_size],   0 <= page < num_cache_blocks,

and its key and value rows are then ``k_cache[page, t % page_size, g, :]``
and ``v_cache[page, t % page_size, g, :]`` for KV head g. Scores, softmax
and output are the dense definition (``attend_rows``) over the valid columns
only. A column that appears twice counts twice, as the kernel's column loop
does. A row with no valid column gives O = 0 (the kernel's ``has_values``
guard) and lse = -inf.

The page computes the scores with the fixed scale 1/sqrt(head_dim). Here
sm_scale is an argument, which callers set to that value. The page's function
returns only O. The log-sum-exp (base 2 of the natural-exponent sum, the
quantity its split partials carry) is returned as well.
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np
import torch

from .oracle import GQA_GROUP, HEAD_DIM, NUM_KV_HEADS, NUM_QO_HEADS, _as_np_int, _f64, attend_rows


def resolve_slots(logical_indices, block_table, token_to_req, page_size: int, num_cache_blocks: int) -> np.ndarray:
    """Physical slot (page * page_size + offset) of every selected column, or -1.

    Applies the validity rule above column by column. Returns int64 [R, TOPK].
    """
    idx = np.asarray(_as_np_int(logical_indices), dtype=np.int64)
    table = np.asarray(_as_np_int(block_table), dtype=np.int64)
    req = np.asarray(_as_np_int(token_to_req), dtype=np.int64)
    num_requests, width = table.shape
    out = np.full(idx.shape, -1, dtype=np.int64)
    for r in range(idx.shape[0]):
        q = int(req[r])
        if q < 0 or q >= num_requests:
            continue
        for c in range(idx.shape[1]):
            t = int(idx[r, c])
            if t < 0:
                continue
            lp = t // page_size
            if lp >= width:
                continue
            page = int(table[q, lp])
            if page < 0 or page >= num_cache_blocks:
                continue
            out[r, c] = page * page_size + t % page_size
    return out


def sparse_paged_decode_oracle(q, k_cache, v_cache, logical_indices, block_table, token_to_req, sm_scale: float,
                               rows: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Float64 (O [R, 32, 128], lse [R, 32]) of the rows in ``rows`` (None: all).

    q: [R, 32, 128] bf16; k_cache, v_cache: [num_cache_blocks, page_size, 4, 128]
    bf16; logical_indices: [R, TOPK] int32; block_table: [num_requests, width]
    int32; token_to_req: [R] int32. Rows not listed are left as NaN.
    """
    num_blocks, page_size = int(k_cache.shape[0]), int(k_cache.shape[1])
    slots = resolve_slots(logical_indices, block_table, token_to_req, page_size, num_blocks)
    n_rows = slots.shape[0]
    out = np.full((n_rows, NUM_QO_HEADS, HEAD_DIM), np.nan)
    lse = np.full((n_rows, NUM_QO_HEADS), np.nan)
    kf = k_cache.reshape(num_blocks * page_size, NUM_KV_HEADS, HEAD_DIM)  # slot-major view
    vf = v_cache.reshape(num_blocks * page_size, NUM_KV_HEADS, HEAD_DIM)
    todo = range(n_rows) if rows is None else rows
    for r in todo:
        sel = slots[r][slots[r] >= 0]                      # valid columns, in column order
        sel_t = torch.as_tensor(sel)
        kr = _f64(kf.index_select(0, sel_t) if isinstance(kf, torch.Tensor) else np.asarray(kf)[sel])
        vr = _f64(vf.index_select(0, sel_t) if isinstance(vf, torch.Tensor) else np.asarray(vf)[sel])
        qr = _f64(q[r])
        for g in range(NUM_KV_HEADS):
            heads = slice(g * GQA_GROUP, (g + 1) * GQA_GROUP)
            out[r, heads], lse[r, heads] = attend_rows(qr[heads], kr[:, g, :], vr[:, g, :], sm_scale)
    return out, lse
