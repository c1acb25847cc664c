"""Reference KV-cache append for paged GQA decode. TEST INFRASTRUCTURE only (tests,
bench.py's CPU baseline); the CUDA library never imports it.

The row store of the split-K GQA path on the sigit.si vLLM "qsa.py" page
(``_store_qsa_rows_kernel`` / ``qsa_store_cache_rows``): each new row r carries a
slot; a slot is valid when 0 <= slot < num_pages * page_size, and then
cache[slot // page_size, slot % page_size] = row. Invalid slots (for example -1
for padding tokens) store nothing. With page size 1 the slot is the page id,
and K and V rows of all 4 KV heads of a token are stored together.
"""
from __future__ import annotations

import numpy as np
import torch


def kv_append_oracle(k_new, v_new, slots, k_cache, v_cache):
    """Return new (k_cache, v_cache) CPU tensors with the valid rows stored.

    k_new, v_new: [N, 4, 128]; slots: [N] int32; caches: [P, 1, 4, 128].
    Rows go in order, so if two valid rows name the same slot the later one is
    kept (the GPU kernel leaves which one unspecified).
    """
    k_out = k_cache.clone()
    v_out = v_cache.clone()
    num_pages = k_cache.shape[0]
    s = np.asarray(slots.cpu() if isinstance(slots, torch.Tensor) else slots, dtype=np.int64)
    for r, slot in enumerate(s.tolist()):
        if 0 <= slot < num_pages:
            k_out[slot, 0] = k_new[r]
            v_out[slot, 0] = v_new[r]
    return k_out, v_out
