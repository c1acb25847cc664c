"""Float64 CPU oracle for paged GQA decode. Test infrastructure only.

Only the tests, the package entry's ``smoke()`` check and ``bench.py``'s
CPU-baseline / reference leg may import it; the CUDA library never does.
"""
from .oracle import (GQA_GROUP, HEAD_DIM, NUM_KV_HEADS, NUM_QO_HEADS, attend_rows,
                     gqa_paged_decode_oracle, merge_partials)

__all__ = ["GQA_GROUP", "HEAD_DIM", "NUM_KV_HEADS", "NUM_QO_HEADS", "attend_rows",
           "gqa_paged_decode_oracle", "merge_partials"]
