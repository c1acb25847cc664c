"""GB300 (sm_103a) paged-KV GQA decode: h32 / kv4 / d128 / page size 1, bf16.

``run(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale=None) -> (out, lse)``
calls the CUDA library through its C ABI (include/gqa_paged_decode.h). The
library is built in-tree by ``paged_kv_gqa_split_gb300.build.build()``; it is
loaded on first use, and every call fails loudly if it is missing.
``sparse_run(q, k_cache, v_cache, logical_indices, block_table, token_to_req)``
is the selected-token variant over a block table of any page size,
``run_fp8`` reads an FP8 (e4m3, per-128 fp32 scale) cache, ``mla_run`` is
the dense MLA decode over one 576-value latent KV head, and
``kv_append`` stores new tokens' K/V rows into the page pool.
"""
from ._lib import GqaError, kv_append, mla_run, run, run_checked, run_fp8, sparse_run  # noqa: F401

__all__ = ["GqaError", "kv_append", "mla_run", "run", "run_checked", "run_fp8", "sparse_run"]
