"""Float64 CPU oracle for paged GQA decode over an FP8 (e4m3) KV cache.

TEST INFRASTRUCTURE. Only the test suite and ``bench.py``'s CPU-baseline leg may
import or run this module. The CUDA library never calls it, and it imports
nothing from the CUDA package.

Cache format. The FP8 KV cache of the flash_mla_with_kvcache page
(docs.flagos.io, FlagGems) stores each token as float8_e4m3 values followed
by float32 scales, one scale per 128 values ("Scale factors: 4 float32
values (each for 128 FP8 values)"), and dequantizes a value as fp8 * scale.
For the GQA shape here (4 KV heads of 128 dims, page size 1) one token row
of the K cache (and likewise of the V cache) is 528 bytes:

    bytes [0, 512)    : e4m3 values of KV heads 0..3, 128 each, head-major
    bytes [512, 528)  : 4 little-endian float32 scales, one per KV head

so K[p, g, d] = e4m3(byte[p, 128 g + d]) * scale[p, g]. The page's MLA
layout also carries a bf16 RoPE part; GQA has none.

e4m3 ("e4m3fn"): sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
exponent field 0 encodes subnormals m/8 * 2^-6; 0x7F and 0xFF are NaN; there
is no infinity; the largest finite value is 448.

Attention is then the dense definition (``gqa_paged_decode_oracle``) over
the dequantized cache, evaluated in float64.
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np
import torch

from .oracle import HEAD_DIM, NUM_KV_HEADS, _as_np_int, gqa_paged_decode_oracle

ROW_BYTES = NUM_KV_HEADS * HEAD_DIM + 4 * NUM_KV_HEADS  # 528


def e4m3_decode(codes) -> np.ndarray:
    """Float64 values of e4m3 codes (any integer array of bytes)."""
    b = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    normal = sign * (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = sign * (m / 8.0) * 2.0 ** -6
    out = np.where(e == 0, sub, normal)
    return np.where((b & 0x7F) == 0x7F, np.nan, out)


def dequantize_rows(cache) -> np.ndarray:
    """[P, 528] uint8 rows -> float64 [P, 4, 128] values times their head's scale."""
    raw = np.ascontiguousarray(_as_np_int(cache), dtype=np.uint8).reshape(-1, ROW_BYTES)
    vals = e4m3_decode(raw[:, :NUM_KV_HEADS * HEAD_DIM]).reshape(-1, NUM_KV_HEADS, HEAD_DIM)
    scales = raw[:, NUM_KV_HEADS * HEAD_DIM:].copy().view("<f4").astype(np.float64)  # [P, 4]
    return vals * scales[:, :, None]


def gqa_paged_decode_fp8_oracle(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale: float,
                                seqs: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Float64 (O [B, 32, 128], lse [B, 32]) over FP8 caches of [P, 528] bytes."""
    k = dequantize_rows(k_cache)[:, None]          # [P, 1, 4, 128] float64, page size 1
    v = dequantize_rows(v_cache)[:, None]
    idx = torch.as_tensor(np.asarray(_as_np_int(kv_indices), dtype=np.int64))
    return gqa_paged_decode_oracle(q, k, v, kv_indptr, idx, sm_scale, seqs)
