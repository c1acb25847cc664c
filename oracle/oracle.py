"""Float64 CPU oracle for batched paged-KV GQA decode attention.

TEST INFRASTRUCTURE. Only the test suite, the package entry's ``smoke()`` check
and ``bench.py``'s CPU-baseline / reference leg may import or run this module.
The CUDA library never calls it, and it imports nothing from the CUDA package.

What it computes (the plain definition, evaluated directly):

For every sequence b with n_b = kv_indptr[b+1] - kv_indptr[b] cached tokens,
every query head h and its KV head g = h // 8 (32 query heads over 4 KV heads,
consecutive groups of 8, as in the kernel of the kernelindex.com page
"gqa_paged_decode_h32_kv4_d128_ps1", step 7 "kv_head_indices = offs_h //
gqa_ratio"):

    p_j  = kv_indices[kv_indptr[b] + j]                 page of token j
    s_j  = sm_scale * sum_d q[b, h, d] * k_cache[p_j, 0, g, d]
    m    = max_j s_j
    l    = sum_j exp(s_j - m)
    O[b, h, :] = sum_j exp(s_j - m) * v_cache[p_j, 0, g, :] / l
    lse[b, h]  = (m + ln l) / ln 2   = log2 sum_j exp(s_j)

The log-sum-exp is base 2 of a natural-exponent sum, which is what the same
page's kernel stores in its final step ("2-based log-sum-exp": (m + log l) *
1/ln 2) and what its ``run()`` docstring calls "log-sum-exp of attention logits
(base 2)". An empty sequence gives O = 0 and lse = -inf (that kernel's step 4,
"Early exit for sequences with no KV cache").

Softmax is taken in two passes (max first, then the shifted exponentials) in
float64; bf16 inputs convert to float64 exactly. Results stay float64: no
rounding to bf16 is applied to O.

``merge_partials`` is the split-combination identity used by the split-K GQA
path on the sigit.si vLLM "qsa.py" page (``_qsa_merge_splitk_kernel``): weights
w_i = 2^(lse_i - max_i lse_i), O = sum_i w_i O_i / sum_i w_i, extended with the
merged log-sum-exp max + log2 sum_i w_i. The oracle uses it only as a checked
identity (tests merge oracle partials and compare with the whole).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np
import torch

NUM_QO_HEADS = 32
NUM_KV_HEADS = 4
GQA_GROUP = NUM_QO_HEADS // NUM_KV_HEADS  # 8 query heads share one KV head
HEAD_DIM = 128
LN2 = math.log(2.0)


def _f64(t) -> np.ndarray:
    """Exact widening of a bf16/fp32 tensor (or array) to float64 numpy."""
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def attend_rows(qg: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float
                ) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of query rows over one key/value list, float64.

    qg: [R, D] query rows sharing one KV head; k, v: [n, D].
    Returns (O [R, D], lse2 [R]) with lse2 = log2 sum_j exp(s_j).
    n == 0 gives zeros and -inf.
    """
    r = qg.shape[0]
    if k.shape[0] == 0:
        return np.zeros((r, qg.shape[1])), np.full(r, -np.inf)
    s = sm_scale * (qg @ k.T)                     # [R, n] scaled scores
    m = s.max(axis=1, keepdims=True)              # pass 1: row maxima
    e = np.exp(s - m)                             # pass 2: shifted exponentials
    l = e.sum(axis=1, keepdims=True)
    o = (e @ v) / l
    lse2 = (m[:, 0] + np.log(l[:, 0])) / LN2
    return o, lse2


def gqa_paged_decode_oracle(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale: float,
                            seqs: Optional[Iterable[int]] = None
                            ) -> Tuple[np.ndarray, np.ndarray]:
    """Float64 outputs (O [B, 32, 128], lse [B, 32]) for the sequences in ``seqs``.

    Inputs are CPU tensors (bf16 q/k/v, int32 indptr/indices) or arrays. Rows of
    sequences not listed in ``seqs`` are left as NaN, so a sampled comparison
    cannot silently pass on them. ``seqs=None`` computes every sequence.
    """
    indptr = np.asarray(_as_np_int(kv_indptr), dtype=np.int64)
    indices = _as_np_int(kv_indices)
    batch = indptr.shape[0] - 1
    out = np.full((batch, NUM_QO_HEADS, HEAD_DIM), np.nan)
    lse = np.full((batch, NUM_QO_HEADS), np.nan)
    todo = range(batch) if seqs is None else seqs
    for b in todo:
        lo, hi = int(indptr[b]), int(indptr[b + 1])
        pages = torch.as_tensor(np.asarray(indices[lo:hi], dtype=np.int64))
        qb = _f64(q[b])                                   # [32, 128]
        kb = _f64(_gather(k_cache, pages))                # [n, 4, 128]
        vb = _f64(_gather(v_cache, pages))
        for g in range(NUM_KV_HEADS):
            heads = slice(g * GQA_GROUP, (g + 1) * GQA_GROUP)
            out[b, heads], lse[b, heads] = attend_rows(qb[heads], kb[:, g, :], vb[:, g, :], sm_scale)
    return out, lse


def merge_partials(parts: Sequence[Tuple[np.ndarray, np.ndarray]]) -> Tuple[np.ndarray, np.ndarray]:
    """Combine per-split (O_i [..., D], lse_i [...]) into the whole, float64.

    w_i = 2^(lse_i - M) with M = max_i lse_i; O = sum_i w_i O_i / sum_i w_i;
    lse = M + log2 sum_i w_i. Where every lse_i is -inf: O = 0, lse = -inf.
    """
    lses = np.stack([p[1] for p in parts])            # [S, ...]
    outs = np.stack([p[0] for p in parts])            # [S, ..., D]
    mx = lses.max(axis=0)
    finite = np.isfinite(mx)
    safe_mx = np.where(finite, mx, 0.0)
    w = np.where(np.isfinite(lses), np.exp2(lses - safe_mx), 0.0)
    den = w.sum(axis=0)
    num = (w[..., None] * np.where(np.isfinite(lses)[..., None], outs, 0.0)).sum(axis=0)
    o = np.where(finite[..., None], num / np.where(den > 0, den, 1.0)[..., None], 0.0)
    lse = np.where(finite, safe_mx + np.log2(np.where(den > 0, den, 1.0)), -np.inf)
    return o, lse


def _gather(cache, pages: torch.Tensor):
    """Pages cache[p, 0, :, :] of one sequence (page size 1): [n, 4, 128]."""
    if isinstance(cache, torch.Tensor):
        return cache.index_select(0, pages)[:, 0, :, :]
    return np.asarray(cache)[pages.numpy(), 0, :, :]


def _as_np_int(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").numpy()
    return np.asarray(x)
