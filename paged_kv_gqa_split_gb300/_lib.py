"""ctypes binding of the C ABI in include/gqa_paged_decode.h.

Argument marshalling only: every step of the computation runs in the CUDA
library. The functions named like the C entry points take raw device pointers
(ints) and return the C status code; ``run`` is the tensor-level convenience
that mirrors the problem's ``run(q, k_cache, v_cache, kv_indptr, kv_indices,
sm_scale)`` (kernelindex.com page "gqa_paged_decode_h32_kv4_d128_ps1") with
caller-visible outputs. There is no CPU path: CPU tensors, or a missing
library, raise.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgqa_paged_decode.so")

GQA_OK = 0
GQA_ERR_INVALID_ARGUMENT = -1
GQA_ERR_WORKSPACE = -2
GQA_ERR_LAUNCH = -3
GQA_ERR_UNSUPPORTED_DEVICE = -4

NUM_QO_HEADS, NUM_KV_HEADS, HEAD_DIM, PAGE_SIZE = 32, 4, 128, 1

_vp = ctypes.c_void_p
_SIGNATURES = {
    "gqa_paged_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.c_int, _vp]),
    "gqa_paged_decode_ws_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64]),
    "gqa_paged_decode_ws": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.c_int, _vp,
                                           _vp, ctypes.c_size_t]),
    "gqa_paged_decode_checked": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.c_int,
                                                _vp, ctypes.c_int, _vp]),
    "gqa_paged_decode_release": (None, []),
    "gqa_paged_decode_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "gqa_paged_decode_set_tuning": (ctypes.c_int, [ctypes.c_int] * 10),
    "gqa_paged_decode_set_profile_events": (ctypes.c_int, [_vp, _vp]),
    "gqa_paged_decode_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
    "gqa_paged_decode_plan": (ctypes.c_int64, [_vp] + [ctypes.c_int] * 7 + [_vp, ctypes.c_int64]),
    "gqa_paged_kv_append": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, _vp]),
    "gqa_paged_decode_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.c_int, _vp]),
    "gqa_sparse_paged_decode": (ctypes.c_int, [_vp] * 6 + [ctypes.c_float, _vp, _vp] + [ctypes.c_int] * 6 + [_vp]),
    "gqa_paged_decode_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.c_int, _vp]),
    "gqa_mla_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp] + [ctypes.c_int] * 6 + [_vp]),
    "gqa_mla_set_tuning": (ctypes.c_int, [ctypes.c_int]),
    "gqa_paged_decode_set_merge_mode": (ctypes.c_int, [ctypes.c_int]),
    "gqa_paged_decode_last_launch_count": (ctypes.c_int, []),
    "gqa_paged_decode_test_fail_allocs": (ctypes.c_int, [ctypes.c_int]),
    "gqa_paged_decode_test_wait_limit_ns": (ctypes.c_int, [ctypes.c_uint64]),
}

_lib: Optional[ctypes.CDLL] = None


class GqaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where} failed with {code}: {strerror(code)}")
        self.code = code


def load() -> ctypes.CDLL:
    """Load the shared library (built by ``paged_kv_gqa_split_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m paged_kv_gqa_split_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


# ------------------------------------------------------ C entry points, 1:1
def gqa_paged_decode(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream) -> int:
    return load().gqa_paged_decode(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream)


def gqa_paged_decode_ws_size(batch: int, total_tokens_upper_bound: int) -> int:
    return load().gqa_paged_decode_ws_size(batch, total_tokens_upper_bound)


def gqa_paged_decode_ws(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream,
                        workspace, workspace_bytes) -> int:
    return load().gqa_paged_decode_ws(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream,
                                      workspace, workspace_bytes)


def gqa_paged_decode_checked(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream,
                             num_pages, dev_err) -> int:
    return load().gqa_paged_decode_checked(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch,
                                           stream, num_pages, dev_err)


def gqa_paged_decode_release() -> None:
    load().gqa_paged_decode_release()


def gqa_paged_decode_strerror(code: int) -> str:
    return load().gqa_paged_decode_strerror(code).decode()


strerror = gqa_paged_decode_strerror


GATHER_LSU, GATHER_TMA, GATHER_LSU_F8, GATHER_LSU_CUDA_CORES = 0, 1, 2, 3


def gqa_paged_decode_set_tuning(num_ctas=0, min_units_per_cta=0, heads_per_cta=0, tile=0, stages=0,
                                gather=GATHER_LSU, fused_merge_max_splits=0, tier2_ctas=0, tier2_permille=0,
                                tier2_min_units=0) -> int:
    return load().gqa_paged_decode_set_tuning(num_ctas, min_units_per_cta, heads_per_cta, tile, stages, gather,
                                              fused_merge_max_splits, tier2_ctas, tier2_permille, tier2_min_units)


def gqa_paged_decode_set_profile_events(decode_start, decode_stop) -> int:
    return load().gqa_paged_decode_set_profile_events(decode_start, decode_stop)


def gqa_paged_decode_plan(kv_indptr, num_ctas: int, min_units_per_cta: int = 0, heads_per_cta: int = 4,
                          tier2_ctas: int = 0, tier2_permille: int = 0, tier2_min_units: int = 0):
    """Host-side split plan for a CPU int32 kv_indptr: a list of 9-tuples (decode CTA,
    sequence, head group, token lo, token hi, slot or -1, merge first CTA, merge last
    CTA, merge first slot). num_ctas tier-1 CTAs plus tier2_ctas tier-2 CTAs."""
    import numpy as np
    ip = np.ascontiguousarray(np.asarray(kv_indptr, dtype=np.int32))
    batch = ip.shape[0] - 1
    ptr = ip.ctypes.data_as(ctypes.c_void_p)
    args = (ptr, batch, num_ctas, min_units_per_cta, heads_per_cta, tier2_ctas, tier2_permille, tier2_min_units)
    n = load().gqa_paged_decode_plan(*args, None, 0)
    if n < 0:
        raise GqaError(int(n), "gqa_paged_decode_plan")
    out = np.zeros((max(n, 1), 9), dtype=np.int64)
    n2 = load().gqa_paged_decode_plan(*args, out.ctypes.data_as(ctypes.c_void_p), n)
    assert n2 == n
    return [tuple(int(x) for x in row) for row in out[:n]]


def gqa_paged_decode_device_error() -> int:
    flags = ctypes.c_int(0)
    rc = load().gqa_paged_decode_device_error(ctypes.byref(flags))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_paged_decode_device_error")
    return flags.value


MERGE_KERNEL, MERGE_ONE_WAVE = 0, 1


def gqa_paged_decode_set_merge_mode(mode: int) -> int:
    return load().gqa_paged_decode_set_merge_mode(mode)


def gqa_paged_decode_last_launch_count() -> int:
    return load().gqa_paged_decode_last_launch_count()


def gqa_paged_decode_test_fail_allocs(count: int) -> int:
    return load().gqa_paged_decode_test_fail_allocs(count)


def gqa_paged_decode_test_wait_limit_ns(ns: int) -> int:
    return load().gqa_paged_decode_test_wait_limit_ns(ns)


def gqa_paged_kv_append(k_new, v_new, slots, k_cache, v_cache, num_tokens, num_pages, stream) -> int:
    return load().gqa_paged_kv_append(k_new, v_new, slots, k_cache, v_cache, num_tokens, num_pages, stream)


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, slots: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Store each new token's K/V rows into page slots[r] of the caches (in place);
    slots outside [0, num_pages) are skipped."""
    for name, t in (("k_new", k_new), ("v_new", v_new), ("slots", slots), ("k_cache", k_cache), ("v_cache", v_cache)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor: the library has no CPU path")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != k_cache.device:
            raise ValueError(f"all tensors must be on {k_cache.device}")
    n = int(slots.shape[0]) if slots.dim() == 1 else -1
    if n < 0 or tuple(k_new.shape) != (n, NUM_KV_HEADS, HEAD_DIM) or k_new.shape != v_new.shape:
        raise ValueError("expected k_new / v_new [N, 4, 128] and slots [N]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM) or \
            v_cache.shape != k_cache.shape:
        raise ValueError("expected k_cache / v_cache [P, 1, 4, 128]")
    if any(t.dtype != torch.bfloat16 for t in (k_new, v_new, k_cache, v_cache)) or slots.dtype != torch.int32:
        raise ValueError("K/V tensors must be bfloat16 and slots int32")
    if stream is None:
        stream = torch.cuda.current_stream(k_cache.device)
    with torch.cuda.device(k_cache.device):
        rc = gqa_paged_kv_append(k_new.data_ptr(), v_new.data_ptr(), slots.data_ptr(), k_cache.data_ptr(),
                                 v_cache.data_ptr(), n, int(k_cache.shape[0]), stream.cuda_stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_paged_kv_append")


def gqa_paged_decode_noalloc(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream) -> int:
    """As gqa_paged_decode, with the split partials in the library's fixed device
    array instead of an allocated workspace (for callers that cannot allocate)."""
    return load().gqa_paged_decode_noalloc(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch,
                                           stream)


# ------------------------------------------------------------- tensor level
def _check_inputs(q, k_cache, v_cache, kv_indptr, kv_indices):
    """Shape / constant checks of the problem's run() wrapper, plus dtype,
    device and contiguity (no host sync: kv_indptr[-1] is not read)."""
    tensors = {"q": q, "k_cache": k_cache, "v_cache": v_cache, "kv_indptr": kv_indptr, "kv_indices": kv_indices}
    for name, t in tensors.items():
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} is on {t.device}: the CUDA library has no CPU path; move inputs to the GPU")
        if t.device != q.device:
            raise ValueError(f"all inputs must be on {q.device}; {name} is on {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected q [B, 32, 128] and k_cache / v_cache [P, 1, 4, 128]")
    batch, heads, dim = q.shape
    _, page_size, kv_heads, kdim = k_cache.shape
    if heads != NUM_QO_HEADS:
        raise ValueError(f"expected num_qo_heads=32, got {heads}")
    if kv_heads != NUM_KV_HEADS:
        raise ValueError(f"expected num_kv_heads=4, got {kv_heads}")
    if dim != HEAD_DIM or kdim != HEAD_DIM:
        raise ValueError(f"expected head_dim=128, got {dim}/{kdim}")
    if page_size != PAGE_SIZE:
        raise ValueError(f"expected page_size=1, got {page_size}")
    for name in ("q", "k_cache", "v_cache"):
        if tensors[name].dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    for name in ("kv_indptr", "kv_indices"):
        if tensors[name].dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if kv_indptr.shape != (batch + 1,):
        raise ValueError(f"expected kv_indptr shape {(batch + 1,)}, got {tuple(kv_indptr.shape)}")
    if kv_indices.dim() != 1:
        raise ValueError("kv_indices must be 1-D")
    return batch


def run(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_indptr: torch.Tensor,
        kv_indices: torch.Tensor, sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
        workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged GQA decode on the GPU. Returns (out [B, 32, 128] bf16, lse [B, 32] fp32, base 2)."""
    batch = _check_inputs(q, k_cache, v_cache, kv_indptr, kv_indices)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((batch, NUM_QO_HEADS), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() or out.device != q.device:
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")
    if lse.shape != (batch, NUM_QO_HEADS) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, 32]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), kv_indptr.data_ptr(), kv_indices.data_ptr(),
                float(sm_scale), out.data_ptr(), lse.data_ptr(), batch, stream.cuda_stream)
        if workspace is None:
            rc = gqa_paged_decode(*args)
            where = "gqa_paged_decode"
        else:
            rc = gqa_paged_decode_ws(*args, workspace.data_ptr(), workspace.numel() * workspace.element_size())
            where = "gqa_paged_decode_ws"
    if rc != GQA_OK:
        raise GqaError(rc, where)
    return out, lse


def run_checked(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale=None, out=None, lse=None):
    """``run`` through the checked entry point. Returns (out, lse, dev_err) with
    dev_err a device int32 tensor [1] (0 = the page table was valid)."""
    batch = _check_inputs(q, k_cache, v_cache, kv_indptr, kv_indices)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((batch, NUM_QO_HEADS), dtype=torch.float32, device=q.device)
    dev_err = torch.zeros(1, dtype=torch.int32, device=q.device)
    stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = gqa_paged_decode_checked(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), kv_indptr.data_ptr(),
                                      kv_indices.data_ptr(), float(sm_scale), out.data_ptr(), lse.data_ptr(), batch,
                                      stream.cuda_stream, int(k_cache.shape[0]), dev_err.data_ptr())
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_paged_decode_checked")
    return out, lse, dev_err


def gqa_sparse_paged_decode(q, k_cache, v_cache, logical_indices, block_table, token_to_req, sm_scale, out, lse,
                            rows, topk, page_size, num_cache_blocks, num_requests, page_table_width, stream) -> int:
    return load().gqa_sparse_paged_decode(q, k_cache, v_cache, logical_indices, block_table, token_to_req, sm_scale,
                                          out, lse, rows, topk, page_size, num_cache_blocks, num_requests,
                                          page_table_width, stream)


def sparse_run(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, logical_indices: torch.Tensor,
               block_table: torch.Tensor, token_to_req: torch.Tensor, sm_scale: Optional[float] = None,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, with_lse: bool = True,
               stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Selected-token paged GQA decode on the GPU (the shape checks of the qsa.py
    page's ``qsa_sparse_paged_attention``, for 32 query heads over 4 KV heads of
    dimension 128). Returns (out [rows, 32, 128] bf16, lse [rows, 32] fp32 or None)."""
    tensors = {"q": q, "k_cache": k_cache, "v_cache": v_cache, "logical_indices": logical_indices,
               "block_table": block_table, "token_to_req": token_to_req}
    for name, t in tensors.items():
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} is on {t.device}: the CUDA library has no CPU path; move inputs to the GPU")
        if t.device != q.device:
            raise ValueError(f"all inputs must be on {q.device}; {name} is on {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected q [rows, 32, 128] and k_cache / v_cache [blocks, page_size, 4, 128]")
    if logical_indices.dim() != 2 or logical_indices.shape[0] != q.shape[0]:
        raise ValueError("logical_indices must have one row per query")
    if token_to_req.shape != (q.shape[0],) or block_table.dim() != 2:
        raise ValueError("token_to_req must be [rows] and block_table [requests, width]")
    if not all(k_cache.shape[:3]) or not all(block_table.shape) or logical_indices.shape[1] <= 0:
        raise ValueError("the cache, the block table and the selection width must be nonempty")
    if tuple(q.shape[1:]) != (NUM_QO_HEADS, HEAD_DIM) or tuple(k_cache.shape[2:]) != (NUM_KV_HEADS, HEAD_DIM):
        raise ValueError("expected 32 query heads over 4 KV heads of dimension 128")
    for name in ("q", "k_cache", "v_cache"):
        if tensors[name].dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    for name in ("logical_indices", "block_table", "token_to_req"):
        if tensors[name].dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    rows, topk = int(logical_indices.shape[0]), int(logical_indices.shape[1])
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() or out.device != q.device:
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")
    if lse is None and with_lse:
        lse = torch.empty((rows, NUM_QO_HEADS), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (rows, NUM_QO_HEADS) or lse.dtype != torch.float32 or
                            not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor [rows, 32]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = gqa_sparse_paged_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), logical_indices.data_ptr(),
                                     block_table.data_ptr(), token_to_req.data_ptr(), float(sm_scale),
                                     out.data_ptr(), lse.data_ptr() if lse is not None else None, rows, topk,
                                     int(k_cache.shape[1]), int(k_cache.shape[0]), int(block_table.shape[0]),
                                     int(block_table.shape[1]), stream.cuda_stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_sparse_paged_decode")
    return out, lse


FP8_ROW_BYTES = NUM_KV_HEADS * HEAD_DIM + 4 * NUM_KV_HEADS  # 512 e4m3 codes + 4 fp32 scales per token


def gqa_paged_decode_fp8(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream) -> int:
    return load().gqa_paged_decode_fp8(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, out, lse, batch, stream)


def run_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_indptr: torch.Tensor,
            kv_indices: torch.Tensor, sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged GQA decode over FP8 caches of [P, 528] uint8 rows (4 KV heads x 128
    e4m3 codes, then the 4 heads' float32 scales). Returns (out [B, 32, 128]
    bf16, lse [B, 32] fp32, base 2)."""
    tensors = {"q": q, "k_cache": k_cache, "v_cache": v_cache, "kv_indptr": kv_indptr, "kv_indices": kv_indices}
    for name, t in tensors.items():
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} is on {t.device}: the CUDA library has no CPU path; move inputs to the GPU")
        if t.device != q.device:
            raise ValueError(f"all inputs must be on {q.device}; {name} is on {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 3 or tuple(q.shape[1:]) != (NUM_QO_HEADS, HEAD_DIM) or q.dtype != torch.bfloat16:
        raise ValueError("expected q [B, 32, 128] bf16")
    for name in ("k_cache", "v_cache"):
        t = tensors[name]
        if t.dtype != torch.uint8 or t.dim() < 2 or t.shape[-1] != FP8_ROW_BYTES:
            raise ValueError(f"{name} must be uint8 rows of {FP8_ROW_BYTES} bytes ([P, {FP8_ROW_BYTES}])")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    for name in ("kv_indptr", "kv_indices"):
        if tensors[name].dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if kv_indptr.dim() != 1 or kv_indptr.shape[0] < 1:
        raise ValueError("kv_indptr must be [B + 1]")
    batch = int(q.shape[0])
    if kv_indptr.shape[0] != batch + 1:
        raise ValueError(f"kv_indptr has {kv_indptr.shape[0]} entries; expected batch + 1 = {batch + 1}")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((batch, NUM_QO_HEADS), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = gqa_paged_decode_fp8(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), kv_indptr.data_ptr(),
                                  kv_indices.data_ptr(), float(sm_scale), out.data_ptr(), lse.data_ptr(), batch,
                                  stream.cuda_stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_paged_decode_fp8")
    return out, lse


MLA_D_QK, MLA_D_V = 576, 512


def gqa_mla_set_tuning(kernel: int) -> int:
    """MLA decode kernel: 0 default (the tensor-memory kernel for 64-row multiples and block sizes
    that are a multiple of 32, else mma.sync with 3 stages), 1 the tensor-memory kernel (block
    sizes that are a multiple of 32), 3 or 4 the mma.sync kernel with that ring depth."""
    return load().gqa_mla_set_tuning(kernel)


def gqa_mla_decode(q, kv_cache, block_table, cache_seqlens, softmax_scale, out, lse, batch, s_q, h_q, page_size,
                   num_blocks, page_table_width, stream) -> int:
    return load().gqa_mla_decode(q, kv_cache, block_table, cache_seqlens, softmax_scale, out, lse, batch, s_q, h_q,
                                 page_size, num_blocks, page_table_width, stream)


def mla_run(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor, cache_seqlens: torch.Tensor,
            softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, with_lse: bool = True,
            stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Dense MLA paged decode on the GPU (flash_mla_with_kvcache's dense path,
    one latent KV head of 576 values, d_v = 512). Returns (out [B, s_q, h_q, 512]
    bf16, lse [B, h_q, s_q] fp32 natural log, or None)."""
    tensors = {"q": q, "kv_cache": kv_cache, "block_table": block_table, "cache_seqlens": cache_seqlens}
    for name, t in tensors.items():
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} is on {t.device}: the CUDA library has no CPU path; move inputs to the GPU")
        if t.device != q.device:
            raise ValueError(f"all inputs must be on {q.device}; {name} is on {t.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or q.shape[-1] != MLA_D_QK or q.dtype != torch.bfloat16:
        raise ValueError("expected q [B, s_q, h_q, 576] bf16")
    if kv_cache.dim() != 4 or kv_cache.shape[2] != 1 or kv_cache.shape[3] != MLA_D_QK or \
            kv_cache.dtype != torch.bfloat16:
        raise ValueError("expected kv_cache [num_blocks, page_size, 1, 576] bf16 (one latent KV head)")
    bsz, s_q, h_q = (int(x) for x in q.shape[:3])
    if block_table.dim() != 2 or block_table.shape[0] != bsz or block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32 [B, width]")
    if cache_seqlens.shape != (bsz,) or cache_seqlens.dtype != torch.int32:
        raise ValueError("cache_seqlens must be int32 [B]")
    if (s_q * h_q) % 16:
        raise ValueError("s_q * h_q must be a multiple of 16")
    if softmax_scale is None:
        softmax_scale = MLA_D_QK ** -0.5
    if out is None:
        out = torch.empty((bsz, s_q, h_q, MLA_D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((bsz, h_q, s_q), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = gqa_mla_decode(q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(), cache_seqlens.data_ptr(),
                            float(softmax_scale), out.data_ptr(), lse.data_ptr() if lse is not None else None, bsz,
                            s_q, h_q, int(kv_cache.shape[1]), int(kv_cache.shape[0]), int(block_table.shape[1]),
                            stream.cuda_stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_mla_decode")
    return out, lse
