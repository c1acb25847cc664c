"""Run the float64 oracle over many sequences on all host cores.

TEST INFRASTRUCTURE. Only the test suite and ``bench.py``'s CPU-baseline /
reference leg may use this module; the CUDA library never does.

The work is split by sequence. Each worker process evaluates
``gqa_paged_decode_oracle`` (unchanged) on a sub-problem that holds only its
sequences: their query rows, the K/V pages they name, copied out in token
order, and a CSR table whose page ids are simply 0, 1, 2, ... over that copy.
Renumbering pages does not change what the oracle computes: it gathers the
same rows in the same order, so every float64 operation is the same and the
rows come back bit-identical to a single-process run (the page-relabelling pin
in ``tests/test_oracle.py`` checks exactly that property of the oracle).

Workers are started with the ``spawn`` method, so this is safe to call after
CUDA has been initialised in the parent, and each worker is limited to one BLAS
/ OpenMP thread: ``cores`` below is the number of threads doing oracle work.
The sub-problems are sent to the workers before any timing starts; a timed
round then runs every worker's share once, and its wall time is that of the
slowest worker plus the return of the (small) results.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time
from typing import List, Optional, Sequence, Tuple

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - not Linux
        return os.cpu_count() or 1


def _bits(t) -> np.ndarray:
    """Raw 16-bit payload of a bf16 CPU tensor (sent as plain uint16)."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _share_plan(lens: Sequence[int], seqs: Sequence[int], workers: int) -> List[List[int]]:
    """Sequences per worker, balanced by token count (longest first, to the lightest worker)."""
    shares: List[List[int]] = [[] for _ in range(workers)]
    load = [0] * workers
    for b in sorted(seqs, key=lambda b: -int(lens[b])):
        i = int(np.argmin(load))
        shares[i].append(b)
        load[i] += max(1, int(lens[b]))
    return [s for s in shares if s]


def _sub_problem(q, k_cache, v_cache, indptr: np.ndarray, indices: np.ndarray, seqs: Sequence[int]):
    """Query rows, K/V rows (token order) and a 0..n-1 page table for `seqs`."""
    import torch
    lens = [int(indptr[b + 1] - indptr[b]) for b in seqs]
    sub_indptr = np.zeros(len(seqs) + 1, dtype=np.int32)
    sub_indptr[1:] = np.cumsum(lens)
    pages = np.concatenate([indices[int(indptr[b]):int(indptr[b + 1])] for b in seqs]) if sum(lens) else \
        np.zeros(0, dtype=np.int64)
    sel = torch.as_tensor(pages.astype(np.int64))
    k = k_cache.index_select(0, sel) if len(pages) else k_cache[:0]
    v = v_cache.index_select(0, sel) if len(pages) else v_cache[:0]
    qs = q.index_select(0, torch.as_tensor(np.asarray(seqs, dtype=np.int64)))
    return {"q": _bits(qs), "k": _bits(k), "v": _bits(v), "q_shape": tuple(qs.shape), "kv_shape": tuple(k.shape),
            "indptr": sub_indptr, "seqs": list(seqs)}


def _worker(conn, sm_scale: float) -> None:
    """Receive one sub-problem, then answer every 'go' with the oracle's rows for it."""
    import torch
    torch.set_num_threads(1)
    from oracle.oracle import gqa_paged_decode_oracle

    job = conn.recv()

    def as_bf16(bits, shape):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(shape)

    q = as_bf16(job["q"], job["q_shape"])
    k = as_bf16(job["k"], job["kv_shape"]) if job["k"].size else torch.zeros((1,) + job["kv_shape"][1:],
                                                                             dtype=torch.bfloat16)
    v = as_bf16(job["v"], job["kv_shape"]) if job["v"].size else torch.zeros_like(k)
    indptr = torch.from_numpy(job["indptr"])
    indices = torch.arange(int(job["indptr"][-1]), dtype=torch.int32)
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg != "go":
            break
        t0 = time.perf_counter()
        out, lse = gqa_paged_decode_oracle(q, k, v, indptr, indices, sm_scale)
        conn.send((out, lse, time.perf_counter() - t0))
    conn.close()


class OraclePool:
    """Worker processes each holding a share of one workload's sequences.

    ``run()`` evaluates every share once (all workers at the same time) and
    returns float64 (O [B, 32, 128], lse [B, 32]) with rows outside ``seqs``
    left NaN, plus the round's wall time in seconds.
    """

    def __init__(self, q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale: float,
                 seqs: Optional[Sequence[int]] = None, workers: Optional[int] = None):
        indptr = np.asarray(kv_indptr.numpy() if hasattr(kv_indptr, "numpy") else kv_indptr, dtype=np.int64)
        indices = np.asarray(kv_indices.numpy() if hasattr(kv_indices, "numpy") else kv_indices, dtype=np.int64)
        self.batch = int(indptr.shape[0] - 1)
        lens = [int(indptr[b + 1] - indptr[b]) for b in range(self.batch)]
        self.seqs = list(range(self.batch)) if seqs is None else [int(b) for b in seqs]
        self.tokens = sum(lens[b] for b in self.seqs)
        n = max(1, min(workers or host_cores(), len(self.seqs) or 1))
        self.shares = _share_plan(lens, self.seqs, n)
        self.cores = len(self.shares)
        ctx = mp.get_context("spawn")
        self._procs, self._conns = [], []
        # A spawned worker imports numpy (and its BLAS) while it unpickles its
        # target, before any of its own code runs, so the one-thread limit has
        # to be in the environment it starts with.
        saved = {var: os.environ.get(var) for var in _THREAD_VARS}
        try:
            for var in _THREAD_VARS:
                os.environ[var] = "1"
            for share in self.shares:
                parent, child = ctx.Pipe()
                p = ctx.Process(target=_worker, args=(child, float(sm_scale)), daemon=True)
                p.start()
                child.close()
                self._procs.append(p)
                self._conns.append(parent)
            for var, val in saved.items():
                if val is None:
                    os.environ.pop(var, None)
                else:
                    os.environ[var] = val
            for conn, share in zip(self._conns, self.shares):
                conn.send(_sub_problem(q, k_cache, v_cache, indptr, indices, share))
            for conn in self._conns:
                if conn.recv() != "ready":
                    raise RuntimeError("oracle worker failed to start")
        except BaseException:
            for var, val in saved.items():
                if val is None:
                    os.environ.pop(var, None)
                else:
                    os.environ[var] = val
            self.close()
            raise

    def run(self) -> Tuple[np.ndarray, np.ndarray, float]:
        out = np.full((self.batch, 32, 128), np.nan)
        lse = np.full((self.batch, 32), np.nan)
        t0 = time.perf_counter()
        for conn in self._conns:
            conn.send("go")
        for conn, share in zip(self._conns, self.shares):
            o, l, _ = conn.recv()
            out[share] = o
            lse[share] = l
        return out, lse, time.perf_counter() - t0

    def close(self) -> None:
        for conn in self._conns:
            try:
                conn.send("stop")
                conn.close()
            except (OSError, BrokenPipeError):
                pass
        for p in self._procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
                p.join(timeout=5)
        self._procs, self._conns = [], []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


def gqa_paged_decode_oracle_parallel(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale: float,
                                     seqs: Optional[Sequence[int]] = None, workers: Optional[int] = None):
    """``gqa_paged_decode_oracle`` evaluated across worker processes (same rows, same NaN convention)."""
    with OraclePool(q, k_cache, v_cache, kv_indptr, kv_indices, sm_scale, seqs=seqs, workers=workers) as pool:
        out, lse, _ = pool.run()
    return out, lse
