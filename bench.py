"""Benchmark of the GB300 paged GQA decode library (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload large] [--no-workloads] [--no-cpu-baseline]

One step is one full ``gqa_paged_decode`` call (decode kernel + LSE merge
kernel) over one batch of the workload, inputs resident in HBM. Counted bytes
per call: 2048 B per cached token (K and V rows of all 4 KV heads) plus, per
sequence, 8192 B of q, 8192 B of out and 128 B of lse. ``value`` is those bytes
over the device time of the K timed steps (CUDA events on the launching
stream; between steps, outside the events, a 256 MB write and a 256 MB read
flush the L2).

``--impl reference`` times the float64 CPU oracle instead (bounded samples of
the same workload on the host cores); only rank 0 runs it.
With N > 1 (torchrun, one rank per GPU) every rank runs its own replica of the
workload (weak scaling, no collective on the data path); the step time is the
max over ranks and ``value`` counts the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_gqa_split_gb300 import _lib  # noqa: E402
from paged_kv_gqa_split_gb300 import workloads as wl  # noqa: E402

METRIC = "paged GQA decode: µs/batch and achieved HBM GB/s (% of GB300 peak)"
WORKLOAD_TEXT = {
    "tiny": "tiny: batch 5, h32/kv4/d128/ps1 bf16, lens U[1,256], sequence 2 empty, pool = sum(lens), randperm pages",
    "mid": "mid batch: batch 64, h32/kv4/d128/ps1 bf16, lens U[512,4096], pool = sum(lens), randperm pages",
    "long": "long context: batch 1, one sequence of 131072 tokens, h32/kv4/d128/ps1 bf16, randperm pages",
    "large": ("large ragged batch: batch 256, h32/kv4/d128/ps1 bf16, lens U[1024,8192], pool 1.25x sum(lens) "
              "N(0,1), pages sampled without replacement"),
    "skewed": ("skewed batch: batch 128, h32/kv4/d128/ps1 bf16, 115 lens U[64,512] + 13 lens U[32768,65536], "
               "pool 2x sum(lens), q ~ 3 N(0,1)"),
}
FLUSH_BYTES = 256 << 20
TABLE_MIN_STEPS, TABLE_MIN_WARMUP = 50, 10
FALLBACK_HBM_GBS = 6800.0


def counted_bytes(lens) -> int:
    return 2048 * sum(lens) + (8192 + 8192 + 128) * len(lens)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity with one rank)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(bytes_per_rank: int, step_ms_max: float, world: int) -> float:
    """Whole-job GB/s of N replicas: every rank's bytes over the slowest rank's step time."""
    return world * bytes_per_rank / (step_ms_max * 1e-3) / 1e9


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("gqa_decode_lsu.cu", "gqa_common.cuh", "gqa_ptx.cuh", "gqa_plan.h"):
        with open(os.path.join(ROOT, "paged_kv_gqa_split_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, total_tokens: int):
    """DRAM bytes per decode launch from the committed ncu summary, scaled to this
    workload's token count, or None if the kernel changed since the capture."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return None
    if doc.get("kernel_hash") != kernel_source_hash():
        return None
    caps = doc.get("captures", {})
    rec = caps.get(workload) or (next(iter(caps.values())) if caps else None)
    if rec is None:
        return None
    # a capture of another workload is scaled by tokens: K/V rows dominate the traffic
    return float(rec["dram_bytes_per_launch"]) * total_tokens / float(rec["total_tokens"])


# ------------------------------------------------------------- our GPU arm
# GPU-side spin before each timed step (~150 us at 2 GHz): the host enqueues the
# step's launches while the GPU spins, so the events time GPU work, not host
# latency between the start event and the first launch.
HOST_LEAD_CYCLES = 300_000


class L2Flush:
    """Evicts the L2 between timed steps: a 256 MB write (more than the 126-129 MB
    L2), then a 256 MB read of a second buffer, so that the dirty lines of the
    write are written back before the timed region and do not compete with it."""

    def __init__(self, device):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def time_steps(call, steps: int, stream, flush, before=None):
    """Per-step device time (ms) of `call` with CUDA events on `stream`; L2 is flushed
    between steps outside the events."""
    times = []
    for i in range(steps):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        if before is not None:
            before(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def bench_workload_gpu(w, device, steps, warmup, world, with_hooks=True):
    g = w.to(device)
    out = torch.empty_like(g.q)
    lse = torch.empty((w.batch, 32), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)

    def call():
        _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale, out=out, lse=lse, stream=stream)

    for _ in range(warmup):
        call()
    launches = _lib.gqa_paged_decode_last_launch_count()
    torch.cuda.synchronize()
    barrier(world, device)
    t_wall0 = time.perf_counter()
    step_ms = time_steps(call, steps, stream, flush)
    barrier(world, device)
    wall = time.perf_counter() - t_wall0

    dec_ms = None
    if with_hooks:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:  # torch creates the underlying cudaEvent_t on first record
            a.record(stream)
            b.record(stream)

        def hook(i):
            _lib.gqa_paged_decode_set_profile_events(evs[i][0].cuda_event, evs[i][1].cuda_event)

        try:
            time_steps(call, steps, stream, flush, before=hook)
        finally:
            _lib.gqa_paged_decode_set_profile_events(None, None)
        dec_ms = [a.elapsed_time(b) for a, b in evs]
    warm_ms = None
    if with_hooks:  # the same calls with L2 left warm between steps (inputs smaller than L2 stay resident)
        warm_ms = time_steps(call, steps, stream, lambda: None)
    del flush
    return {"step_ms": step_ms, "decode_ms": dec_ms, "warm_ms": warm_ms, "wall_s": wall, "gpu": g, "out": out,
            "lse": lse, "launches_per_call": launches}


def bench_e2e(w, device, steps, warmup):
    """Same metric through the public API with host buffers: pinned host inputs are
    copied to the device, the call runs, out/lse come back, all inside the events."""
    host = [w.q.pin_memory(), w.k_cache.pin_memory(), w.v_cache.pin_memory(), w.kv_indptr.pin_memory(),
            w.kv_indices.pin_memory()]
    dev = [torch.empty_like(t, device=device) for t in host]
    out_h = torch.empty_like(host[0]).pin_memory()
    lse_h = torch.empty((w.batch, 32), dtype=torch.float32).pin_memory()
    out_d = torch.empty_like(dev[0])
    lse_d = torch.empty((w.batch, 32), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    def call():
        for hd, dd in zip(host, dev):
            dd.copy_(hd, non_blocking=True)
        _lib.run(dev[0], dev[1], dev[2], dev[3], dev[4], w.sm_scale, out=out_d, lse=lse_d, stream=stream)
        out_h.copy_(out_d, non_blocking=True)
        lse_h.copy_(lse_d, non_blocking=True)

    def copies():
        for hd, dd in zip(host, dev):
            dd.copy_(hd, non_blocking=True)

    for _ in range(max(1, warmup)):
        call()
    torch.cuda.synchronize()
    ms = time_steps(call, steps, stream, flush)
    copy_ms = time_steps(copies, steps, stream, flush)  # the same host-to-device copies alone
    del flush, dev
    return ms, copy_ms, h2d, d2h


# ------------------------------------------------------------- KV append
def bench_append(device, steps, warmup, step_tokens, peak):
    """KV-cache append: a bulk append of 262,144 tokens into a 1 Mi-page pool
    (2 KB read + 2 KB written per token) and one decode step's append of
    `step_tokens` tokens. Same timing method as the decode line."""
    g = torch.Generator(device=device).manual_seed(7)
    num_pages, bulk = 1 << 20, 1 << 18
    k = torch.empty(num_pages, 1, 4, 128, dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    kn = torch.randn(bulk, 4, 128, generator=g, device=device).to(torch.bfloat16)
    vn = torch.randn(bulk, 4, 128, generator=g, device=device).to(torch.bfloat16)
    slots = torch.randperm(num_pages, generator=g, device=device)[:bulk].to(torch.int32)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    res = {}
    for name, n in (("bulk", bulk), ("step", step_tokens)):
        def call(n=n):
            _lib.kv_append(kn[:n], vn[:n], slots[:n], k, v, stream=stream)
        for _ in range(warmup):
            call()
        ms = statistics.median(time_steps(call, steps, stream, flush))
        gbs = 4096 * n / (ms * 1e-3) / 1e9
        res[name] = {"tokens": n, "us": ms * 1e3, "gbs": gbs, "frac_of_peak": gbs / peak}
    del k, v, kn, vn, slots, flush
    return res


# ---------------------------------------------------- selected-token decode
def bench_sparse(device, steps, warmup, peak):
    """Selected-token decode of the sparse workload (128 rows x 2048 selected
    positions, blocks of 64): µs per call and GB/s of the K/V rows of the used
    columns (2048 B each) plus 16,512 B of q, O and LSE per row. Same timing
    method as the decode line."""
    w = wl.make_sparse_config()
    # every non-negative position of this generator is below its request's
    # length and inside its mapped blocks, so it is a used column
    used = int((w.logical_indices >= 0).sum())
    g = w.to(device)
    out = torch.empty_like(g.q)
    lse = torch.empty((w.rows, 32), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)

    def call():
        _lib.sparse_run(g.q, g.k_cache, g.v_cache, g.logical_indices, g.block_table, g.token_to_req, w.sm_scale,
                        out=out, lse=lse, stream=stream)
    for _ in range(warmup):
        call()
    ms = statistics.median(time_steps(call, steps, stream, flush))
    b = 2048 * used + 16512 * w.rows
    res = {"rows": w.rows, "topk": w.topk, "page_size": w.page_size, "used_columns": used,
           "us_per_batch": ms * 1e3, "gbs": b / (ms * 1e-3) / 1e9, "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
           "counted_bytes": b, "launches_per_call": 3}
    del g, out, lse, flush
    return res


# ------------------------------------------------------------ FP8 KV cache
def bench_fp8(w, g, device, steps, warmup, peak):
    """Decode of workload w over an FP8 copy of its cache (528-byte rows: 4 KV
    heads x 128 e4m3 codes + 4 fp32 scales, quantized on the device from the
    bf16 cache already in HBM, outside the timed region). Counted bytes: 1056 B
    per token (K and V rows) + 16,512 B of q, O and LSE per sequence. Times every
    compiled FP8 variant (16-token stages in rings of 2, 3 and 4; 32-token stages in
    a ring of 2) and the default."""
    k8 = wl.quantize_fp8_rows(g.k_cache)
    v8 = wl.quantize_fp8_rows(g.v_cache)
    out = torch.empty_like(g.q)
    lse = torch.empty((w.batch, 32), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)
    b = 1056 * w.total_tokens + 16512 * w.batch
    res = {"workload": w.name, "counted_bytes": b, "bytes_vs_bf16": b / counted_bytes(w.lens)}
    variants = [("stages_2", (0, 0, 4, 16, 2, _lib.GATHER_LSU_F8)), ("stages_3", (0, 0, 4, 16, 3, _lib.GATHER_LSU_F8)),
                ("stages_4", (0, 0, 4, 16, 4, _lib.GATHER_LSU_F8)), ("stage32", (0, 0, 4, 32, 2, _lib.GATHER_LSU_F8)),
                ("default", (0, 0, 0, 0, 0, 0))]
    for key, tuning in variants:
        if _lib.gqa_paged_decode_set_tuning(*tuning) != 0:
            raise RuntimeError(f"FP8 tuning {tuning} rejected")

        def call():
            _lib.run_fp8(g.q, k8, v8, g.kv_indptr, g.kv_indices, w.sm_scale, out=out, lse=lse, stream=stream)
        for _ in range(warmup):
            call()
        ms = statistics.median(time_steps(call, steps, stream, flush))
        res[key] = {"us_per_batch": ms * 1e3, "gbs": b / (ms * 1e-3) / 1e9,
                    "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak}
    _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
    res.update(res["default"])
    del k8, v8, out, lse, flush
    return res


# ------------------------------------------- mma.sync against CUDA cores
def bench_cuda_cores(names, device, steps, warmup, peak, variant_only=False):
    """The default decode (both contractions on mma.sync) against the same
    pipeline with the contractions on the CUDA cores (gather 3), per workload:
    µs per call and of the decode kernel alone, same timing method as the main
    line. variant_only: time the CUDA-core variant only (for a profiler run)."""
    res = {}
    for name in names:
        w = wl.make_config(name)
        cb = counted_bytes(w.lens)
        row = {}
        for label, gather in (() if variant_only else (("mma_sync", 0),)) + (("cuda_cores", 3),):
            assert _lib.gqa_paged_decode_set_tuning(0, 0, 4, 16, 2, gather) == 0
            try:
                r = bench_workload_gpu(w, device, steps, warmup, 1, with_hooks=not variant_only)
            finally:
                _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
            ms = statistics.median(r["step_ms"])
            row[label] = {"us_per_batch": ms * 1e3, "gbs": cb / (ms * 1e-3) / 1e9,
                          "frac_of_peak": cb / (ms * 1e-3) / 1e9 / peak}
            if r["decode_ms"]:
                dm = statistics.median(r["decode_ms"])
                row[label]["decode_kernel_us"] = dm * 1e3
                row[label]["decode_frac_of_peak"] = cb / (dm * 1e-3) / 1e9 / peak
            del r
        if "mma_sync" in row:
            row["cuda_cores_over_mma_sync"] = row["cuda_cores"]["us_per_batch"] / row["mma_sync"]["us_per_batch"]
        res[name] = row
    return res


# ------------------------------------------------------------ MLA decode
def bench_mla_heads(device, steps, warmup, peak, heads=(16, 32, 64, 128)):
    """Both MLA kernels on the MLA batch's lengths and cache with h_q query heads each:
    where the tensor-memory kernel overtakes the mma.sync one."""
    res = {}
    for h in heads:
        w = wl.make_mla_config(h_q=h)
        g = w.to(device)
        rows = int(w.q.shape[1] * w.q.shape[2])
        out = torch.empty((w.batch, w.q.shape[1], w.q.shape[2], 512), dtype=torch.bfloat16, device=device)
        lse = torch.empty((w.batch, w.q.shape[2], w.q.shape[1]), dtype=torch.float32, device=device)
        stream = torch.cuda.current_stream(device)
        flush = L2Flush(device)
        b = 1152 * w.total_tokens + (1152 + 1024 + 4) * rows * w.batch
        r = {"counted_bytes": b}
        for kernel, key in ((1, "tensor_memory"), (3, "mma_sync")):
            _lib.gqa_mla_set_tuning(kernel)
            try:
                def call():
                    _lib.mla_run(g.q, g.kv_cache, g.block_table, g.cache_seqlens, w.softmax_scale, out=out, lse=lse,
                                 stream=stream)
                for _ in range(warmup):
                    call()
                ms = statistics.median(time_steps(call, steps, stream, flush))
            finally:
                _lib.gqa_mla_set_tuning(0)
            r[key] = {"us_per_batch": ms * 1e3, "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak}
        r["default"] = "tensor_memory" if rows % 32 == 0 else "mma_sync"
        res[f"h_q={h}"] = r
        del g, out, lse, flush
    return res


def bench_mla(device, steps, warmup, peak, wide: bool = False):
    """Dense MLA decode of the MLA workload (128 sequences of U[1024, 8192]
    cached tokens, 16 query heads, blocks of 64; with `wide`, 64 query heads on
    the same lengths): µs per call and GB/s of the counted bytes, 1152 B of
    latent row per cached token plus q (1152 B), O (1024 B) and LSE (4 B) per
    query row. FLOPs: 2 * (576 + 512) per (token, query row). Both kernels are
    timed; the line's figures are the default one's."""
    w = wl.make_mla_config(wide)
    g = w.to(device)
    rows = int(w.q.shape[1] * w.q.shape[2])
    out = torch.empty((w.batch, w.q.shape[1], w.q.shape[2], 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.batch, w.q.shape[2], w.q.shape[1]), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)

    def call():
        _lib.mla_run(g.q, g.kv_cache, g.block_table, g.cache_seqlens, w.softmax_scale, out=out, lse=lse,
                     stream=stream)
    t = w.total_tokens
    b = 1152 * t + (1152 + 1024 + 4) * rows * w.batch
    flops = 2 * (576 + 512) * t * rows

    def timed(kernel):
        _lib.gqa_mla_set_tuning(kernel)
        try:
            for _ in range(warmup):
                call()
            ms = statistics.median(time_steps(call, steps, stream, flush))
        finally:
            _lib.gqa_mla_set_tuning(0)
        return {"us_per_batch": ms * 1e3, "gbs": b / (ms * 1e-3) / 1e9, "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                "tflops": flops / (ms * 1e-3) / 1e12}
    tc = timed(1)   # the tensor-memory (tcgen05) kernel: 16- or 64-row pieces
    mma = timed(3)  # the mma.sync kernel: 16-row pieces
    default_tc = rows % 32 == 0 and w.page_size % 32 == 0
    d = tc if default_tc else mma
    res = {"batch": w.batch, "h_q": int(w.q.shape[2]), "s_q": int(w.q.shape[1]), "page_size": w.page_size,
           "total_tokens": t, "us_per_batch": d["us_per_batch"], "gbs": d["gbs"], "frac_of_peak": d["frac_of_peak"],
           "tflops": d["tflops"], "counted_bytes": b,
           "kernel": ("tensor memory, %d-row pieces" % (64 if rows % 64 == 0 else 32)) if default_tc
           else "mma.sync, 3-stage ring",
           "tensor_memory_kernel": dict(tc, launches_per_call=3), "mma_sync_kernel": dict(mma, launches_per_call=4)}
    del g, out, lse, flush
    return res


# -------------------------------------------------------------- CPU oracle
# CPU work (core-seconds) the oracle baseline aims for: enough repeated rounds
# over the workload that the median round is stable, bounded to a few seconds of
# wall time on the host's cores.
ORACLE_TARGET_CPU_S = 12.0
ORACLE_MAX_ROUNDS = 20
# rounds of the oracle per workload-table row (median reported)
TABLE_ORACLE_ROUNDS = 3


def oracle_rounds(w, rounds=None, target_cpu_s=ORACLE_TARGET_CPU_S):
    """The float64 oracle over every sequence of `w`, on all host cores (one worker
    process per core, one BLAS thread each). Runs `rounds` rounds (default: enough
    for about target_cpu_s core-seconds) and returns the first round's (O, lse),
    the per-round wall times and the worker count."""
    from oracle.pool import OraclePool
    with OraclePool(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale) as pool:
        o_ref, l_ref, first = pool.run()
        if rounds is None:
            rounds = max(1, min(ORACLE_MAX_ROUNDS, math.ceil(target_cpu_s / max(first * pool.cores, 1e-3))))
        times = [first] + [pool.run()[2] for _ in range(rounds - 1)]
        return o_ref, l_ref, times, pool.cores


def parity_summary(w, out, lse, o_ref, l_ref):
    """Element-wise comparison of the GPU's (out, lse) with the oracle over every sequence."""
    import numpy as np
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    fin = np.isfinite(l_ref)
    o_err = float(np.abs(o - o_ref).max())
    l_err = float(np.abs(l[fin] - l_ref[fin]).max()) if fin.any() else 0.0
    ok = bool(np.all(np.abs(o - o_ref) <= 2e-2 + 2e-2 * np.abs(o_ref)) and l_err <= 1e-3 and
              np.array_equal(np.isneginf(l), np.isneginf(l_ref)))
    return {"sequences": w.batch, "tokens": w.total_tokens, "max_abs_dO": o_err, "max_abs_dlse": l_err,
            "within_tolerance": ok}


def cpu_baseline(w, out=None, lse=None):
    """The oracle timed on the host's cores over the whole workload (median of
    repeated rounds). With the GPU's (out, lse) of the timed run, the first round
    also gives the run's parity figures over every sequence."""
    from oracle.pool import host_cores
    o_ref, l_ref, times, cores = oracle_rounds(w)
    dt = statistics.median(times)
    gbs = counted_bytes(w.lens) / dt / 1e9
    base = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"all {w.batch} sequences ({w.total_tokens} tokens) of the {w.name} workload per round, "
                      f"float64 NumPy oracle in {cores} worker processes (one BLAS thread each); "
                      f"median of {len(times)} rounds, {dt:.3f} s per round",
            "host_cores_available": host_cores(), "threads_per_worker": 1,
            "rounds_s": [round(t, 4) for t in times]}
    parity = parity_summary(w, out, lse, o_ref, l_ref) if out is not None else None
    return base, parity


# ------------------------------------------------------------- variant sweep
SWEEP_VARIANTS = [
    # (num_ctas, min_units_per_cta, heads_per_cta, tile, stages, gather[, fused_merge_max_splits, tier2_ctas,
    # tier2_permille, tier2_min_units]): gather 0 = cp.async, 1 = TMA bulk; 0 = default; fused-merge threshold
    # -1 = every split sequence to the merge kernel; tier2_ctas -1 = one tier
    (0, 0, 4, 16, 2, 0), (0, 0, 4, 16, 3, 0), (0, 0, 2, 16, 2, 0), (0, 0, 1, 16, 2, 0), (0, 0, 4, 16, 5, 1),
    (0, 0, 4, 16, 2, 0, 0, -1), (0, 0, 4, 16, 3, 0, 0, -1),
    (0, 0, 4, 16, 2, 0, 0, 912), (0, 0, 4, 16, 2, 0, 0, 3648),
    (0, 0, 4, 16, 2, 0, 0, 0, 50), (0, 0, 4, 16, 2, 0, 0, 0, 150), (0, 0, 4, 16, 2, 0, 0, 0, 200),
    (0, 0, 4, 16, 2, 0, 0, 0, 0, 16), (0, 0, 4, 16, 2, 0, 0, 0, 0, 32), (0, 0, 4, 16, 2, 0, 0, 0, 0, 128),
    (0, 0, 4, 16, 2, 0, 0, 0, 150, 32), (0, 0, 4, 16, 2, 0, 0, 3648, 150, 32),
    (0, 0, 4, 16, 2, 0, 4), (0, 0, 4, 16, 2, 0, 16),
]


def sweep(device, steps, warmup, names):
    """Median µs per call of every decode variant on the named workloads (same timing
    method as the main line); prints one JSON line per (workload, variant)."""
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)
    for name in names:
        w = wl.make_config(name)
        g = w.to(device)
        out = torch.empty_like(g.q)
        lse = torch.empty((w.batch, 32), dtype=torch.float32, device=device)
        cb = counted_bytes(w.lens)
        for v in SWEEP_VARIANTS:
            if _lib.gqa_paged_decode_set_tuning(*v) != 0:
                continue

            def call():
                _lib.run(g.q, g.k_cache, g.v_cache, g.kv_indptr, g.kv_indices, w.sm_scale, out=out, lse=lse,
                         stream=stream)

            for _ in range(warmup):
                call()
            ms = statistics.median(time_steps(call, steps, stream, flush))
            print(json.dumps({"sweep": name, "variant": dict(zip(
                ["num_ctas", "min_units_per_cta", "heads_per_cta", "tile", "stages", "gather",
                 "fused_merge_max_splits", "tier2_ctas", "tier2_permille", "tier2_min_units"],
                tuple(v) + (0,) * (10 - len(v)))),
                "us_per_batch": ms * 1e3, "gbs": cb / (ms * 1e-3) / 1e9}), flush=True)
        _lib.gqa_paged_decode_set_tuning(0, 0, 0, 0, 0, 0)
        del g, out, lse


# ---------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(wl.CONFIGS), default="large")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="time every decode variant instead of the contract line")
    ap.add_argument("--merge-mode", type=int, choices=[0, 1], default=0,
                    help="0: decode grid + merge kernel (default); 1: one-wave decode with the merge inside the kernel")
    ap.add_argument("--only", choices=["fp8", "sparse", "mla", "mla-wide", "mla-heads", "cuda-cores"], default=None,
                    help="time only the FP8-cache decode of --workload, or only the selected-token decode, and "
                         "print its result (for profiling a small case)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)

    world, rank, local = dist_info()
    if args.impl == "reference":
        return main_reference(args, world, rank, warmup)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from paged_kv_gqa_split_gb300.build import build
    if rank == 0 or world == 1:
        build()
    barrier(world, device)
    _lib.load()
    if _lib.gqa_paged_decode_set_merge_mode(args.merge_mode) != 0:
        raise SystemExit("bad --merge-mode")

    if args.sweep:
        sweep(device, args.steps, warmup, ["tiny", "mid", "long", "large", "skewed"])
        return
    if args.only is not None:
        peak, _ = hbm_peak()
        if args.only == "fp8":
            w = wl.make_config(args.workload)
            res = bench_fp8(w, w.to(device), device, args.steps, warmup, peak)
        elif args.only == "mla":
            res = bench_mla(device, args.steps, warmup, peak)
        elif args.only == "mla-wide":
            res = bench_mla(device, args.steps, warmup, peak, wide=True)
        elif args.only == "mla-heads":
            res = bench_mla_heads(device, args.steps, warmup, peak)
        elif args.only == "cuda-cores":
            res = bench_cuda_cores([args.workload], device, args.steps, warmup, peak, variant_only=True)
        else:
            res = bench_sparse(device, args.steps, warmup, peak)
        if rank == 0:
            print(json.dumps({"only": args.only, "result": res}), flush=True)
        return

    peak, peak_kind = hbm_peak()
    w = wl.make_config(args.workload)
    cb = counted_bytes(w.lens)
    with ClockSampler(local) as clk:
        r = bench_workload_gpu(w, device, args.steps, warmup, world)
    step_ms = statistics.median(r["step_ms"])
    step_ms_max = max_over_ranks(step_ms, world, device)
    dec_ms = statistics.median(r["decode_ms"])
    value = replica_value(cb, step_ms_max, world)
    achieved = cb / (dec_ms * 1e-3) / 1e9

    # the GPU result of the timed run, for the parity check of the CPU-baseline leg
    run_out, run_lse = r["out"].cpu(), r["lse"].cpu()
    step_ms_mean = statistics.mean(r["step_ms"])
    launches_per_call = r["launches_per_call"]
    del r

    e2e = None
    if not args.no_e2e:
        ms, copy_ms, h2d, d2h = bench_e2e(w, device, max(3, args.steps // 4), 1)
        e_ms = max_over_ranks(statistics.median(ms), world, device)
        c_ms = statistics.median(copy_ms)
        e2e = {"value": world * cb / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "h2d_gbs": h2d / (c_ms * 1e-3) / 1e9, "h2d_ms": c_ms,
               "note": "each step copies the whole K/V pool (pinned host -> HBM), runs the call and reads "
                       "out/lse back; h2d_gbs times the same copies alone in the same run"}

    table = {}
    if not args.no_workloads:
        for name in ["tiny", "mid", "long", "large", "skewed"]:
            ww = w if name == args.workload else wl.make_config(name)
            # at least 10 warm-up and 50 timed calls per workload; the table reports their median
            rr = bench_workload_gpu(ww, device, max(args.steps, TABLE_MIN_STEPS), max(warmup, TABLE_MIN_WARMUP),
                                    world)
            ms = statistics.median(rr["step_ms"])
            dm = statistics.median(rr["decode_ms"])
            b = counted_bytes(ww.lens)
            table[name] = {"us_per_batch": ms * 1e3, "gbs": b / (ms * 1e-3) / 1e9,
                           "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                           "us_per_batch_mean": statistics.mean(rr["step_ms"]) * 1e3,
                           "decode_kernel_us": dm * 1e3, "launches_per_call": rr["launches_per_call"],
                           "batch": ww.batch, "total_tokens": ww.total_tokens,
                           "counted_bytes": b, "us_per_batch_l2_warm": statistics.median(rr["warm_ms"]) * 1e3}
            del rr
            if rank == 0 and not args.no_cpu_baseline and name != args.workload:
                # the oracle over the same batch on the host's cores (the headline
                # workload's figure comes from the CPU-baseline leg below)
                _, _, times, cores = oracle_rounds(ww, rounds=TABLE_ORACLE_ROUNDS)
                table[name].update({"oracle_s_per_batch": statistics.median(times), "oracle_cores": cores})
            if ww is not w:
                del ww

    append = sparse = fp8 = mla = mla_wide = cuda_cores = None
    if not args.no_workloads:
        cuda_cores = bench_cuda_cores(["mid", "large"], device, args.steps, warmup, peak)
        append = bench_append(device, args.steps, warmup, w.batch, peak)
        sparse = bench_sparse(device, args.steps, warmup, peak)
        fp8 = bench_fp8(w, w.to(device), device, args.steps, warmup, peak)
        mla = bench_mla(device, args.steps, warmup, peak)
        mla_wide = bench_mla(device, args.steps, warmup, peak, wide=True)

    cpu, parity = None, None
    if rank == 0 and not args.no_cpu_baseline:
        cpu, parity = cpu_baseline(w, run_out, run_lse)
        if args.workload in table:
            table[args.workload].update({"oracle_s_per_batch": statistics.median(cpu["rounds_s"]),
                                         "oracle_cores": cpu["cores"]})

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    clocks = clk.summary()
    traffic = ncu_traffic(args.workload, w.total_tokens)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": warmup,
        "ms_per_step": step_ms_max,
        "ms_per_step_mean": step_ms_mean,
        "timing": "median of the timed steps (CUDA events; ms_per_step_mean is their mean)",
        "us_per_batch": step_ms_max * 1e3,
        "frac_of_peak": value / world / peak,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded torch.Generator, CPU-drawn, copied to HBM before timing)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "batch": w.batch, "total_tokens": w.total_tokens,
                   "num_pages": w.num_pages, "counted_bytes_per_step": cb,
                   "l2": "flushed between steps (256 MB device write, then 256 MB read; outside the timed events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "gqa_decode_lsu_kernel", "peak_kind": f"{peak_kind} (hbm_gbs)",
                     "algorithmic_bytes_per_launch": cb},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_call * args.steps,
        "launches_per_call": launches_per_call,
        "clocks": clocks,
        "parity": parity,
        "workloads": table,
        "kv_append": append,
        "sparse_decode": sparse,
        "fp8_decode": fp8,
        "mla_decode": mla,
        "mla_decode_64_heads": mla_wide,
        "cuda_core_variant": cuda_cores,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main_reference(args, world, rank, warmup):
    """The float64 oracle on the host's cores: each step evaluates the whole
    workload once across the worker pool (one process per core)."""
    if rank != 0:
        return
    from oracle.pool import OraclePool, host_cores
    w = wl.make_config(args.workload)
    cb = counted_bytes(w.lens)
    with OraclePool(w.q, w.k_cache, w.v_cache, w.kv_indptr, w.kv_indices, w.sm_scale) as pool:
        for _ in range(warmup):
            pool.run()
        secs = [pool.run()[2] for _ in range(args.steps)]
        cores = pool.cores
    dt = statistics.median(secs)
    value = cb / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": warmup,
        "ms_per_step": dt * 1e3,
        "ms_per_step_mean": statistics.mean(secs) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded torch.Generator)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "batch": w.batch, "total_tokens": w.total_tokens,
                   "parallelism": f"{cores} host worker processes"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": cores,
                         "host_cores_available": host_cores(), "threads_per_worker": 1,
                         "sample": f"each step: all {w.batch} sequences ({w.total_tokens} tokens) of the workload, "
                                   f"float64 NumPy oracle across {cores} worker processes; median step time"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
