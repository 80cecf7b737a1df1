#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on one GB300 per rank.

A step is one decode step of the batched GQA workload (32 requests, 32 query
heads over 8 kv heads, head_dim 128, bf16, contexts uniform in [512, 4096],
262144-slot pool, layer 2 of 4): the cache write of the 32 new K/V rows
followed by paged decode attention (split kernel + merge) through
req_to_token.  `value` is the step's algorithmic HBM bytes / step time (KV
GB/s); the line also reports decode tokens/s, the decode kernel's roofline,
the ragged-prefill TFLOP/s, the B=1 32K-context decode, an end-to-end figure
through the public API with host buffers, and the fp64 oracle timed on the
host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the workload (the path shards by request with no exchange), `value` is the
sum over ranks of the bytes divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
L2_FLUSH_BYTES = 256 << 20        # > 2x the 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--chunk", type=int, default=0, help="decode split size (0: automatic)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the prefill / long-context / e2e / cpu legs")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--decode-sweep", action="store_true",
                    help="print decode KV GB/s over batch x context (uniform contexts) and exit")
    ap.add_argument("--profile-case", choices=["decode", "long", "prefill", "prefill64", "prefill_full",
                                               "kvwrite", "prefix_shared"],
                    help="run a few untimed calls of one kernel's case (for ncu) and exit")
    return ap.parse_args()


DECODE_SWEEP = [(1, 16384), (8, 1024), (8, 4096), (8, 16384), (32, 1024), (32, 4096), (32, 16384),
                (128, 1024), (128, 4096), (256, 1024), (256, 2048), (512, 512), (512, 1024),
                (1100, 256)]


def run_decode_sweep() -> None:
    """Decode (automatic plan) over batch x uniform context, 32/8 heads, d=128,
    bf16, permuted slots; L2 flushed before each call; one JSON line per point."""
    import torch
    import paged_kv_cache_loc_gb300 as pkv
    from paged_kv_cache_loc_gb300 import build
    from paged_kv_cache_loc_gb300 import workloads as W
    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    flush = make_l2_flush(torch, dev)
    stream = torch.cuda.Stream(device=dev)
    peaks = measured_peaks()
    for batch, ctx in DECODE_SWEEP:
        tokens = batch * ctx
        size = max(65536, ((tokens + batch + 4095) // 4096) * 4096)
        case = W.make_case("sweep", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=size,
                           n_heads=32, n_kv_heads=8, head_dim=128, kv_lens=[ctx] * batch,
                           seed=batch + ctx)
        cache, q, kn, vn = W.upload(case, dev)
        pkv.kv_write(cache, 0, kn, vn)
        ws = pkv.Workspace(batch, 32, 128, max(2, -(-(152 + batch) // batch)), device=dev)
        chunk, parts = pkv.decode_plan(cache, 32, ws)
        o = torch.empty_like(q)
        with torch.cuda.stream(stream):
            ms, _ = timed(torch, stream, lambda: pkv.paged_decode(cache, 0, q, o, workspace=ws,
                                                                stream=stream), 30, 5, flush)
        st, detail = pkv.last_device_error(stream, dev)
        if st != 0:
            raise RuntimeError(f"device error word set in the sweep (detail {detail})")
        t = statistics.median(ms)
        b = decode_bytes(case)
        print(json.dumps({"batch": batch, "context": ctx, "us_per_decode": round(t * 1e3, 1),
                          "kv_gbs": round(b / (t * 1e-3) / 1e9, 1),
                          "frac_of_hbm_peak": round(b / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                          "plan": f"balanced: {parts} CTAs" if chunk == 0 else f"chunked: {chunk}"}),
              flush=True)
        del cache, q, kn, vn, ws, o, case
        torch.cuda.empty_cache()


def run_profile_case(which: str) -> None:
    """A few untimed calls of one workload, sized for an ncu capture (a few GB
    on the device at most): decode = the batched decode (98,304-slot pool),
    long = B=1 at 32,768 tokens, prefill = 4 ragged-prefill requests (prefill64:
    the same at head_dim 64; prefill_full: the whole ragged-prefill workload, ~2.2 GB),
    kvwrite = the ragged prefill's cache write (17,418 tokens), prefix_shared =
    the prefix-shared workload through the page table with its 128 shared
    pages stated."""
    import torch
    import paged_kv_cache_loc_gb300 as pkv
    from paged_kv_cache_loc_gb300 import build
    from paged_kv_cache_loc_gb300 import workloads as W
    build.build()
    torch.cuda.set_device(0)
    if which in ("decode", "long"):
        case = W.batched_decode(size=98304) if which == "decode" else W.long_decode(32768)
        cache, q, kn, vn = W.upload(case)
        pkv.kv_write(cache, case.layer_id, kn, vn)
        ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1024)
        o = torch.empty_like(q)
        for _ in range(3):
            pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws)
    elif which == "prefix_shared":
        case = W.prefix_shared_decode()
        cache, q, kn, vn = W.upload(case)
        pkv.kv_write(cache, case.layer_id, kn, vn)
        ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1024)
        o = torch.empty_like(q)
        ps = case.page_size
        table = torch.from_numpy(np.ascontiguousarray(case.req_to_token[:, ::ps] // ps)).cuda()
        for _ in range(3):
            pkv.paged_decode_pages(cache, case.layer_id, table, ps, q, o, workspace=ws,
                                   shared_pages=case.shared_prefix // ps)
    elif which in ("prefill", "prefill64", "prefill_full"):
        case = (W.ragged_prefill() if which == "prefill_full" else
                W.ragged_prefill(batch=4, size=32768, head_dim=64 if which == "prefill64" else 128))
        cache, q, kn, vn = W.upload(case)
        pkv.kv_write(cache, case.layer_id, kn, vn)
        o = torch.empty_like(q)
        ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1)   # entries longest first
        for _ in range(2):
            pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, o=o, workspace=ws)
    else:
        case = W.ragged_prefill()
        cache, q, kn, vn = W.upload(case)
        for _ in range(3):
            pkv.kv_write(cache, case.layer_id, kn, vn)
    torch.cuda.synchronize()
    st, detail = pkv.last_device_error()
    if st != 0:
        raise RuntimeError(f"device error word set ({detail})")
    print(f"profile case {which}: done")


# ---------------------------------------------------------------------------
# environment: ranks, peaks, clocks
# ---------------------------------------------------------------------------

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_config(case, world: int) -> dict:
    """The workload description both arms report (the implementation adds its plan)."""
    return {"workload": "batched GQA decode", "batch": case.batch, "n_heads": case.n_heads,
            "n_kv_heads": case.n_kv_heads, "head_dim": case.head_dim,
            "seq_lens": "uniform [512, 4096]", "total_kv_tokens": int(case.seq_lens.sum()),
            "pool_slots": case.size, "n_layers": case.n_layers, "layer_id": case.layer_id,
            "page_size": 1, "new_tokens_per_step": int(case.out_cache_loc.size),
            "parallelism": f"replicas x{world}"}


def rank_seed(rank: int) -> int:
    """Seed of a rank's copy of the workload: the same shapes on every rank
    (weak scaling), different values."""
    return 1002 + 100 * rank


def job_step_ms(torch, local_ms: float, dev) -> float:
    """The job's step time: the slowest rank's (max over ranks)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_ms
    t = torch.tensor([local_ms], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value_gbs(world: int, bytes_per_rank_step: float, job_ms: float) -> float:
    """Whole-job throughput: the bytes every rank processed per step, over the job's step time."""
    return world * bytes_per_rank_step / (job_ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        d = {}

    def pick(*keys):
        for k in keys:
            v = d.get(k)
            if isinstance(v, (int, float)) and v > 0:
                return float(v)
        return None
    hbm = pick("hbm_gbs")
    bf16 = pick("bf16_tflops")
    bf16s = pick("bf16_tflops_sustained")
    return {
        "hbm_gbs": hbm or FALLBACK_HBM_GBS,
        "hbm_source": "measured" if hbm else "fallback",
        "bf16_tflops": bf16 or FALLBACK_BF16_TFLOPS,
        "bf16_source": "measured" if bf16 else "fallback",
        "bf16_tflops_sustained": bf16s or FALLBACK_BF16_TFLOPS_SUSTAINED,
    }


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def profile_traffic(name: str, *sources: str):
    """DRAM bytes per launch from a committed ncu summary, or None if the kernel
    sources changed since it was captured (the summary records their sha256)."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_sha256")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    h = hashlib.sha256()
    for source in sources:
        h.update(open(os.path.join(ROOT, "paged_kv_cache_loc_gb300", "csrc", source), "rb").read())
    digest = h.hexdigest()
    if fields.get("source_sha256") != digest or "traffic_bytes_per_launch" not in fields:
        return None
    return float(fields["traffic_bytes_per_launch"])


# ---------------------------------------------------------------------------
# algorithmic work (the figures the rooflines use)
# ---------------------------------------------------------------------------

def decode_bytes(case) -> float:
    """K and V rows read + slot indices + q read + o written."""
    eb = case.elem_bytes
    tokens = float(case.seq_lens.sum())
    row = case.n_kv_heads * case.head_dim * eb
    return tokens * 2 * row + tokens * 4 + 2.0 * case.batch * case.n_heads * case.head_dim * eb


def kv_write_bytes(case) -> float:
    """New K and V rows read and written + write locations."""
    n = float(case.out_cache_loc.size)
    row = case.n_kv_heads * case.head_dim * case.elem_bytes
    return n * 2 * row * 2 + n * 4


def prefill_flops(case) -> float:
    """4 * d * H * (causal query-key pairs): QK^T and PV over unmasked pairs."""
    ql = case.q_lens.astype(np.float64)
    pre = case.seq_lens.astype(np.float64) - ql
    pairs = float(np.sum(ql * pre + ql * (ql + 1) / 2))
    return 4.0 * case.head_dim * case.n_heads * pairs


# ---------------------------------------------------------------------------
# the pkv arm
# ---------------------------------------------------------------------------

class DecodeStep:
    """Pre-marshalled C-ABI calls for one decode step: the fused pkv_decode_step,
    or its two halves (pkv_kv_write, then pkv_paged_decode) for per-kernel times."""

    def __init__(self, lib, cache, q, kn, vn, o, ws, layer_id, chunk, stream):
        from paged_kv_cache_loc_gb300 import _lib
        self.lib = lib
        self.c = cache.c_struct()
        self.cref = ctypes.byref(self.c)
        self.layer = layer_id
        self.k, self.v = ctypes.c_void_p(kn.data_ptr()), ctypes.c_void_p(vn.data_ptr())
        self.n_new = int(kn.shape[0])
        self.q, self.o = ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(o.data_ptr())
        self.heads = int(q.shape[1])
        self.scale = 1.0 / math.sqrt(int(q.shape[2]))
        self.chunk = chunk
        self.ws = ctypes.byref(ws.desc)
        self.s = ctypes.c_void_p(stream.cuda_stream)
        self.check = _lib.check

    def fused(self):
        self.check(self.lib.pkv_decode_step(self.cref, self.layer, self.k, self.v, self.n_new,
                                            self.q, self.o, self.heads, self.scale, self.ws,
                                            self.s), "pkv_decode_step")

    def write(self):
        self.check(self.lib.pkv_kv_write(self.cref, self.layer, self.k, self.v, self.n_new, self.s),
                   "pkv_kv_write")

    def decode(self):
        self.check(self.lib.pkv_paged_decode_chunked(self.cref, self.layer, self.q, self.o,
                                                     self.heads, self.scale, self.chunk, self.ws,
                                                     self.s), "pkv_paged_decode")


def graph_replay_ms(torch, stream, fn, steps, warmup, flush):
    """Capture fn() once in a CUDA graph on `stream` and time its replays with
    the L2 flushed before each (the flush stays outside the graph)."""
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    ms, _ = timed(torch, stream, g.replay, steps, warmup, flush)
    return ms, g


def make_l2_flush(torch, dev):
    """Evict L2 between timed steps: write a 256 MB buffer, then read another
    256 MB so that the dirty lines of the write are written back before the
    step starts (their write-backs are not charged to the measured kernel)."""
    wbuf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        wbuf.add_(1.0)
        rbuf.sum()
    return flush


def timed(torch, stream, fn, steps, warmup, flush, parts=None):
    """Run the step `warmup` times, then `steps` times with an L2 flush before
    each; CUDA events on `stream` bracket each step and each of its parts.
    The step is fn(), or the calls in `parts` one after another."""
    calls = list(parts) if parts else [fn]
    for _ in range(warmup):
        flush()
        for c in calls:
            c()
    torch.cuda.synchronize()
    ev = []
    for _ in range(steps):
        flush()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(1 + len(calls))]
        e[0].record(stream)
        for j, c in enumerate(calls):
            c()
            e[1 + j].record(stream)
        ev.append(e)
    torch.cuda.synchronize()
    total = [e[0].elapsed_time(e[-1]) for e in ev]
    per_part = [[e[j].elapsed_time(e[j + 1]) for e in ev] for j in range(len(calls))]
    return total, (per_part if parts else None)


def tstats(ms):
    """Mean and median of per-rep times (ms) in microseconds, with the rep count."""
    return {"mean_us": round(statistics.mean(ms) * 1e3, 2),
            "median_us": round(statistics.median(ms) * 1e3, 2), "reps": len(ms)}


def run_pkv(args):
    import torch
    import paged_kv_cache_loc_gb300 as pkv
    from paged_kv_cache_loc_gb300 import _lib, build
    from paged_kv_cache_loc_gb300 import workloads as W

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    lib = _lib.load()
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = make_l2_flush(torch, dev)

    # ---- the workload: batched GQA decode -------------------------------
    case = W.batched_decode(seed=rank_seed(rank))
    cache, q, kn, vn = W.upload(case, dev)
    o = torch.empty_like(q)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1024, device=dev)
    chunk = args.chunk
    if chunk == 0:
        plan_chunk, n_splits = pkv.decode_plan(cache, case.n_heads, ws)
        mode = (f"balanced: {n_splits} CTAs share all tokens (kv_indptr)" if plan_chunk == 0
                else f"chunked: {plan_chunk}-token splits")
    else:
        n_splits = -(-case.max_len // chunk)
        mode = f"chunked: {chunk}-token splits"
    step = DecodeStep(lib, cache, q, kn, vn, o, ws, case.layer_id, chunk, stream)
    launches_per_step = 1 + 1 + (0 if (n_splits == 1 and chunk != 0) else 1)

    with torch.cuda.stream(stream):
        if world > 1:
            torch.distributed.barrier()
        sampler = ClockSampler(local)
        sampler.start()
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        # the step as a user makes it: one pkv_decode_step call (the automatic
        # plan), or the two calls when a split size is forced
        if chunk == 0:
            step_ms, _ = timed(torch, stream, step.fused, args.steps, args.warmup, flush)
        else:
            step_ms, _ = timed(torch, stream, None, args.steps, args.warmup, flush,
                               parts=[step.write, step.decode])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall0
        # per-kernel times: the write and the decode as separate calls, each
        # bracketed by events (these give the roofline of the decode kernels)
        _, parts = timed(torch, stream, None, args.steps, args.warmup, flush,
                         parts=[step.write, step.decode])
        torch.cuda.synchronize()
        clocks = sampler.stop()
    st, detail = pkv.last_device_error(stream, dev)
    if st != 0:
        raise RuntimeError(f"device error word set during the benchmark (detail {detail})")

    ms_step = statistics.mean(step_ms)
    ms_write = statistics.mean(parts[0])
    ms_decode = statistics.mean(parts[1])
    b_dec = decode_bytes(case)
    b_wr = kv_write_bytes(case)
    total_ms = job_step_ms(torch, ms_step, dev)
    value = job_value_gbs(world, b_dec + b_wr, total_ms)

    achieved = b_dec / (ms_decode * 1e-3) / 1e9
    roofline = {
        "bound": "hbm", "kernel": "paged_decode (split + merge)",
        "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": round(achieved / peaks["hbm_gbs"], 4),
        "peak_source": peaks["hbm_source"],
        "traffic": profile_traffic("decode_split_batched_b32.md", "pkv_decode.cu", "pkv_decode_mma.cu"),
        "traffic_note": "split + merge DRAM bytes of one call from the committed ncu summary",
        "algorithmic_bytes_per_launch": b_dec,
        "ms_per_launch": round(ms_decode, 5),
    }

    out = {
        "metric": "paged-decode attention KV GB/s (decode step: kv_write + paged_decode), batched GQA decode",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) K/V/q, permuted slots)",
        "config": dict(workload_config(case, world), decode_plan=mode,
                       l2="flushed before every timed step (256 MB write, then 256 MB read)"),
        "decode_tokens_per_s": round(world * case.batch / (total_ms * 1e-3), 1),
        "attention_stack_tokens_per_s": round(world * case.batch / (case.n_layers * total_ms * 1e-3), 1),
        "kv_write_ms": round(ms_write, 5),
        "roofline": roofline,
        "gpu_launches": launches_per_step * args.steps,
        "step_call": ("pkv_decode_step (kv_write, then the decode split kernel as its programmatic "
                      "dependent, then the merge)" if chunk == 0 else "pkv_kv_write + pkv_paged_decode_chunked"),
        "decode_only_ms": round(ms_decode, 5),
        "timing": {"statistic": "mean of the timed reps (value, ms_per_step); medians beside",
                   "step": tstats(step_ms), "kv_write": tstats(parts[0]),
                   "decode": tstats(parts[1])},
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }

    if not args.no_extras:
        out["e2e"] = e2e_leg(torch, pkv, lib, case, cache, ws, chunk, stream, flush, args, dev)
        if chunk == 0:
            out["graph_step"] = graph_step_leg(torch, step, stream, flush, args, b_dec + b_wr,
                                               ms_step, peaks)
        out["long_context_b1"] = long_context_leg(torch, pkv, W, stream, flush, peaks, dev)
        out["prefix_shared_pages"] = prefix_shared_leg(torch, pkv, W, stream, flush, peaks, dev)
        out["prefill"] = prefill_leg(torch, pkv, W, stream, flush, peaks, args, dev)
    if rank == 0 and not args.no_extras:
        out["cpu_baseline"] = cpu_baseline(case, b_dec + b_wr)
        out["oracle_per_config"] = oracle_per_config(W)
        out["host_allocator"] = allocator_leg()
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def graph_step_leg(torch, step, stream, flush, args, step_bytes, eager_ms, peaks):
    """The decode step as a serving loop replays it: the pkv_decode_step call
    captured once in a CUDA graph (its programmatic edge becomes a graph
    edge), replayed with the L2 flushed before each replay."""
    with torch.cuda.stream(stream):
        ms, g = graph_replay_ms(torch, stream, step.fused, args.steps, args.warmup, flush)
    t = statistics.mean(ms)
    del g
    return {"us_per_step": round(t * 1e3, 2), "timing": tstats(ms),
            "kv_gbs": round(step_bytes / (t * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(step_bytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "eager_us_per_step": round(eager_ms * 1e3, 2),
            "what": "pkv_decode_step captured in a CUDA graph, replayed; L2 flushed before each replay"}


def e2e_leg(torch, pkv, lib, case, cache, ws, chunk, stream, flush, args, dev):
    """Same step through the public API with the step's inputs in pinned host
    memory, packed the way a serving loop sends them: q, k_new, v_new and the
    per-step metadata in one pinned buffer, one host-to-device copy, the step
    call (decode_step) on views of the device copy, one device-to-host copy of
    o -- all inside the events."""
    parts = [np.ascontiguousarray(a) for a in (case.q, case.k_new, case.v_new, case.seq_lens,
                                               case.req_pool_indices, case.out_cache_loc,
                                               case.kv_indptr)]
    offs, total = [], 0
    for a in parts:   # 256-byte aligned fields
        offs.append(total)
        total += (a.nbytes + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    hb = host.numpy()
    for a, off in zip(parts, offs):
        hb[off: off + a.nbytes] = a.view(np.uint8).reshape(-1)
    devbuf = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(i, dtype, shape):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        return devbuf[offs[i]: offs[i] + n].view(dtype).view(shape)

    bf = torch.bfloat16
    dq = view(0, bf, case.q.shape)
    dk = view(1, bf, case.k_new.shape)
    dv = view(2, bf, case.v_new.shape)
    c = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                    req_to_token=cache.req_to_token,
                    req_pool_indices=view(4, torch.int32, case.req_pool_indices.shape),
                    seq_lens=view(3, torch.int32, case.seq_lens.shape),
                    out_cache_loc=view(5, torch.int32, case.out_cache_loc.shape),
                    kv_indptr=view(6, torch.int32, case.kv_indptr.shape), max_len=case.max_len)
    ho = torch.empty(case.q.shape, dtype=bf).pin_memory()
    do = torch.empty(case.q.shape, dtype=bf, device=dev)

    def step():
        devbuf.copy_(host, non_blocking=True)
        if chunk == 0:
            pkv.decode_step(c, case.layer_id, dk, dv, dq, do, workspace=ws, stream=stream)
        else:
            pkv.kv_write(c, case.layer_id, dk, dv, stream=stream)
            pkv.paged_decode(c, case.layer_id, dq, do, workspace=ws, chunk=chunk, stream=stream)
        ho.copy_(do, non_blocking=True)

    n = max(20, args.steps // 4)
    with torch.cuda.stream(stream):
        ms, _ = timed(torch, stream, step, n, 5, flush)
    assert torch.equal(ho, do.cpu())
    h2d = total
    d2h = ho.numel() * ho.element_size()
    b = decode_bytes(case) + kv_write_bytes(case)
    t = statistics.mean(ms)
    copies = {"value": round(b / (t * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(t, 5),
              "timing": tstats(ms),
              "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
              "path": ("one pinned host -> device copy of the packed step inputs (q, k_new, v_new, "
                       "seq_lens, req_pool_indices, out_cache_loc, kv_indptr), the public API call, "
                       "device -> pinned host copy of o")}
    if chunk != 0:
        return copies

    # The same step with no copies: the public API call takes the pinned host
    # buffers themselves, and its kernels read the inputs and write o over
    # the host link (the GPU maps pinned host memory).
    def hview(i, dtype, shape):
        nb = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        return host[offs[i]: offs[i] + nb].view(dtype).view(shape)

    hc = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                     req_to_token=cache.req_to_token,
                     req_pool_indices=hview(4, torch.int32, case.req_pool_indices.shape),
                     seq_lens=hview(3, torch.int32, case.seq_lens.shape),
                     out_cache_loc=hview(5, torch.int32, case.out_cache_loc.shape),
                     kv_indptr=hview(6, torch.int32, case.kv_indptr.shape), max_len=case.max_len)
    hq, hk, hv = hview(0, bf, case.q.shape), hview(1, bf, case.k_new.shape), hview(2, bf, case.v_new.shape)
    ho2 = torch.empty(case.q.shape, dtype=bf).pin_memory()

    def step_in_place():
        pkv.decode_step(hc, case.layer_id, hk, hv, hq, ho2, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        ms2, _ = timed(torch, stream, step_in_place, n, 5, flush)
    torch.cuda.synchronize()
    assert torch.equal(ho2, ho)
    t2 = statistics.mean(ms2)
    return {"value": round(b / (t2 * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(t2, 5),
            "timing": tstats(ms2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "path": ("the public API call (decode_step) on pinned host buffers: the kernels read q, "
                     "k_new, v_new and the metadata (seq_lens, req_pool_indices, out_cache_loc, "
                     "kv_indptr) from host memory and write o to host memory, no copy calls"),
            "with_copies": copies}


def long_context_leg(torch, pkv, W, stream, flush, peaks, dev):
    """B=1 decode over the long-context sweep (1K-32K tokens, split-K across
    the SMs); the 32,768-token point is the headline."""
    sweep = []
    for ctx in W.LONG_CONTEXTS:
        case = W.long_decode(ctx)
        cache, q, kn, vn = W.upload(case, dev)
        pkv.kv_write(cache, case.layer_id, kn, vn)
        ws = pkv.Workspace(1, case.n_heads, case.head_dim, 1024, device=dev)
        o = torch.empty_like(q)
        plan_chunk, n_splits = pkv.decode_plan(cache, case.n_heads, ws)
        with torch.cuda.stream(stream):
            ms, _ = timed(torch, stream,
                          lambda: pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws,
                                                   stream=stream), 100, 10, flush)
            gms, g = graph_replay_ms(
                torch, stream, lambda: pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws,
                                                        stream=stream), 100, 10, flush)
            del g
        # means: the event clock here ticks in ~1 us steps, which a median
        # of microsecond-scale calls would round to
        t = statistics.mean(ms)
        tg = statistics.mean(gms)
        b = decode_bytes(case)
        gbs = b / (t * 1e-3) / 1e9
        sweep.append({"context": ctx, "us_per_decode": round(t * 1e3, 2), "timing": tstats(ms),
                      "graph_timing": tstats(gms), "kv_gbs": round(gbs, 1),
                      "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                      "graph_us_per_decode": round(tg * 1e3, 2),
                      "graph_frac_of_hbm_peak": round(b / (tg * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                      "decode_plan": (f"balanced: {n_splits} CTAs" if plan_chunk == 0
                                      else f"chunked: {plan_chunk}-token splits"),
                      "algorithmic_bytes": b})
        del cache, q, kn, vn, ws, o
    out = dict(sweep[-1])
    out["sweep"] = [{k: s[k] for k in ("context", "us_per_decode", "kv_gbs", "frac_of_hbm_peak",
                                       "graph_us_per_decode", "timing")}
                    for s in sweep]
    return out


def prefix_shared_leg(torch, pkv, W, stream, flush, peaks, dev):
    """The prefix-shared workload (64 requests reading the same 2048-slot
    prefix, private tails in 16-slot pages) decoded through the page table.
    Logical bytes count every request's rows; unique bytes count each slot
    once.  Timed with the L2 flushed before each call and without (then the
    shared prefix stays in L2)."""
    case = W.prefix_shared_decode()
    cache, q, kn, vn = W.upload(case, dev)
    pkv.kv_write(cache, case.layer_id, kn, vn)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1024, device=dev)
    o = torch.empty_like(q)
    ps = case.page_size
    table = torch.from_numpy(np.ascontiguousarray(case.req_to_token[:, ::ps] // ps)).to(dev)
    used = np.unique(np.concatenate([case.slots_of(b) for b in range(case.batch)]))
    row = case.n_kv_heads * case.head_dim * case.elem_bytes
    logical = decode_bytes(case)
    unique = float(used.size) * 2 * row + float(case.seq_lens.sum()) * 4 + \
        2.0 * case.batch * case.n_heads * case.head_dim * case.elem_bytes
    n_shared = case.shared_prefix // ps
    call = lambda: pkv.paged_decode_pages(cache, case.layer_id, table, ps, q, o, workspace=ws,
                                          stream=stream, shared_pages=n_shared)
    plain = lambda: pkv.paged_decode_pages(cache, case.layer_id, table, ps, q, o, workspace=ws,
                                           stream=stream)
    out = {"batch": case.batch, "page_size": ps, "shared_prefix_tokens": case.shared_prefix,
           "logical_bytes": logical, "unique_bytes": unique,
           "call": f"paged_decode_pages with shared_pages={n_shared} (the shared pages are read once "
                   f"per launch by a tensor-core kernel over all requests' query heads; the private "
                   f"pages by the split kernel on the other SMs)"}

    def rates(ms):
        t = statistics.mean(ms)
        return {"us_per_decode": round(t * 1e3, 2), "timing": tstats(ms),
                "logical_gbs": round(logical / (t * 1e-3) / 1e9, 1),
                "unique_gbs": round(unique / (t * 1e-3) / 1e9, 1),
                "unique_frac_of_hbm_peak": round(unique / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    with torch.cuda.stream(stream):
        for name, fl in (("l2_flushed", flush), ("l2_warm", lambda: None)):
            ms, _ = timed(torch, stream, call, 100, 10, fl)
            out[name] = rates(ms)
        # the same decode without the statement: every request reads the prefix
        ms, _ = timed(torch, stream, plain, 100, 10, flush)
        out["without_shared_pages_l2_flushed"] = rates(ms)
    st, detail = pkv.last_device_error(stream, dev)
    if st != 0:
        raise RuntimeError(f"device error word set in the prefix-shared leg (detail {detail})")
    return out


def prefill_leg(torch, pkv, W, stream, flush, peaks, args, dev):
    """Ragged causal prefill: 16 requests, q_len U[128, 2048], prefix U[0, 4096]."""
    case = W.ragged_prefill()
    cache, q, kn, vn = W.upload(case, dev)
    o = torch.empty_like(q)
    # a workspace lets the prefill take its entries longest first
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1, device=dev)

    def write():
        pkv.kv_write(cache, case.layer_id, kn, vn, stream=stream)

    def attend():
        pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, o=o,
                          workspace=ws, stream=stream)
    # the fused RoPE write of the same rows: standard rotary table
    # (theta = 10000^(-2i/d), [max_pos, d/2, 2] f32), each new token at its
    # position P + i in its request
    d = case.head_dim
    max_pos = int(case.seq_lens.max())
    inv = 10000.0 ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    table = torch.from_numpy(np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32)).to(dev)
    pos = np.concatenate([np.arange(int(case.seq_lens[b] - case.q_lens[b]), int(case.seq_lens[b]))
                          for b in range(case.batch)]).astype(np.int32)
    positions = torch.from_numpy(pos).to(dev)

    def rope_write():
        pkv.rope_kv_write(cache, case.layer_id, kn, vn, table, positions, stream=stream)
    with torch.cuda.stream(stream):
        ms_r, _ = timed(torch, stream, rope_write, args.prefill_steps, 3, flush)
        # the plain write last, so the prefill attends to the unrotated rows
        ms, parts = timed(torch, stream, None, args.prefill_steps, 3, flush, parts=[write, attend])
    t_attn = statistics.mean(parts[1])
    t_wr = statistics.mean(parts[0])
    t_rope = statistics.mean(ms_r)
    fl = prefill_flops(case)
    tf = fl / (t_attn * 1e-3) / 1e12
    wb = kv_write_bytes(case)
    rb = wb + float(pos.size) * (4 + (d // 2) * 2 * 4)   # + position and table row per token
    return {"workload": "ragged causal prefill", "total_q": int(case.q_lens.sum()),
            "launch_order": "kv heads of a query-tile pair together; entries by decreasing kv_len (planning kernel, workspace given)",
            "causal_flops": fl, "ms_prefill": round(t_attn, 4),
            "tflops": round(tf, 1), "roofline": {
                "bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                "peak_source": peaks["bf16_source"],
                "traffic": profile_traffic("prefill_tc_ragged.md", "pkv_prefill_tc.cu"),
                "traffic_note": "DRAM bytes read + written per launch of the whole workload, from the committed ncu summary"},
            "kv_write_ms": round(t_wr, 4), "kv_write_gbs": round(wb / (t_wr * 1e-3) / 1e9, 1),
            "kv_write_frac_of_hbm": round(wb / (t_wr * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "rope_kv_write_ms": round(t_rope, 4),
            "rope_kv_write_gbs": round(rb / (t_rope * 1e-3) / 1e9, 1),
            "rope_kv_write_frac_of_hbm": round(rb / (t_rope * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "ms_per_step": round(statistics.mean(ms), 4),
            "timing": {"prefill": tstats(parts[1]), "kv_write": tstats(parts[0]),
                       "rope_kv_write": tstats(ms_r)},
            "head_dim_64": prefill_d64_leg(torch, pkv, W, stream, flush, peaks, args, dev)}


def prefill_d64_leg(torch, pkv, W, stream, flush, peaks, args, dev):
    """The same ragged causal prefill shape at head_dim 64 (the tcgen05 kernel's
    head_dim-64 instantiation)."""
    case = W.ragged_prefill(head_dim=64)
    cache, q, kn, vn = W.upload(case, dev)
    pkv.kv_write(cache, case.layer_id, kn, vn, stream=stream)
    o = torch.empty_like(q)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1, device=dev)
    with torch.cuda.stream(stream):
        ms, _ = timed(torch, stream, lambda: pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len,
                                                              case.max_len, o=o, workspace=ws,
                                                              stream=stream),
                      args.prefill_steps, 3, flush)
    st, detail = pkv.last_device_error(stream, dev)
    if st != 0:
        raise RuntimeError(f"device error word set in the head_dim 64 prefill (detail {detail})")
    t = statistics.mean(ms)
    fl = prefill_flops(case)
    tf = fl / (t * 1e-3) / 1e12
    return {"causal_flops": fl, "ms_prefill": round(t, 4), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4), "timing": tstats(ms)}


def allocator_leg():
    """The host page allocator (C++) on the prefix-shared workload's shapes:
    64 tasks whose prompts share a 2048-token prefix (128 pages of 16) plus
    U[0, 1024] private tokens, each allocated (prefix pages found by hash),
    its hashes recorded, then all freed; 20 rounds.  The Python oracle of the
    same allocator is timed on the same sequence."""
    import oracle.pool_oracle as po
    from paged_kv_cache_loc_gb300.pool import PagePool
    rng = np.random.Generator(np.random.PCG64(1004))
    prefix = rng.integers(0, 32000, 2048).tolist()
    prompts = [prefix + rng.integers(0, 32000, int(n)).tolist()
               for n in rng.integers(0, 1024, 64, endpoint=True)]
    pages_per_round = sum(-(-len(p) // 16) for p in prompts)

    def run(pool, record):
        t0 = time.perf_counter()
        for rnd in range(20):
            for i, p in enumerate(prompts):
                rc, _ = pool.task_alloc(rnd * 64 + i, p)
                assert rc == 0
                record(pool, rnd * 64 + i, p)
            for i in range(64):
                pool.task_free(rnd * 64 + i)
        return time.perf_counter() - t0

    t_py = run(po.PoolOracle(8192, 16), lambda pool, t, p: pool.task_record_hashes(t, p))
    prompts = [np.asarray(p, np.int32) for p in prompts]   # the C++ pool takes int32 arrays
    t_c = run(PagePool(8192, 16), lambda pool, t, p: pool.task_record_hashes(t, p))
    n = 20 * 64
    return {"tasks": n, "pages_mapped": 20 * pages_per_round,
            "us_per_task": round(t_c / n * 1e6, 2),
            "tasks_per_s": round(n / t_c, 1),
            "oracle_us_per_task": round(t_py / n * 1e6, 2),
            "what": "task_alloc (prefix lookup by page hash) + task_record_hashes + task_free, "
                    "C++ pool through the ctypes binding on int32 prompt arrays; the Python "
                    "oracle on the same sequence"}


def cpu_baseline(case, step_bytes):
    """The fp64 oracle (single-threaded C) on the same decode step."""
    import oracle
    from paged_kv_cache_loc_gb300 import workloads as W  # noqa: F401
    # the oracle's write goes to copies of the touched rows only: rebuild a
    # small pool holding just this layer so the copy stays cheap
    t0 = time.perf_counter()
    kb = case.k_buffer[case.layer_id:case.layer_id + 1].copy()
    vb = case.v_buffer[case.layer_id:case.layer_id + 1].copy()
    t_copy = time.perf_counter() - t0
    reps = []
    for _ in range(2):
        t0 = time.perf_counter()
        oracle.kv_write(kb, vb, 0, case.k_new, case.v_new, case.out_cache_loc)
        oracle.decode(kb, vb, case.req_to_token, case.req_pool_indices, case.seq_lens, case.q, 0)
        reps.append(time.perf_counter() - t0)
    t = min(reps)
    return {"value": round(step_bytes / t / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "seconds_per_step": round(t, 3),
            "sample": "the full decode step (kv_write of 32 rows + decode of all 32 requests, "
                      "all heads), best of 2; pool restricted to the target layer "
                      f"(copy {t_copy:.2f}s, untimed)", "host_threads_available": os.cpu_count()}


def oracle_per_config(W):
    """The fp64 oracle (1 host core) on the other workloads, each on a bounded
    sample: the B=1 32K decode whole, 8 of the 64 prefix-shared requests, and
    ~4 sampled query rows per request of the ragged prefill (extrapolated to
    the whole prefill by its count of unmasked (query, key) pairs)."""
    import oracle
    out = {}
    case = W.long_decode(32768)
    t0 = time.perf_counter()
    oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                  case.seq_lens, case.q, case.layer_id)
    t = time.perf_counter() - t0
    out["b1_32k_decode"] = {"seconds": round(t, 3), "kv_gbs": round(decode_bytes(case) / t / 1e9, 4),
                            "sample": "the whole decode"}
    del case
    case = W.prefix_shared_decode()
    sel = np.arange(8)
    t0 = time.perf_counter()
    oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices[sel],
                  case.seq_lens[sel], case.q[sel], case.layer_id)
    t = time.perf_counter() - t0
    row = case.n_kv_heads * case.head_dim * case.elem_bytes
    logical = float(case.seq_lens[sel].sum()) * (2 * row + 4)
    out["prefix_shared_decode"] = {"seconds": round(t, 3), "logical_kv_gbs": round(logical / t / 1e9, 4),
                                   "sample": "8 of the 64 requests (all heads)",
                                   "extrapolated_seconds": round(t * float(case.seq_lens.sum()) /
                                                                 float(case.seq_lens[sel].sum()), 2)}
    del case
    case = W.ragged_prefill()
    rows = W.prefill_sample_rows(case, n_random=1)
    t0 = time.perf_counter()
    oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                   case.qo_indptr, case.kv_indptr, case.q, case.layer_id, rows=rows)
    t = time.perf_counter() - t0
    # unmasked keys of each sampled row, against those of every row
    seen = 0
    for r in rows:
        b = int(np.searchsorted(case.qo_indptr, r, side="right") - 1)
        i = int(r - case.qo_indptr[b])
        seen += int(case.kv_indptr[b + 1] - case.kv_indptr[b] - (case.qo_indptr[b + 1] - case.qo_indptr[b])) + i + 1
    flops_sampled = 4.0 * case.head_dim * case.n_heads * seen
    flops_all = prefill_flops(case)
    out["ragged_prefill"] = {"seconds": round(t, 3), "rows": int(rows.size),
                             "rows_per_s": round(rows.size / t, 2),
                             "gflops": round(flops_sampled / t / 1e9, 3),
                             "extrapolated_seconds": round(t * flops_all / flops_sampled, 1),
                             "sample": f"{rows.size} query rows (per request rows 0, 1, q_len-1 and one "
                                       "seeded row), all heads"}
    return out


# ---------------------------------------------------------------------------
# the reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_loc_gb300 import workloads as W
    case = W.batched_decode()
    kb = case.k_buffer[case.layer_id:case.layer_id + 1].copy()
    vb = case.v_buffer[case.layer_id:case.layer_id + 1].copy()
    oracle.kv_write(kb, vb, 0, case.k_new, case.v_new, case.out_cache_loc)
    # each step: the decode of one request (all heads) and its cache write,
    # cycling through the batch
    per_req = []
    for b in range(case.batch):
        sub = dict(req_pool_indices=case.req_pool_indices[b:b + 1], seq_lens=case.seq_lens[b:b + 1],
                   q=case.q[b:b + 1])
        tok = int(case.seq_lens[b])
        row = case.n_kv_heads * case.head_dim * 2
        nbytes = tok * 2 * row + tok * 4 + 2 * case.n_heads * case.head_dim * 2 + (2 * row * 2 + 4)
        per_req.append((sub, nbytes, b))

    def one(i):
        sub, nbytes, b = per_req[i % case.batch]
        oracle.kv_write(kb, vb, 0, case.k_new[b:b + 1], case.v_new[b:b + 1],
                        case.out_cache_loc[b:b + 1])
        oracle.decode(kb, vb, case.req_to_token, sub["req_pool_indices"], sub["seq_lens"], sub["q"], 0)
        return nbytes
    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    total = 0
    for i in range(args.steps):
        total += one(i)
    t = time.perf_counter() - t0
    value = total / t / 1e9
    print(json.dumps({
        "impl": "reference",
        "metric": "paged-decode attention KV GB/s (decode step: kv_write + paged_decode), batched GQA decode",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V/q, permuted slots)",
        "config": dict(workload_config(case, world), decode_plan="oracle: one plain pass per request",
                       l2="host memory (the oracle runs on the host cores)"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "each step = one request's cache write + decode (all 32 heads), "
                                   "cycling through the 32 requests of the workload"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.decode_sweep:
        run_decode_sweep()
    elif args.profile_case:
        run_profile_case(args.profile_case)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
