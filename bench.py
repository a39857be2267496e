#!/usr/bin/env python3
"""Decode-step benchmark of the paged KV-cache attention library.

One step = the whole hot path over one batch: the cache write of every
sequence's new token (reshape_and_cache) followed by paged decode attention
(plus its log-sum-exp combine when the context is partitioned).  Inputs are
seeded synthetic workloads resident in HBM before timing starts.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --workload gqa_8b --dtype f16 --block-size 64 --only
  python bench.py --impl reference ...   # the float64 CPU oracle as the reference arm

The default workload is long_ctx, the largest single-GPU batch (GQA 64/8
heads, contexts of 32k-128k tokens split into 512-token partitions).  The
same JSON line carries, under "other_workloads", the decode call of the
gqa_8b, shared_prefix and mha_7b batches timed in the same process.  Shape
flags (--dtype, --block-size, --head-dim, --num-heads, --num-kv-heads,
--partition) rebuild the chosen workload's lengths and placement with other
storage, block or head geometry; with any of them, or with --only, the other
workloads are skipped.

For N > 1 launch under torchrun; every rank runs its own batch (weak
scaling, no collective on the data path) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time


ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

DEFAULT_WORKLOAD = "long_ctx"
OTHER_WORKLOADS = ("gqa_8b", "shared_prefix", "mha_7b")
# device time the decode-alone loop behind the roofline covers, at least
ROOFLINE_SECONDS = 0.25
METRIC = "paged decode attention effective KV-read GB/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per decode launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum of the decode kernel alone), keyed by
# workload and kernel family, valid only while the kernel sources hash to
# `src`; a shape override (dtype, block or head size) has no record.
NCU_TRAFFIC: dict = {
    ("mha_7b", "plain"): {"bytes": 1106876544, "src": "b53d7a8325de8b4e"},
    ("gqa_8b", "plain"): {"bytes": 2371565696, "src": "b53d7a8325de8b4e"},
    ("long_ctx", "plain"): {"bytes": 2981254784, "src": "b53d7a8325de8b4e"},
    # the shared-prefix kernel's sources include the plain kernel's header,
    # so a change there re-dates this record too
    ("shared_prefix", "shared"): {"bytes": 858577792, "src": "e76b915b6c7498aa"},
}


# Source files of each timed kernel family (a change to any of them makes the
# recorded DRAM traffic stale).
KERNEL_SOURCES = {
    "plain": ["decode_kernel.cuh", "pkv_device.cuh", "pkv_internal.h", "api.cu",
              "decode_bf16_d128.cu", "decode_bf16_d64.cu", "decode_f32_d128.cu", "decode_f32_d64.cu"],
    "shared": ["shared_prefix_kernel.cuh", "shared_prefix.cu", "shared_prefix_d128.cu",
               "decode_kernel.cuh", "pkv_device.cuh", "pkv_internal.h", "api.cu"],
}


def kernel_source_hash(family: str = "plain") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_249_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[family]):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peak_gbs() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed
    regions run (read-only queries; no setting is changed)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int = 0, period_ms: int = 20):
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.window = (0.0, 0.0)
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={uuid}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 5.0:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    @staticmethod
    def now() -> float:
        return time.monotonic()

    def mark_start(self):
        self.window = (time.monotonic(), self.window[1])

    def mark_end(self):
        self.window = (self.window[0], time.monotonic())

    def stop(self) -> dict:
        """End sampling; the summary of the window marked by mark_start/mark_end."""
        if self.proc is None:
            return self.summary(0.0, 0.0)
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        return self.summary(*self.window)

    def summary(self, t0: float, t1: float) -> dict:
        """Median SM clock, the largest max clock and the active throttle
        reasons of the samples taken between t0 and t1 (monotonic seconds)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = "timed region"
        if not inside and self.samples:  # region shorter than the sampling period
            nearest = min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))
            inside = [nearest[1]]
            note = "nearest sample (region shorter than the sampling period)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in inside if len(s) > 8 and num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if len(s) > 8 and num(s[2]) is not None]
        reasons = sorted({self.REASONS[i] for s in inside if len(s) > 8
                          for i, v in enumerate(s[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "seconds": round(t1 - t0, 3), "window": note}


# ----------------------------------------------------------------- ranks --

def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (the job is as slow as its slowest rank)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------ workloads --

def shape_overrides(args) -> dict:
    """Keyword overrides of workload.make from the shape flags."""
    ov = {}
    for flag, key in (("dtype", "dtype"), ("block_size", "block_size"), ("head_dim", "head_dim"),
                      ("num_heads", "num_heads"), ("num_kv_heads", "num_kv_heads"),
                      ("partition", "partition_tokens")):
        v = getattr(args, flag, None)
        if v is not None:
            ov[key] = v
    return ov


def make_workload(name: str, overrides: dict):
    from paged_kv_cache_249_gb300 import workload as wl
    return wl.make(name, **overrides)


def algorithmic_bytes(w) -> dict:
    """Bytes the decode step must move at minimum (per rank, per step)."""
    e = w.elem_bytes
    kv_logical = w.kv_bytes_logical()
    kv_unique = w.kv_bytes_unique()
    q = w.num_seqs * w.num_heads * w.head_dim * e
    out = w.num_seqs * w.num_heads * w.head_dim * 2  # bf16 output
    table = int(np.sum((w.context_lens.astype(np.int64) + w.block_size - 1) // w.block_size)) * 4
    new_kv = 2 * w.num_seqs * w.num_kv_heads * w.head_dim * e
    return {"kv_logical": kv_logical, "kv_unique": kv_unique, "q": q, "out": out,
            "table": table, "new_kv": new_kv,
            "decode_launch": kv_unique + q + out + table + w.num_seqs * 4}


def workload_config(w, name: str, world: int, overrides: dict | None = None) -> dict:
    from paged_kv_cache_249_gb300 import workload as wl
    desc = f"{name}: {wl.WORKLOADS[name]['desc']}"
    if overrides:
        desc += " [shape flags: " + ", ".join(f"{k}={v}" for k, v in overrides.items()) + "]"
    return {"workload": desc, "num_seqs": w.num_seqs,
            "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "kv_dtype": w.dtype, "out_dtype": "bf16",
            "accumulate": "f32", "mean_context": float(w.context_lens.mean()),
            "kv_bytes_per_step": w.kv_bytes_logical(),
            "partition_tokens": w.partition_tokens or "auto",
            "l2": f"inputs larger than L2 ({w.kv_bytes_unique() / 1e6:.0f} MB of unique KV per "
                  "step vs 129 MB L2); no flush",
            "parallelism": f"replicas x{world} (each rank its own batch)"}


def shared_prefix_supported(w) -> bool:
    """Shapes the shared-prefix decode takes (16-bit pools, or fp32 pools up
    to head size 128; blocks that are whole 16-row runs; groups up to 16)."""
    return ((w.dtype in ("bf16", "f16") or (w.dtype == "f32" and w.head_dim <= 128))
            and w.block_size % 16 == 0 and w.num_heads // w.num_kv_heads <= 16)


def time_launches(fn, stream, min_seconds: float, warmup: int = 3,
                  max_launches: int = 20000) -> dict:
    """Launch fn back to back until the launches cover at least min_seconds
    of device time, each bracketed by CUDA events on the launching stream.
    Returns per-launch milliseconds (and the loop's monotonic window)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    probe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(3)]
    for a_, b_ in probe:
        a_.record(stream)
        fn()
        b_.record(stream)
    torch.cuda.synchronize()
    per = max(1e-6, float(np.median([a_.elapsed_time(b_) for a_, b_ in probe])) / 1e3)
    n = int(min(max_launches, max(20, np.ceil(min_seconds / per))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    t0 = time.monotonic()
    for a_, b_ in ev:
        a_.record(stream)
        fn()
        b_.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    ms = [a_.elapsed_time(b_) for a_, b_ in ev]
    return {"ms": ms, "window": (t0, t1), "launches": n,
            "device_seconds": float(np.sum(ms)) / 1e3}


def launch_stats(ms: list, alg_bytes: int, peak: float) -> dict:
    """Mean and median launch time and the roofline fraction of both."""
    mean_s = float(np.mean(ms)) / 1e3
    med_s = float(np.median(ms)) / 1e3
    return {"us_mean": round(mean_s * 1e6, 2), "us_median": round(med_s * 1e6, 2),
            "achieved_gbs": round(alg_bytes / mean_s / 1e9, 1),
            "frac": round(alg_bytes / mean_s / 1e9 / peak, 4),
            "frac_median": round(alg_bytes / med_s / 1e9 / peak, 4),
            "launches": len(ms), "device_seconds": round(float(np.sum(ms)) / 1e3, 3)}


# ------------------------------------------------------------ CPU oracle --

def _oracle_sample(w, target_s: float, threads: int):
    """Pick a prefix of the batch whose oracle run takes about target_s."""
    import oracle
    from paged_kv_cache_249_gb300 import workload as wl
    first = wl.subset(w, [0])
    t0 = time.perf_counter()
    oracle.paged_decode(first.q, w.k_pool, w.v_pool, first.block_tables, first.context_lens,
                        w.scale, num_threads=threads)
    per_token = (time.perf_counter() - t0) / max(1, int(w.context_lens[0]))
    budget_tokens = target_s / max(per_token, 1e-12)
    csum = np.cumsum(w.context_lens.astype(np.int64))
    n = int(np.searchsorted(csum, budget_tokens, side="right"))
    n = max(1, min(w.num_seqs, n))
    return wl.subset(w, range(n)), n


def _oracle_time(sub, w, threads: int) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.paged_decode(sub.q, w.k_pool, w.v_pool, sub.block_tables, sub.context_lens, w.scale,
                        num_threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, target_s: float = 12.0) -> dict:
    """The float64 oracle as it stands, timed on this host's cores on a
    bounded sample of the same batch: a prefix of its sequences, or the
    whole batch repeated when one pass takes less than target_s."""
    threads = os.cpu_count() or 1
    sub, n = _oracle_sample(w, target_s, threads)
    secs = _oracle_time(sub, w, threads)
    reps = 1
    if n == w.num_seqs and secs < target_s:
        reps = max(1, int(target_s / max(secs, 1e-3)))
        secs = sum(_oracle_time(sub, w, threads) for _ in range(reps))
    kv = sub.kv_bytes_logical() * reps
    what = f"first {n} of {w.num_seqs} sequences" if n < w.num_seqs else \
        f"all {n} sequences x {reps} passes"
    return {"value": kv / secs / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{what} ({kv / 1e9:.3f} GB of KV), {secs:.2f} s on {threads} threads",
            "seqs_per_s": n * reps / secs}


# ---------------------------------------------------------------- native --

def _decode_path(args, w) -> bool:
    """True when the step decodes through the shared-prefix entry point."""
    if args.decode == "shared":
        if not shared_prefix_supported(w):
            raise SystemExit("bench.py: the shared-prefix decode does not take this shape "
                             f"(dtype {w.dtype}, head_dim {w.head_dim}, block_size {w.block_size})")
        return True
    return args.decode == "auto" and w.group_size > 1 and shared_prefix_supported(w)


def _setup_decode(dw, w, shared: bool, partition):
    """(decode call, launches per step excluding the cache write, kernel family)."""
    if shared:
        dw.shared_prefix_setup(partition_tokens=partition or 0)
        return dw.decode_shared_prefix, 3, "shared"  # plan, decode, combine
    return dw.decode, 1 + (1 if dw.workspace is not None else 0), "plain"


def _traffic(name: str, family: str, overrides: dict):
    rec = NCU_TRAFFIC.get((name, family))
    if overrides or not rec or rec.get("src") != kernel_source_hash(family):
        return None
    return rec["bytes"]


def _cycles(us: float, clocks: dict):
    """Launch time x median SM clock: SM cycles per launch (clock-normalised time)."""
    mhz = clocks.get("sm_mhz") if clocks else None
    return None if mhz is None else round(us * mhz)


def _shared_prefix_extras(dw, w, ab, peak, stream, seconds: float) -> dict:
    """On a shared-prefix batch: the plain decode of the same tables, and the
    decode + combine of a run that reuses the step's plan (a model's later
    layers).  Leaves the shared-prefix output in dw.out."""
    ref_out = dw.out.clone()
    pl = time_launches(dw.decode, stream, seconds)
    plain_same = float((dw.out.float() - ref_out.float()).abs().max())
    dw.shared_prefix_plan()
    run = time_launches(dw.decode_shared_prefix_run, stream, seconds)
    dw.decode_shared_prefix()
    torch.cuda.synchronize()
    pl_us = float(np.mean(pl["ms"])) * 1e3
    return {"plain_decode_us": round(pl_us, 2),
            "plain_decode_frac_logical_bytes": round(
                (ab["kv_logical"] + ab["decode_launch"] - ab["kv_unique"]) / (pl_us * 1e-6) / 1e9
                / peak, 4),
            "max_abs_diff_plain_vs_shared": plain_same,
            "per_layer_run": launch_stats(run["ms"], ab["decode_launch"], peak),
            "per_layer_note": "decode + combine from one plan (a step's layers share its plan); "
                              "the decode call above includes the plan"}


def other_workload(name: str, args, peak: float, stream, clocks) -> dict:
    """Step and decode-call timing of one more standard workload, in the same
    process as the main line (decode loop of at least ROOFLINE_SECONDS)."""
    from paged_kv_cache_249_gb300 import pagedkv
    w = make_workload(name, {})
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.bfloat16)
    shared = _decode_path(argparse.Namespace(decode="auto"), w)
    decode, n_dec, family = _setup_decode(dw, w, shared, None)
    ab = algorithmic_bytes(w)

    def step():
        pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
        decode()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    step_s = t0.elapsed_time(t1) / 1e3 / args.steps
    dec = time_launches(decode, stream, args.roofline_seconds)
    st = launch_stats(dec["ms"], ab["decode_launch"], peak)
    res = {"workload": workload_config(w, name, 1)["workload"],
           "decode_path": "shared_prefix" if shared else "plain",
           "step_us": round(step_s * 1e6, 2),
           "effective_kv_gbs_step": round(ab["kv_logical"] / step_s / 1e9, 1),
           "seqs_per_s": round(w.num_seqs / step_s, 1),
           "seqs_per_s_decode_call": round(w.num_seqs / (st["us_mean"] * 1e-6), 1),
           "decode_us_mean": st["us_mean"], "decode_us_median": st["us_median"],
           "algorithmic_bytes_per_launch": ab["decode_launch"],
           "bytes_basis": "unique (shared prefix once per group and kv head)" if shared
           else "logical = unique",
           "achieved_gbs": st["achieved_gbs"], "frac": st["frac"],
           "frac_median": st["frac_median"], "peak": peak,
           "launches": st["launches"], "device_seconds": st["device_seconds"],
           "traffic": _traffic(name, family, {}),
           "clocks": None, "sm_cycles_per_launch": None,  # filled in once sampling ends
           "gpu_launches_per_step": 1 + n_dec, "_window": dec["window"]}
    if shared:
        res.update(_shared_prefix_extras(dw, w, ab, peak, stream, 0.1))
    fault = pagedkv.get_device_error(dw.pool)
    if fault:
        raise SystemExit(f"bench.py: device fault bits {fault} on {name}")
    del dw
    torch.cuda.empty_cache()
    return res


def run_native(args, world: int, rank: int) -> dict | None:
    from paged_kv_cache_249_gb300 import build as pkv_build
    from paged_kv_cache_249_gb300 import pagedkv

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the native arm needs a CUDA device")
    pkv_build.build()
    pagedkv.load()
    overrides = shape_overrides(args)
    w = make_workload(args.workload, overrides)
    peak, peak_kind = measured_peak_gbs()
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.bfloat16)
    shared = _decode_path(args, w)
    decode, n_dec, family = _setup_decode(dw, w, shared, args.partition)
    launches_per_step = 1 + n_dec
    stream = torch.cuda.current_stream()
    ab = algorithmic_bytes(w)

    def step():
        pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
        decode()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    # whole steps back to back (no event between the step's kernels, so each
    # kernel's launch can overlap the end of the one before it)
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    # the decode call alone, for the roofline of its kernels: enough launches
    # to cover ROOFLINE_SECONDS of device time
    dec = time_launches(decode, stream, args.roofline_seconds, warmup=0)
    if clocks:
        clocks.mark_end()
    barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = dec["ms"]
    # the cache write alone (reported beside the decode, outside the timed step)
    ev_rc = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(200)]
    for a_, b_ in ev_rc:
        a_.record(stream)
        pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
        b_.record(stream)
    torch.cuda.synchronize()
    rc_us = float(np.median([a_.elapsed_time(b_) for a_, b_ in ev_rc])) * 1e3
    fault = pagedkv.get_device_error(dw.pool)
    if fault:
        raise SystemExit(f"bench.py: device fault bits {fault}")

    max_s = max_over_ranks(total_ms / 1e3, world)
    ms_per_step = max_s * 1e3 / args.steps
    value = whole_job_rate(ab["kv_logical"] * args.steps, world, max_s) / 1e9
    seqs_per_s = whole_job_rate(w.num_seqs * args.steps, world, max_s)

    # ---- the same step captured once in a CUDA graph and replayed (what a
    # serving loop that replays its decode step pays; launch-bound batches gain)
    graph_us = None
    if world == 1:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_us = g0.elapsed_time(g1) * 1e3 / args.steps
        del graph

    # ---- the plain decode kernel on the same batch (what prefix awareness buys)
    plain_cmp = None
    if shared and world == 1:
        plain_cmp = _shared_prefix_extras(dw, w, ab, peak, stream, 0.1)
        plain_cmp["shared_prefix_decode_us"] = round(float(np.mean(dec_ms)) * 1e3, 2)
        plain_cmp["plain_over_shared"] = round(plain_cmp["plain_decode_us"] /
                                               plain_cmp["shared_prefix_decode_us"], 4)

    # ---- the same decode over a contiguous cache (what paging costs)
    paging = None
    if world == 1 and not args.no_contiguous and not shared:
        cache = pagedkv.ContiguousCache.from_paged(w, k_pool=dw.k_pool, v_pool=dw.v_pool)
        cout = torch.empty_like(dw.out)

        def contig_decode():
            pagedkv.contiguous_attention_decode(cache, cout, dw.q, dw.context_lens,
                                                dw.max_context_len, w.scale,
                                                partition_tokens=dw.partition_tokens,
                                                workspace=dw.workspace)
        cl = time_launches(contig_decode, stream, 0.1)
        c_us = float(np.mean(cl["ms"])) * 1e3
        p_us = float(np.mean(dec_ms)) * 1e3
        paging = {"paged_decode_us": round(p_us, 2), "contiguous_decode_us": round(c_us, 2),
                  "paged_over_contiguous": round(p_us / c_us, 4),
                  "same_output": bool(torch.equal(cout.view(torch.int16), dw.out.view(torch.int16)))}
        del cache, cout
        torch.cuda.empty_cache()

    # ---- end to end through the C ABI with host buffers: every step copies
    # its inputs from pinned host memory and its output back, double-buffered
    # so that step k+1's copies (on a copy stream) overlap step k's kernels
    pin = lambda t: t.pin_memory()  # noqa: E731
    q_h, nk_h, nv_h = pin(w.q), pin(w.new_key), pin(w.new_value)
    sm_h = pin(torch.from_numpy(w.slot_mapping))
    cl_h = pin(torch.from_numpy(w.context_lens))
    bt_h = pin(torch.from_numpy(w.block_tables))
    out_h = [torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (q_h, nk_h, nv_h, sm_h, cl_h, bt_h))
    d2h = out_h[0].numel() * out_h[0].element_size()
    bufs = [dict(q=dw.q, nk=dw.new_key, nv=dw.new_value, sm=dw.slot_mapping, cl=dw.context_lens,
                 bt=dw.block_tables, out=dw.out)]
    bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})
    copy = torch.cuda.Stream()

    def run_step(t):
        pagedkv.reshape_and_cache(dw.pool, t["nk"], t["nv"], t["sm"])
        if shared:
            pagedkv.paged_attention_decode_shared_prefix(
                dw.pool, t["out"], t["q"], t["bt"], t["cl"], dw.max_context_len, w.scale,
                dw.group_starts, dw.prefix_lens, dw.max_prefix_len, dw.sp_workspace,
                w.num_kv_heads, dw.sp_partition)
        else:
            pagedkv.paged_attention_decode(dw.pool, t["out"], t["q"], t["bt"], t["cl"],
                                           dw.max_context_len, w.scale, w.num_kv_heads,
                                           dw.partition_tokens, dw.workspace)

    def e2e_run(n, e_start=None, e_end=None):
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]

        def h2d_copy(b):
            with torch.cuda.stream(copy):
                copy.wait_event(free[b])  # the buffer's previous step has been read back
                t = bufs[b]
                for key, src in (("q", q_h), ("nk", nk_h), ("nv", nv_h), ("sm", sm_h),
                                 ("cl", cl_h)):
                    t[key].copy_(src, non_blocking=True)
                pagedkv.block_table_upload(t["bt"], bt_h, w.num_blocks, stream=copy)
                ready[b].record(copy)

        if e_start is not None:
            e_start.record(stream)
        copy.wait_stream(stream)
        h2d_copy(0)
        for k in range(n):
            b = k % 2
            stream.wait_event(ready[b])
            run_step(bufs[b])
            done[b].record(stream)
            if k + 1 < n:
                h2d_copy((k + 1) % 2)
            with torch.cuda.stream(copy):
                copy.wait_event(done[b])
                out_h[b].copy_(bufs[b]["out"], non_blocking=True)
                free[b].record(copy)
        stream.wait_stream(copy)
        if e_end is not None:
            e_end.record(stream)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, e0, e1)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = whole_job_rate(ab["kv_logical"] * args.steps, world, e2e_s) / 1e9
    e2e_ok = all(torch.equal(o.view(torch.int16), dw.out.cpu().view(torch.int16)) for o in out_h) \
        if dw.out.dtype == torch.bfloat16 else None
    fault = pagedkv.get_device_error(dw.pool)
    if fault:
        raise SystemExit(f"bench.py: device fault bits {fault}")
    del dw, bufs
    torch.cuda.empty_cache()

    if rank != 0:
        return None
    st = launch_stats(dec_ms, ab["decode_launch"], peak)

    # ---- the other standard workloads, timed in the same process
    others = None
    if world == 1 and not overrides and not args.only:
        others = {name: other_workload(name, args, peak, stream, clocks)
                  for name in OTHER_WORKLOADS if name != args.workload}
    clock_info = clocks.stop() if clocks else None
    roof_clocks = clocks.summary(*dec["window"]) if clocks else None
    for res in (others or {}).values():
        window = res.pop("_window")
        if clocks:
            res["clocks"] = clocks.summary(*window)
            res["sm_cycles_per_launch"] = _cycles(res["decode_us_mean"], res["clocks"])

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1), PCG64)",
        "config": workload_config(w, args.workload, world, overrides),
        "seqs_per_s": round(seqs_per_s, 1),
        "pct_hbm_peak": round(100.0 * value / world / peak, 2),
        # reported beside the KV bytes: the decode call's other traffic, the
        # cache write's time, and sequences per second of the decode call alone
        "graph_replay": None if graph_us is None else {
            "us_per_step": round(graph_us, 2),
            "note": "the same step captured once in a CUDA graph, replayed back to back"},
        "side": {"q_bytes": ab["q"], "out_bytes": ab["out"], "block_table_bytes": ab["table"],
                 "context_len_bytes": w.num_seqs * 4, "new_kv_bytes": ab["new_kv"],
                 "reshape_and_cache_us": round(rc_us, 2),
                 "seqs_per_s_decode_call": round(w.num_seqs / (st["us_mean"] * 1e-6), 1)},
        "roofline": {"bound": "hbm", "achieved": st["achieved_gbs"], "peak": peak,
                     "unit": "GB/s", "frac": st["frac"],
                     "traffic": _traffic(args.workload, family, overrides),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6800 GB/s",
                     "kernel": "shared_prefix_decode_kernel (+ plan and combine)" if shared
                     else "paged_decode_kernel (+ lse_combine when split)",
                     "algorithmic_bytes_per_launch": ab["decode_launch"],
                     "bytes_basis": "unique (shared prefix once per group and kv head)"
                     if shared else "logical = unique",
                     "decode_us_avg": st["us_mean"], "decode_us_median": st["us_median"],
                     "frac_median": st["frac_median"], "launches": st["launches"],
                     "device_seconds": st["device_seconds"],
                     "clocks": roof_clocks,
                     "sm_cycles_per_launch": _cycles(st["us_mean"], roof_clocks)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3 / args.steps, 5),
                "pipelining": "two input/output buffer sets; step k+1's host-to-device copies "
                              "and step k's device-to-host copy run on a copy stream beside "
                              "step k's kernels",
                "outputs_match_device_run": e2e_ok},
        "gpu_launches": launches_per_step * args.steps,
        "paging_overhead": paging,
        "decode_path": "shared_prefix" if shared else "plain",
        "plain_decode_comparison": plain_cmp,
        "clocks": clock_info,
        "clocks_note": "sampled every 20 ms from the first timed step to the end of the "
                       "decode-alone loop behind roofline",
        "other_workloads": others,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return line


# -------------------------------------------------------- reference arm --

def run_reference(args, world: int, rank: int) -> dict | None:
    """The float64 CPU oracle on the same workload, each step a bounded
    prefix of the batch (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    from paged_kv_cache_249_gb300 import workload as wl
    oracle.build()
    overrides = shape_overrides(args)
    w = make_workload(args.workload, overrides)
    threads = os.cpu_count() or 1
    step_budget = min(5.0, max(0.2, args.reference_seconds / max(1, args.steps + args.warmup)))
    sub, n = _oracle_sample(w, step_budget, threads)
    for _ in range(args.warmup):
        _oracle_time(sub, w, threads)
    times = [_oracle_time(sub, w, threads) for _ in range(args.steps)]
    secs = float(np.sum(times))
    kv = sub.kv_bytes_logical()
    value = kv * args.steps / secs / 1e9
    sample = (f"first {n} of {w.num_seqs} sequences per step ({kv / 1e9:.3f} GB of KV), "
              f"float64 oracle on {threads} threads")
    return {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), PCG64)", "impl": "reference",
        "config": workload_config(w, args.workload, 1, overrides),
        "seqs_per_s": round(n * args.steps / secs, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    from paged_kv_cache_249_gb300 import workload as wl
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", choices=sorted(wl.WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--decode", choices=["auto", "plain", "shared"], default="auto",
                   help="decode entry point: auto = the shared-prefix kernel for batches "
                        "with shared-prefix groups, the plain kernel otherwise")
    p.add_argument("--only", action="store_true",
                   help="time the chosen workload alone (no other_workloads)")
    p.add_argument("--dtype", choices=["bf16", "f16", "f32"], default=None,
                   help="storage type of q, the pools and the new K/V (default: the workload's)")
    p.add_argument("--block-size", type=int, choices=[16, 32, 64, 128, 256], default=None)
    p.add_argument("--head-dim", type=int, choices=[64, 128, 256], default=None)
    p.add_argument("--num-heads", type=int, default=None)
    p.add_argument("--num-kv-heads", type=int, default=None)
    p.add_argument("--partition", type=int, default=None,
                   help="partition tokens: 0 = automatic, -1 = never split, N = N tokens "
                        "(default: the workload's)")
    p.add_argument("--roofline-seconds", type=float, default=ROOFLINE_SECONDS,
                   help="device time the decode-alone loop behind roofline covers, at least")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-contiguous", action="store_true",
                   help="skip the contiguous-cache comparison")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU time budget of the oracle baseline sample")
    p.add_argument("--reference-seconds", type=float, default=120.0,
                   help="CPU time budget of the whole reference arm")
    p.add_argument("--json-out", default=None, help="also append the JSON line to this file")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    world, rank, _ = dist_setup(args.gpus)
    line = run_reference(args, world, rank) if args.impl == "reference" else \
        run_native(args, world, rank)
    if line is not None:
        text = json.dumps(line)
        print(text, flush=True)
        if args.json_out:
            with open(args.json_out, "a") as f:
                f.write(text + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
