#!/usr/bin/env python3
"""Benchmark of the data-parallel ZeRO-2 gradient step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl dpg|reference]

One step = one pass of the whole hot path over one batch of synthetic input:
(for accumulation workloads, the no_sync accumulation of every microbatch but
the last, then) the fused reduce-scatter -> 1/G normalisation -> Adam ->
bf16 all-gather over every bucket, with the per-bucket squared norms.  The R
data-parallel replicas are R gradient buffers in this GPU's HBM.  The default
workload is the 1B Llama-shaped parameter list with R = 8 and 25 MiB buckets
(50.6 GB of HBM traffic per step, far larger than L2, so no flush is needed).

Under torchrun every rank runs its own independent step on its own GPU (no
collective on the data path; the replicas are simulated inside each GPU);
value = parameters updated by all ranks per second (weak scaling).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (one
host core) on a bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (CONFIGS, KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32,  # noqa: E402
                       segments, stream_seed, token_counts)

KERNEL_SRCS = [os.path.join(ROOT, "zero_optimizer_step_gb300", "csrc", f)
               for f in ("dpg_device.cuh", "dpg_fused.cu", "dpg_host.h", "dpg_internal.h",
                         "dpg_runtime.cu", "dpg_staged.cu", "dpg_stream.cu")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
CPU_SAMPLE_ELEMS = 16 << 20          # oracle sample per CPU step


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="llama1b", choices=sorted(set(CONFIGS) - {"tiny"}))
    ap.add_argument("--cap-mib", type=float, default=None, help="override the bucket cap")
    ap.add_argument("--hockney-config", default="sweep", choices=["sweep", "llama1b"],
                    help="parameter list of the --hockney cap sweep")
    ap.add_argument("--impl", default="dpg", choices=["dpg", "reference"])
    ap.add_argument("--variant", default="direct", choices=["direct", "staged"],
                    help="fused pass: direct vector loads, or bulk-copy staging in shared memory")
    ap.add_argument("--traffic-from", default=None, metavar="CSV",
                    help="no GPU: read an ncu launch list (--csv with dram__bytes_read.sum and "
                         "dram__bytes_write.sum) of this bench's --config run and write the "
                         "fused kernel's mean DRAM bytes per launch to profiles/traffic.json")
    ap.add_argument("--replicas", type=int, default=None,
                    help="override the workload's R (simulated data-parallel replicas, 1..64)")
    ap.add_argument("--microbatches", type=int, default=None,
                    help="override the workload's K (microbatches accumulated per step, 1..16)")
    ap.add_argument("--deferred", action="store_true",
                    help="K >= 2: deferred accumulation (K bf16 gradient buffers per replica, all "
                         "summed inside the fused step; no accumulation pass)")
    ap.add_argument("--fold2", action="store_true",
                    help="K >= 3: paired accumulation (two bf16 gradient buffers per replica), "
                         "the last two microbatches folded into the fused step")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sharded", action="store_true",
                    help="ZeRO-2 split across the torchrun ranks (R = number of GPUs): each "
                         "rank exchanges gradient slices (NCCL point-to-point), updates its "
                         "shard with the library's fused pass and all-gathers the bf16 shards")
    ap.add_argument("--sharded-groups", type=int, default=1,
                    help="--sharded: pipeline the step over this many bucket ranges (the "
                         "exchange of one range in flight while the previous one is updated)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="default line only: skip its extra legs (the Hockney records, the "
                         "4.5B workload, the GPT-2 list)")
    ap.add_argument("--cpu-sample-elems", type=int, default=CPU_SAMPLE_ELEMS,
                    help="elements of each oracle sample (CPU baseline and reference arm)")
    ap.add_argument("--kernels", action="store_true",
                    help="time every kernel of the path on the workload, against its algorithmic bytes")
    ap.add_argument("--schedules", action="store_true",
                    help="DDP (all-reduce + R replica updates) against the ZeRO-2 step")
    ap.add_argument("--overlap", action="store_true",
                    help="bucket updates overlapped with a simulated backward, exposed tail vs cap")
    ap.add_argument("--backward-kind", default="spin", choices=["spin", "gemm"],
                    help="--overlap: backward simulated by one-CTA spin kernels, or by the bf16 "
                         "GEMMs of each weight's dW and dX over --tokens tokens")
    ap.add_argument("--tokens", type=int, default=4096, help="--backward-kind gemm: tokens per rank")
    ap.add_argument("--overlap-caps-mib", default="1,4,25,100,400,1048576",
                    help="--overlap: bucket caps in MiB")
    ap.add_argument("--overlap-max-ctas", default="0",
                    help="--overlap: fused-pass grid caps to sweep (0: one CTA per SM)")
    ap.add_argument("--backward-priority", action="store_true",
                    help="--overlap: give the backward stream the higher priority")
    ap.add_argument("--backward-ms", type=float, default=30.0,
                    help="duration of the simulated backward (--overlap)")
    ap.add_argument("--launch-floor", action="store_true",
                    help="one fused launch over one bucket of n elements, n = 1M..128M (R = 8), "
                         "timed from CUDA graphs with L2 flushed: the fixed cost per launch "
                         "(T = T0 + bytes / bandwidth)")
    ap.add_argument("--hockney", action="store_true",
                    help="bucket-cap sweep: per-bucket launches vs one fused launch, alpha-beta fit")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.deferred and a.fold2:
        ap.error("--deferred and --fold2 are two different accumulation schedules")
    return a


def dist_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over all ranks (the job is as slow as its slowest
    rank); a no-op for one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_slowest: float) -> float:
    """Whole-job units per second: every rank processes units_per_rank units
    in the slowest rank's time (weak scaling)."""
    return units_per_rank * world / (ms_slowest * 1e-3)


SPIN_CYCLES = 4_000_000              # about 2 ms of SM clock at 2 GHz


def device_times_ms(fn, reps: int, spin_cycles: int = SPIN_CYCLES):
    """Device time of one call of fn per sample, in ms.

    A GPU spin queued before the start event keeps the device busy while the
    host checks and marshals fn's arguments and launches its kernels, so the
    interval holds fn's kernels and the device-side gaps between them, not
    the Python call overhead (about 80 us for a 147-tensor pack)."""
    import torch
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(spin_cycles)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return ts


def cap_of(cfg, a) -> int:
    return int(a.cap_mib * (1 << 20)) if a.cap_mib else cfg.cap_bytes


def workload_desc(cfg, cap, plan_nb, total, fold2=False, deferred=False) -> dict:
    d = {"workload": f"{cfg.name}: {len(cfg.shapes)} tensors, psi={cfg.psi}, R={cfg.R} simulated "
                     f"replicas, {cap / (1 << 20):g} MiB buckets, K={cfg.K} microbatch(es), ZeRO-2 "
                     f"fused reduce-scatter+Adam+all-gather",
         "psi": cfg.psi, "R": cfg.R, "K": cfg.K, "cap_bytes": cap, "n_buckets": plan_nb,
         "total_padded": total, "grad_dtype": "bf16", "state_dtype": "f32",
         "param_views": 1, "l2": "inputs larger than L2 (no flush)"}
    if cfg.K > 1:
        d["accumulation"] = ("deferred: K bf16 gradient buffers per replica, every microbatch "
                             "summed inside the fused step (no accumulation pass)" if deferred else
                             "paired: two bf16 gradient buffers per replica; microbatches folded "
                             "into the fp32 buffers two at a time, the last two into the fused "
                             "step" if fold2 else
                             "one fp32 pass per microbatch, the last folded into the fused step")
    return d


L2_FLUSH_BELOW = 4 * 129_000_000      # bytes: four times the GB300's L2


def resident_bytes(cfg, total_padded, fold2=False, deferred=False) -> int:
    """Bytes of the step's device buffers: replica gradients (or microbatch
    buffers), fp32 accumulators, master/m/v and the bf16 parameters."""
    R, K = cfg.R, cfg.K
    grads = 2 * R * (K if deferred and K > 1 else 2 if fold2 and K >= 3 else 1)
    acc = 4 * R if K > 1 and not deferred else 0
    return (grads + acc + 12 + 2) * total_padded


def fold2_schedule(K: int):
    """Microbatches 0..K-3 as (first, pair?) accumulation passes; the last two
    are folded into the fused step."""
    out, k = [], 0
    while k + 1 < K - 2:
        out.append((k, True))
        k += 2
    if k < K - 2:
        out.append((k, False))
    return out


def algorithmic_bytes_per_param(cfg, fold2=False, deferred=False) -> dict:
    R, K = cfg.R, cfg.K
    if K > 1 and deferred:
        return {"fused": 2 * K * R + 26, "step": 2 * K * R + 26}
    if K > 1 and fold2:
        fused = 8 * R + 26
        acc = sum((8 if k == 0 else 12) * R if pair else (6 if k == 0 else 10) * R
                  for k, pair in fold2_schedule(K))
        return {"fused": fused, "step": fused + acc}
    fused = (6 * R + 26) if K > 1 else (2 * R + 26)
    step = fused + ((6 * R + (K - 2) * 10 * R) if K > 1 else 0)
    return {"fused": fused, "step": step}


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"dpg_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle baseline (rank 0, N = 1 only)
# --------------------------------------------------------------------------
def oracle_sample_step(cfg, h_grads, h_last, tokens, w, m, v, t):
    """One oracle step over a contiguous sample (elementwise: reduce, scale,
    Adam, bf16 cast)."""
    import oracle
    g = oracle.reduce(h_grads, oracle.grad_scale(tokens), last=h_last)
    oracle.adam(g, w, m, v, t=t)
    oracle.f32_to_bf16(w)


def cpu_sample_inputs(cfg, n, device):
    """Host copies of a contiguous n-element sample of the workload's inputs
    (drawn like the full workload; accumulation workloads get fp32 buffers
    holding K-1 microbatches plus a last bf16 microbatch)."""
    import torch
    seg = [(0, n)]
    R, K = cfg.R, cfg.K
    bf = lambda r, k: flat_grads_bf16(seg, n, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r, k),
                                      device=device).cpu().view(torch.int16).numpy().view(np.uint16)
    if K > 1:
        import oracle
        grads, last = [], []
        for r in range(R):
            acc = np.empty(n, np.float32)
            for k in range(K - 1):
                oracle.accumulate(bf(r, k), acc, first=(k == 0))
            grads.append(acc)
            last.append(bf(r, K - 1))
    else:
        grads, last = [bf(r, 0) for r in range(R)], None
    w = master_f32(n, stream_seed(cfg.seed, KIND_MASTER), device=device).cpu().numpy()
    return grads, last, w, np.zeros(n, np.float32), np.zeros(n, np.float32)


def host_cpu() -> str:
    """Machine, core count and CPU model of the host the oracle is timed on."""
    import platform
    model = ""
    try:
        for ln in open("/proc/cpuinfo"):
            k, _, val = ln.partition(":")
            if k.strip() in ("model name", "CPU part") and val.strip():
                model = val.strip()
                break
    except OSError:
        pass
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
                 "0xd49": "Arm Neoverse N2", "0xd8f": "Arm Neoverse V3"}
    model = arm_parts.get(model.lower(), model)
    return f"{platform.machine()}, {os.cpu_count()} cores, {model or 'model unknown'}"


def cpu_baseline(cfg, device, target_s=12.0) -> dict:
    """Time the oracle, as it stands, on one host core over a bounded sample."""
    import oracle
    oracle.build()
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except (AttributeError, OSError):
        pass
    n = CPU_SAMPLE_ELEMS
    grads, last, w, m, v = cpu_sample_inputs(cfg, n, device)
    tokens = token_counts(cfg)
    t0 = time.perf_counter()
    reps = 0
    while True:
        reps += 1
        oracle_sample_step(cfg, grads, last, tokens, w, m, v, reps)
        if time.perf_counter() - t0 >= target_s:
            break
    dt = time.perf_counter() - t0
    cores = 1
    return {"value": reps * n / dt, "unit": "params/s", "cores": cores, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"{reps} oracle steps over the first {n} elements of the workload "
                      f"(elementwise reduce+scale+Adam+bf16 cast; fixed-order fp32), one pinned core"}


# --------------------------------------------------------------------------
# GPU run
# --------------------------------------------------------------------------
def load_peak():
    try:
        pk = json.load(open(PEAKS_FILE))
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha256() -> str:
    """Hash of the kernel sources' code: comments and whitespace removed, so a
    stored capture stays valid across edits that change no code."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SRCS:
        src = open(f).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()


def traffic_key(cfg, fold2=False, deferred=False) -> str:
    """Entry of profiles/traffic.json for the fused kernel a workload launches:
    the kernel's input mode depends on R, K and the accumulation schedule."""
    sched = ("bf16" if cfg.K == 1 else "deferred" if deferred else "fold2" if fold2
             else "acc_fp32_last_bf16")
    return f"k_rs_adam_chunk R={cfg.R} K={cfg.K} {sched}"


def traffic_per_launch(cfg, cap, total_padded, fold2=False, deferred=False):
    """DRAM bytes per fused launch from the committed ncu summary, if it was
    taken on the current kernel code for the same kernel variant; scaled by
    elements when the capture ran a smaller case (the pass streams every
    element once, so its traffic grows in proportion).  None otherwise."""
    try:
        t = json.load(open(TRAFFIC_FILE))["entries"][traffic_key(cfg, fold2, deferred)]
    except (OSError, KeyError, ValueError, TypeError):
        return None
    if t.get("source_sha256") != kernel_source_sha256():
        return None
    return float(t["dram_bytes_per_launch"]) * total_padded / float(t["elements"])


def config_of(a):
    """The named workload, with R and K overridden by --replicas and
    --microbatches when given."""
    import dataclasses
    cfg = CONFIGS[a.config]
    r = getattr(a, "replicas", None)
    if r is not None:
        if not 1 <= r <= 64:
            raise SystemExit(f"--replicas {r}: R must be 1..64")
        cfg = dataclasses.replace(cfg, R=r)
    k = getattr(a, "microbatches", None)
    if k is not None:
        if not 1 <= k <= 16:
            raise SystemExit(f"--microbatches {k}: K must be 1..16")
        cfg = dataclasses.replace(cfg, K=k)
    return cfg


def fused_kernel_name(a, R, K, fold2=False, deferred=False) -> str:
    """The fused kernel the timed step launches (for the roofline label)."""
    if getattr(a, "variant", "direct") == "staged":
        return f"k_rs_adam_staged<R={R}>"
    mode = ("" if K == 1 else f" (K={K} bf16 microbatches per replica)" if deferred else
            " (fp32 accumulators + two last microbatches)" if fold2 else
            " (fp32 accumulators + last microbatch)")
    return f"k_rs_adam_chunk<R={R}>" + mode


def write_traffic(a):
    """Add the fused kernel's DRAM bytes per launch, from an ncu launch list of
    this bench's run (same arguments), to profiles/traffic.json."""
    import csv
    import re
    cfg = config_of(a)
    cap = cap_of(cfg, a)
    fold2 = bool(a.fold2) and cfg.K >= 3
    deferred = bool(a.deferred) and cfg.K >= 2
    per = {}
    with open(a.traffic_from, newline="") as fh:
        rows = [r for r in csv.reader(fh) if len(r) > 14 and r[0].isdigit()]
    for r in rows:
        name, metric, value = r[4], r[12], float(r[14].replace(",", ""))
        if not re.match(r"(void )?(dpg::)?k_rs_adam_chunk<", name):
            continue
        per.setdefault(r[0], {})[metric] = value
    launches = [d for d in per.values()
                if "dram__bytes_read.sum" in d and "dram__bytes_write.sum" in d]
    if not launches:
        raise SystemExit(f"{a.traffic_from}: no k_rs_adam_chunk launch with DRAM byte counts")
    rd = statistics.mean(d["dram__bytes_read.sum"] for d in launches)
    wr = statistics.mean(d["dram__bytes_write.sum"] for d in launches)
    import zero_optimizer_step_gb300 as dpg
    plan = dpg.dpg_plan_buckets(cfg.numels, cap, cfg.R)
    elements = plan.total_padded
    plan.destroy()
    bpp = algorithmic_bytes_per_param(cfg, fold2, deferred)["fused"]
    args = " ".join(f"--{k.replace('_', '-')} {v}" for k, v in
                    (("config", a.config), ("replicas", a.replicas),
                     ("microbatches", a.microbatches), ("cap_mib", a.cap_mib)) if v is not None)
    args += " --deferred" if deferred else " --fold2" if fold2 else ""
    entry = {
        "workload": f"{cfg.name} ({cfg.psi:,} params, {elements:,} padded elements, R={cfg.R}, "
                    f"K={cfg.K}, {cap / (1 << 20):g} MiB buckets)",
        "R": cfg.R, "K": cfg.K, "elements": elements,
        "dram_bytes_read": rd, "dram_bytes_write": wr, "dram_bytes_per_launch": rd + wr,
        "algorithmic_bytes_per_launch": bpp * cfg.psi,
        "traffic_over_algorithmic": (rd + wr) / (bpp * cfg.psi),
        "launches": len(launches), "source_sha256": kernel_source_sha256(),
        "how": "ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum "
               "--clock-control none -k regex:k_rs_adam_chunk -c 3 --csv on python bench.py "
               f"{args} --no-e2e --no-cpu-baseline --steps 3 --warmup 3; mean per launch"}
    try:
        out = json.load(open(TRAFFIC_FILE))
        if "entries" not in out:
            raise ValueError
    except (OSError, ValueError):
        out = {"entries": {}}
    out["hash"] = ("sha256 of the library's CUDA sources and headers with comments and "
                   "whitespace removed")
    out["scaling"] = ("bench.py scales an entry to another workload of the same kernel variant "
                      "by padded elements (the pass streams every element once)")
    out["entries"][traffic_key(cfg, fold2, deferred)] = entry
    with open(TRAFFIC_FILE, "w") as fh:
        json.dump(out, fh, indent=1)
    print(json.dumps(entry), flush=True)


def timed_cycles(fn, steps, warm, world, dev, stream):
    """Run fn() warm times, then steps times between two events; returns the
    mean ms per call (max over ranks) and the sorted fused-launch intervals
    that fn recorded into the event pairs it was given."""
    import torch
    for _ in range(warm):
        fn(None)
    torch.cuda.synchronize()
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(steps)]
    for e0, e1 in ev_k:
        e0.record(stream)
        e1.record(stream)
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e_start.record(stream)
    for i in range(steps):
        fn(ev_k[i])
    e_stop.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e_start.elapsed_time(e_stop) / steps, world, dev)
    return ms, sorted(e0.elapsed_time(e1) for e0, e1 in ev_k)


def fused_roofline(kernel, bpp, psi, k_all, peak, peak_kind, traffic):
    k_ms = statistics.mean(k_all)
    achieved = bpp * psi / (k_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
            "peak_kind": f"{peak_kind} (copy bandwidth)", "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "algorithmic_bytes_per_param": bpp,
            "algorithmic_bytes_per_launch": bpp * psi, "kernel_ms": k_ms,
            "kernel_ms_p10_p50_p90": [k_all[int(round(q * (len(k_all) - 1)))]
                                      for q in (0.1, 0.5, 0.9)]}


def optional_leg(fn, world: int):
    """Run one of the default line's extra legs; on one GPU, a device out of
    memory records the leg as skipped instead of losing the whole line."""
    import torch
    try:
        return fn()
    except torch.cuda.OutOfMemoryError as e:
        if world > 1:
            raise
        torch.cuda.empty_cache()
        return {"skipped": "out of device memory: " + str(e).splitlines()[0][:200]}


def all_ranks_agree(ok: bool, world: int, device) -> bool:
    """True only if `ok` holds on every rank (the same answer on all)."""
    if world <= 1:
        return bool(ok)
    import torch
    import torch.distributed as dist
    t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def device_room(needed_bytes: int, world: int, device) -> bool:
    """Whether every rank's GPU has needed_bytes free, with 2 GB to spare."""
    import torch
    free, _ = torch.cuda.mem_get_info(device)
    return all_ranks_agree(free >= needed_bytes + (2 << 30), world, device)


def run_gpt2_leg(a, dpg, dev, world):
    """The GPT-2-small-shaped list (R = 8, 25 MiB buckets) in the default line:
    the whole step (fused pass + norm finalize) and its fused launch."""
    import torch
    cfg = CONFIGS["gpt2"]
    plan = dpg.dpg_plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    N = plan.total_padded
    if not device_room(resident_bytes(cfg, N), world, dev):
        return {"skipped": f"needs {resident_bytes(cfg, N) / 1e9:.0f} GB free on the device"}
    dpg.dpg_plan_upload(plan)
    segs = segments(plan.param_offset, cfg.numels)
    g = [flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r), device=dev)
         for r in range(cfg.R)]
    w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
    param = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(plan.n_buckets, device=dev)
    tokens = token_counts(cfg)
    stream = torch.cuda.current_stream()
    state = {"t": 0}

    def step(ev):
        state["t"] += 1
        if ev is not None:
            dpg.dpg_time_next_fused_launch(*ev)
        dpg.dpg_step(plan, g, tokens, dpg.HParams(step=state["t"]), w, m, v, [param],
                     bucket_sqnorm=sq, stream=stream)

    ms, k_all = timed_cycles(step, max(3, a.steps), 3, world, dev, stream)
    peak, peak_kind = load_peak()
    bpp = algorithmic_bytes_per_param(cfg)
    out = {"config": workload_desc(cfg, cfg.cap_bytes, plan.n_buckets, N),
           "steps": max(3, a.steps), "warmup": 3, "ms_per_step": ms,
           "value": job_throughput(cfg.psi, world, ms), "unit": "params/s",
           "hbm_gbs_step": bpp["step"] * cfg.psi / (ms * 1e-3) / 1e9,
           "roofline": fused_roofline(fused_kernel_name(a, cfg.R, 1), bpp["fused"], cfg.psi, k_all,
                                      peak, peak_kind, traffic_per_launch(cfg, cfg.cap_bytes, N))}
    del g, w, m, v, param, sq
    plan.destroy()
    torch.cuda.empty_cache()
    return out


def run_secondary(a, dpg, dev, world):
    """The 4.5B accumulation workload (Llama-3-8B shapes cut to 16 layers,
    R = 4, K = 4 microbatches, 100 MiB buckets) measured in the default line:
    the whole K-microbatch cycle with one fp32 pass per microbatch (the pages'
    no_sync schedule: K - 1 accumulations, the last microbatch folded into the
    fused step), the fused step alone, and the same cycle as one deferred
    pass over K bf16 buffers per replica.  Microbatch gradients are drawn on
    the device."""
    import torch
    cfg = CONFIGS["llama8b16l"]
    R, K = cfg.R, cfg.K
    plan = dpg.dpg_plan_buckets(cfg.numels, cfg.cap_bytes, R)
    N = plan.total_padded
    torch.cuda.empty_cache()
    if not device_room(resident_bytes(cfg, N), world, dev):
        return {"skipped": f"needs {resident_bytes(cfg, N) / 1e9:.0f} GB free on the device"}
    dpg.dpg_plan_upload(plan)
    segs = segments(plan.param_offset, cfg.numels)
    tokens = token_counts(cfg)
    stream = torch.cuda.current_stream()
    peak, peak_kind = load_peak()
    grad = lambda r, k: flat_grads_bf16(segs, N, cfg.grad_std,
                                        stream_seed(cfg.seed, KIND_GRAD, r, k), device=dev)
    gd = [[grad(r, 0)] for r in range(R)]
    acc = [torch.empty(N, device=dev) for _ in range(R)]
    w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
    param = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(plan.n_buckets, device=dev)
    nf = torch.empty(plan.n_buckets, dtype=torch.int64, device=dev)
    state = {"t": 0}
    steps, warm = max(3, min(a.steps, 6)), 3

    def cycle(ev):
        # one fp32 pass per microbatch; the backward of every microbatch
        # writes the same bf16 gradient buffer of its replica
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        for k in range(K - 1):
            for r in range(R):
                dpg.dpg_accumulate(plan, gd[r][0], acc[r], first=(k == 0), stream=stream)
        if ev is not None:
            dpg.dpg_time_next_fused_launch(*ev)
        dpg.dpg_step(plan, acc, tokens, hp, w, m, v, [param], last_micro=[gd[r][0] for r in range(R)],
                     bucket_sqnorm=sq, bucket_nonfinite=nf, stream=stream)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    l0 = dpg.dpg_launch_count()
    cyc_ms, k_acc = timed_cycles(cycle, steps, warm, world, dev, stream)
    n_cycle = (dpg.dpg_launch_count() - l0) // (steps + warm)
    bpp = algorithmic_bytes_per_param(cfg)
    out = {"config": workload_desc(cfg, cfg.cap_bytes, plan.n_buckets, N),
           "steps": steps, "warmup": warm, "ms_per_step": cyc_ms,
           "value": job_throughput(cfg.psi, world, cyc_ms), "unit": "params/s",
           "hbm_gbs_step": bpp["step"] * cfg.psi / (cyc_ms * 1e-3) / 1e9,
           "cycle_bytes_per_param": bpp["step"],
           "cycle_frac": bpp["step"] * cfg.psi / (cyc_ms * 1e-3) / 1e9 / peak,
           "gpu_launches_per_cycle": int(n_cycle),
           "roofline": fused_roofline(fused_kernel_name(a, R, K), bpp["fused"], cfg.psi, k_acc,
                                      peak, peak_kind, traffic_per_launch(cfg, cfg.cap_bytes, N))}
    # deferred: every replica's K microbatches held in bf16, summed in the step
    del acc
    torch.cuda.empty_cache()
    if not device_room((K - 1) * R * N * 2, world, dev):
        out["deferred"] = {"skipped": f"needs {(K - 1) * R * N * 2 / 1e9:.0f} GB more free on "
                                      f"the device"}
        out["clocks"] = clocks.stop()
        del gd, w, m, v, param, sq, nf
        plan.destroy()
        torch.cuda.empty_cache()
        return out
    for r in range(R):
        gd[r] += [grad(r, k) for k in range(1, K)]

    def deferred(ev):
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        if ev is not None:
            dpg.dpg_time_next_fused_launch(*ev)
        dpg.dpg_step_deferred(plan, gd, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                              bucket_nonfinite=nf, stream=stream)

    d_ms, k_def = timed_cycles(deferred, steps, warm, world, dev, stream)
    bpd = algorithmic_bytes_per_param(cfg, deferred=True)
    out["deferred"] = {
        "accumulation": workload_desc(cfg, cfg.cap_bytes, plan.n_buckets, N,
                                      deferred=True)["accumulation"],
        "ms_per_step": d_ms, "value": job_throughput(cfg.psi, world, d_ms), "unit": "params/s",
        "cycle_bytes_per_param": bpd["step"],
        "cycle_frac": bpd["step"] * cfg.psi / (d_ms * 1e-3) / 1e9 / peak,
        "roofline": fused_roofline(f"k_rs_adam_chunk<R={R}> (K={K} bf16 microbatches per "
                                   f"replica)", bpd["fused"], cfg.psi, k_def, peak, peak_kind,
                                   traffic_per_launch(cfg, cfg.cap_bytes, N, deferred=True))}
    out["clocks"] = clocks.stop()
    del gd, w, m, v, param, sq, nf
    plan.destroy()
    torch.cuda.empty_cache()
    return out


def run_dpg(a):
    import torch
    import torch.distributed as dist
    rank, local, world = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from zero_optimizer_step_gb300 import build as _build
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    import zero_optimizer_step_gb300 as dpg

    cfg = config_of(a)
    cap = cap_of(cfg, a)
    R, K = cfg.R, cfg.K
    plan = dpg.dpg_plan_buckets(cfg.numels, cap, R)
    dpg.dpg_plan_upload(plan)
    N = plan.total_padded
    segs = segments(plan.param_offset, cfg.numels)
    dev = torch.device("cuda", local)
    tokens = token_counts(cfg)
    deferred = bool(a.deferred) and K >= 2
    fold2 = bool(a.fold2) and K >= 3
    # deferred accumulation keeps every microbatch: R x K distinct bf16 buffers
    gd = ([[flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r, k),
                            device=dev) for k in range(K)] for r in range(R)]
          if deferred else None)
    g = (None if deferred else
         [flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r, 0), device=dev)
          for r in range(R)])
    acc = [torch.empty(N, device=dev) for _ in range(R)] if K > 1 and not deferred else None
    # paired accumulation keeps a second bf16 gradient buffer per replica
    g2 = ([flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r, 1), device=dev)
           for r in range(R)] if fold2 else None)
    w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    m = torch.zeros(N, device=dev)
    v = torch.zeros(N, device=dev)
    param = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(plan.n_buckets, device=dev)
    nf = torch.empty(plan.n_buckets, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()
    state = {"t": 0}

    def step(ev_pair=None):
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        if deferred:
            if ev_pair is not None:
                dpg.dpg_time_next_fused_launch(*ev_pair)
            dpg.dpg_step_deferred(plan, gd, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                                  bucket_nonfinite=nf, stream=stream)
            return
        if fold2:
            for k, pair in fold2_schedule(K):
                for r in range(R):
                    if pair:
                        dpg.dpg_accumulate_pair(plan, g[r], g2[r], acc[r], first=(k == 0),
                                                stream=stream)
                    else:
                        dpg.dpg_accumulate(plan, g[r], acc[r], first=(k == 0), stream=stream)
            if ev_pair is not None:
                dpg.dpg_time_next_fused_launch(*ev_pair)
            dpg.dpg_step_fold2(plan, acc, g, g2, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                               bucket_nonfinite=nf, stream=stream)
            return
        if K > 1:
            for k in range(K - 1):
                for r in range(R):
                    dpg.dpg_accumulate(plan, g[r], acc[r], first=(k == 0), stream=stream)
        if ev_pair is not None:
            dpg.dpg_time_next_fused_launch(*ev_pair)
        if K > 1:
            dpg.dpg_step(plan, acc, tokens, hp, w, m, v, [param], last_micro=g,
                         bucket_sqnorm=sq, bucket_nonfinite=nf, stream=stream)
        elif a.variant == "staged":
            dpg.dpg_step_staged(plan, g, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                                bucket_nonfinite=nf, stream=stream)
        else:
            dpg.dpg_step(plan, g, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                         bucket_nonfinite=nf, stream=stream)

    if a.variant == "staged" and K > 1:
        raise SystemExit("--variant staged covers bf16 gradients without accumulation")
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()

    # events that bracket the fused kernel inside each timed step
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(a.steps)]
    for e0, e1 in ev_k:
        e0.record(stream)
        e1.record(stream)
    ev_start, ev_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a workload whose buffers do not dwarf the 129 MB L2 is timed step by
    # step with L2 flushed (a 256 MB write) before each step, outside its events
    flush = (torch.empty(256 << 20, dtype=torch.uint8, device=dev)
             if resident_bytes(cfg, N, fold2, deferred) < L2_FLUSH_BELOW else None)
    ev_s = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(a.steps if flush is not None else 0)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = dpg.dpg_launch_count()
    ev_start.record(stream)
    for i in range(a.steps):
        if flush is not None:
            flush.zero_()
            ev_s[i][0].record(stream)
        step(ev_k[i])
        if flush is not None:
            ev_s[i][1].record(stream)
    ev_stop.record(stream)
    torch.cuda.synchronize()
    launches = dpg.dpg_launch_count() - launches0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = (ev_start.elapsed_time(ev_stop) / a.steps if flush is None else
          statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev_s))
    k_all = sorted(e0.elapsed_time(e1) for e0, e1 in ev_k)
    k_ms = statistics.mean(k_all)
    k_pct = [k_all[int(round(q * (len(k_all) - 1)))] for q in (0.1, 0.5, 0.9)]
    ms = max_over_ranks(ms, world, dev)

    # end to end: host (pinned) gradients copied in, norms copied out, every step
    e2e = None
    if not a.no_e2e and not deferred:
        e2e = run_e2e(a, dpg, plan, g, acc, w, m, v, param, sq, nf, tokens, cfg, dev, stream,
                      state, world, fold2)

    # the 1B default line also carries the alpha-beta record and the 4.5B
    # accumulation workload, each measured after the 1B buffers are freed
    extra = {}
    if (a.config == "llama1b" and a.cap_mib is None and getattr(a, "replicas", None) is None
            and getattr(a, "microbatches", None) is None
            and a.variant == "direct" and not a.no_secondary):
        del g, gd, acc, g2, w, m, v, param, sq, nf
        torch.cuda.empty_cache()
        extra["hockney"] = optional_leg(lambda: hockney_compact(dpg), world)
        # the 10,000-tensor latency list at four caps: 2595 / 149 / 10 / 1 buckets
        extra["hockney_sweep"] = optional_leg(
            lambda: hockney_compact(dpg, name="sweep",
                                    caps=(4 << 10, 64 << 10, 1 << 20, 16 << 20)), world)
        extra["secondary"] = optional_leg(lambda: run_secondary(a, dpg, dev, world), world)
        extra["gpt2"] = optional_leg(lambda: run_gpt2_leg(a, dpg, dev, world), world)

    bpp = algorithmic_bytes_per_param(cfg, fold2, deferred)
    peak, peak_kind = load_peak()
    achieved = bpp["fused"] * cfg.psi / (k_ms * 1e-3) / 1e9
    traffic = traffic_per_launch(cfg, cap, N, fold2, deferred)
    value = job_throughput(cfg.psi, world, ms)
    line = {
        "metric": "params/s of the fused bucket reduce-scatter + Adam + all-gather step "
                  "(achieved HBM GB/s vs GB300 peak in roofline)",
        "value": value, "unit": "params/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {**workload_desc(cfg, cap, plan.n_buckets, N, fold2, deferred),
                   **({"l2": "buffers below 4 x L2: L2 flushed (256 MB write) before each timed "
                             "step, outside its events"} if flush is not None else {})},
        "hbm_gbs_step": bpp["step"] * cfg.psi / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": fused_kernel_name(a, R, K, fold2, deferred),
                     "achieved": achieved,
                     "peak": peak, "peak_kind": f"{peak_kind} (copy bandwidth)", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": bpp["fused"] * cfg.psi,
                     "kernel_ms": k_ms, "kernel_ms_p10_p50_p90": k_pct},
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": e2e,
        **extra,
    }
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_sharded(a):
    """The ZeRO-2 split across ranks, one GPU each: rank r holds replica r's
    gradient; per step the ranks exchange gradient slices, each updates its
    own shard of every bucket, and the bf16 shards are all-gathered
    (zero_optimizer_step_gb300.sharded).  value = parameters of the model
    updated per second by the whole job."""
    import torch
    import torch.distributed as dist
    rank, local, world = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    else:
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                world_size=1, device_id=dev)
    from zero_optimizer_step_gb300 import build as _build
    if rank == 0:
        _build.build()
    dist.barrier()
    import dataclasses

    import zero_optimizer_step_gb300 as dpg
    from zero_optimizer_step_gb300.sharded import ShardedStep
    cfg = dataclasses.replace(CONFIGS[a.config], R=world)
    if getattr(a, "microbatches", None) is not None:
        cfg = dataclasses.replace(cfg, K=a.microbatches)
    K = cfg.K
    cap = cap_of(cfg, a)
    plan = dpg.dpg_plan_buckets(cfg.numels, cap, world)
    N = plan.total_padded
    segs = segments(plan.param_offset, cfg.numels)
    grad = flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, rank), device=dev)
    # K > 1: every microbatch is added into an fp32 buffer on the rank, whose
    # fp32 slices are exchanged
    acc = torch.empty(N, device=dev) if K > 1 else None
    st = ShardedStep(plan, rank, world, dev, grad_dtype=torch.float32 if K > 1 else None)
    dpg.dpg_plan_upload(st.shard)
    S = st.shard.total_padded
    master = st.state_from_global(master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev))
    m, v = torch.zeros(S, device=dev), torch.zeros(S, device=dev)
    param = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(plan.n_buckets, device=dev)
    local_tokens = token_counts(cfg)[rank * K:(rank + 1) * K]
    stream = torch.cuda.current_stream()
    state = {"t": 0}

    groups = max(1, a.sharded_groups)

    def step(ev=None):
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        for k in range(K if K > 1 else 0):
            dpg.dpg_accumulate(plan, grad, acc, first=(k == 0), stream=stream)
        src = acc if K > 1 else grad
        if groups > 1:
            st.step(src, local_tokens, hp, master, m, v, param, bucket_sqnorm=sq, groups=groups)
            return
        tokens = st.all_tokens(local_tokens)
        st.exchange(src)
        if ev is not None:
            dpg.dpg_time_next_fused_launch(*ev)
        st.update(tokens, hp, master, m, v, bucket_sqnorm=sq, stream=stream)
        st.allgather(param)

    ms, k_all = timed_cycles(step, a.steps, a.warmup, world, dev, stream)
    k_all = [max_over_ranks(x, world, dev) for x in k_all]
    peak, peak_kind = load_peak()
    bpp = (4 if K > 1 else 2) * world + 26
    line = {"metric": "params/s of the fused bucket reduce-scatter + Adam + all-gather step "
                      "(achieved HBM GB/s vs GB300 peak in roofline)",
            "value": cfg.psi / (ms * 1e-3), "unit": "params/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {**workload_desc(cfg, cap, plan.n_buckets, N),
                       **({"accumulation": "every microbatch added into the rank's fp32 "
                                           "buffer, then its fp32 slices exchanged"}
                          if K > 1 else {}),
                       "sharded": "ZeRO-2 split: rank r owns shard r of every bucket; NCCL "
                                  "point-to-point exchange of " +
                                  ("fp32 slices of the rank's K-microbatch accumulator"
                                   if K > 1 else "bf16 gradient slices") +
                                  ", the fused update of the rank's shard, NCCL all-gather of "
                                  "bf16 shards",
                       "shard_elements_per_rank": S},
            "roofline": (fused_roofline(f"k_rs_adam_chunk<R={world}> on the rank's shard", bpp,
                                        S, k_all, peak, peak_kind, None) if groups == 1 else
                         None)}
    if groups > 1:
        line["config"]["pipelined_groups"] = len(st.bucket_groups(groups))
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.barrier()
    dist.destroy_process_group()


def host_mem_available() -> int:
    """MemAvailable of /proc/meminfo in bytes (0 if unknown)."""
    try:
        for ln in open("/proc/meminfo"):
            if ln.startswith("MemAvailable:"):
                return int(ln.split()[1]) * 1024
    except OSError:
        pass
    return 0


def run_e2e(a, dpg, plan, g, acc, w, m, v, param, sq, nf, tokens, cfg, dev, stream, state, world,
            fold2=False):
    import torch
    R, K = cfg.R, cfg.K
    N = plan.total_padded
    # one pinned host staging buffer per replica, the source of every
    # microbatch's copy (R*K copies of N bf16 elements per step); when the
    # ranks of this node could not pin that much without crowding the host,
    # every replica reads the same pinned buffer (the same bytes cross the
    # link either way)
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    distinct = R * N * 2 * local_world <= host_mem_available() // 2
    n_host = R if distinct else 1
    h_rep = [torch.empty(N, dtype=torch.bfloat16, pin_memory=True) for _ in range(n_host)]
    for r in range(n_host):
        h_rep[r].copy_(g[r])
    h_rep = h_rep * (R // n_host)
    h_in = [[h_rep[r]] * K for r in range(R)]
    h_sq = torch.empty(plan.n_buckets, pin_memory=True)
    h_nf = torch.empty(plan.n_buckets, dtype=torch.int64, pin_memory=True)

    # K == 1: the copies are cut into chunks of whole buckets on a copy stream;
    # each chunk's fused update starts as soon as its gradients have landed
    n_chunks = min(plan.n_buckets, 16)
    bounds = [0]
    if K == 1:
        ends = plan.bucket_offset + plan.bucket_padded
        for c in range(1, n_chunks):
            bounds.append(int(np.searchsorted(ends, N * c / n_chunks)) + 1)
        bounds.append(plan.n_buckets)
        bounds = sorted(set(min(b, plan.n_buckets) for b in bounds))
    copy_stream = torch.cuda.Stream()

    def e2e_step_pipelined():
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        copy_stream.wait_stream(stream)
        for b0, b1 in zip(bounds[:-1], bounds[1:]):
            lo = int(plan.bucket_offset[b0])
            hi = int(plan.bucket_offset[b1 - 1] + plan.bucket_padded[b1 - 1])
            with torch.cuda.stream(copy_stream):
                for r in range(R):
                    g[r][lo:hi].copy_(h_in[r][0][lo:hi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
            stream.wait_event(ev)
            dpg.dpg_reduce_scatter_adam(plan, g, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                                        bucket_nonfinite=nf, b0=b0, b1=b1, stream=stream)
        h_sq.copy_(sq, non_blocking=True)
        h_nf.copy_(nf, non_blocking=True)

    def e2e_step():
        if K == 1:
            return e2e_step_pipelined()
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        for k in range(K):
            for r in range(R):
                g[r].copy_(h_in[r][k], non_blocking=True)
            if k < K - 1:
                for r in range(R):
                    dpg.dpg_accumulate(plan, g[r], acc[r], first=(k == 0), stream=stream)
        if K > 1:
            dpg.dpg_step(plan, acc, tokens, hp, w, m, v, [param], last_micro=g, bucket_sqnorm=sq,
                         bucket_nonfinite=nf, stream=stream)
        else:
            dpg.dpg_step(plan, g, tokens, hp, w, m, v, [param], bucket_sqnorm=sq,
                         bucket_nonfinite=nf, stream=stream)
        h_sq.copy_(sq, non_blocking=True)
        h_nf.copy_(nf, non_blocking=True)

    def e2e_step_zero_copy():
        # the kernels read the pinned host gradients in place over the host link
        state["t"] += 1
        hp = dpg.HParams(step=state["t"])
        if fold2:
            for k, pair in fold2_schedule(K):
                for r in range(R):
                    if pair:
                        dpg.dpg_accumulate_pair(plan, h_in[r][k], h_in[r][k + 1], acc[r],
                                                first=(k == 0), stream=stream)
                    else:
                        dpg.dpg_accumulate(plan, h_in[r][k], acc[r], first=(k == 0),
                                           stream=stream)
            dpg.dpg_step_fold2(plan, acc, [h_in[r][K - 2] for r in range(R)],
                               [h_in[r][K - 1] for r in range(R)], tokens, hp, w, m, v, [param],
                               bucket_sqnorm=sq, bucket_nonfinite=nf, stream=stream)
            h_sq.copy_(sq, non_blocking=True)
            h_nf.copy_(nf, non_blocking=True)
            return
        for k in range(K - 1):
            for r in range(R):
                dpg.dpg_accumulate(plan, h_in[r][k], acc[r], first=(k == 0), stream=stream)
        if K > 1:
            dpg.dpg_step(plan, acc, tokens, hp, w, m, v, [param],
                         last_micro=[h_in[r][K - 1] for r in range(R)], bucket_sqnorm=sq,
                         bucket_nonfinite=nf, stream=stream)
        else:
            dpg.dpg_step(plan, [h_in[r][0] for r in range(R)], tokens, hp, w, m, v, [param],
                         bucket_sqnorm=sq, bucket_nonfinite=nf, stream=stream)
        h_sq.copy_(sq, non_blocking=True)
        h_nf.copy_(nf, non_blocking=True)

    steps = max(3, min(a.steps, 10))

    def time_mode(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / steps, world, dev)

    how = {
        "zero_copy": "the kernels read the pinned host gradients in place over the host link "
                     "(unified addressing; no staging copy)" + ("" if K == 1 else
                     ", paired accumulations then the fused step with the last two microbatches"
                     if fold2 else
                     ", K-1 accumulations then the fused step with the last microbatch") +
                     "; norms read back",
        "copy": (f"pinned host gradients copied in {len(bounds) - 1} bucket chunks on a copy "
                 f"stream, each chunk's fused update overlapping the next chunk's copy; "
                 f"norms read back" if K == 1 else
                 "pinned host gradients copied in per microbatch, accumulated, fused step; "
                 "norms read back"),
    }
    modes = {"zero_copy": time_mode(e2e_step_zero_copy)}
    if not fold2:
        modes["copy"] = time_mode(e2e_step)
    best = min(modes, key=modes.get)
    ms = modes[best]
    return {"value": job_throughput(cfg.psi, world, ms), "unit": "params/s", "steps": steps,
            "host_buffers": "one pinned buffer per replica" if distinct else
                            "one pinned buffer shared by the replicas (host memory bound)",
            "h2d_bytes_per_step": R * K * N * 2, "d2h_bytes_per_step": plan.n_buckets * 12,
            "ms_per_step": ms, "h2d_gbs": R * K * N * 2 / (ms * 1e-3) / 1e9,
            "mode": best, "how": how[best],
            "ms_per_step_by_mode": modes}


# --------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# --------------------------------------------------------------------------
def reference_sample_fields(cfg, n: int) -> dict:
    """What one timed step of the reference arm covers: a contiguous n-element
    sample of the workload (one full oracle step over the 1B list takes about
    20 s on one host core)."""
    return {"timed_per_step": f"a contiguous sample of {n} elements of the workload's inputs",
            "sample_elems_per_step": int(n), "sample_share_of_psi": n / cfg.psi}


def run_reference(a):
    rank, _, world = dist_info()
    if rank != 0:
        return
    cfg = config_of(a)
    cap = cap_of(cfg, a)
    import oracle
    oracle.build()
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except (AttributeError, OSError):
        pass
    n = a.cpu_sample_elems
    grads, last, w, m, v = cpu_sample_inputs(cfg, n, "cpu")
    tokens = token_counts(cfg)
    t = 0
    for _ in range(a.warmup):
        t += 1
        oracle_sample_step(cfg, grads, last, tokens, w, m, v, t)
    t0 = time.perf_counter()
    for _ in range(a.steps):
        t += 1
        oracle_sample_step(cfg, grads, last, tokens, w, m, v, t)
    dt = (time.perf_counter() - t0) / a.steps
    value = n / dt
    plan = oracle.plan_buckets(cfg.numels, cap, cfg.R)
    sample = (f"each step: oracle reduce+scale+Adam+bf16 cast over the first {n} elements of the "
              f"workload, one pinned host core")
    config = workload_desc(cfg, cap, plan.n_buckets, plan.total_padded)
    config.update(reference_sample_fields(cfg, n))
    line = {"metric": "params/s of the fused bucket reduce-scatter + Adam + all-gather step "
                      "(achieved HBM GB/s vs GB300 peak in roofline)",
            "value": value, "unit": "params/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": cfg.psi / value * 1e3,
            "ms_per_step_basis": "the full workload's step time at the rate the timed sample "
                                 "ran (the oracle step is elementwise); psi / value",
            "sample_ms_per_step": dt * 1e3, "timed_s": dt * a.steps,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config,
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                             "host": host_cpu(), "sample": sample},
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# Hockney alpha-beta sweep ("Parallelisms", section "Gradient bucketing":
# T(m) = alpha + beta m; K small operations cost K alpha + beta M, one fused
# operation alpha + beta M)
# --------------------------------------------------------------------------
def hockney_points(dpg, cfg, caps, reps, modes=("per_bucket", "per_bucket_plain", "fused")):
    """For each bucket cap: the step's fused update over the whole plan as one
    launch per bucket and as one launch over all buckets, each replayed from a
    CUDA graph with L2 flushed before every replay (median ms)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    R = cfg.R
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (129 MB)
    points = []
    for cap in caps:
        plan = dpg.dpg_plan_buckets(cfg.numels, cap, R)
        dpg.dpg_plan_upload(plan)
        N = plan.total_padded
        segs = segments(plan.param_offset, cfg.numels)
        g = [flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r), device=dev)
             for r in range(R)]
        w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
        m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
        p = torch.empty(N, dtype=torch.bfloat16, device=dev)
        tok = token_counts(cfg)
        hp = dpg.HParams(step=1)
        graphs = {}
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):     # warm the occupancy cache and the plan upload
                dpg.dpg_reduce_scatter_adam(plan, g, tok, hp, w, m, v, [p])
        torch.cuda.current_stream().wait_stream(s)
        # per_bucket: launches with programmatic stream serialization (the
        # library's default); per_bucket_plain: the same launches without it
        for mode in modes:
            gr = torch.cuda.CUDAGraph()
            dpg.dpg_set_programmatic_launch(mode != "per_bucket_plain")
            try:
                with torch.cuda.graph(gr):
                    if mode == "fused":
                        dpg.dpg_reduce_scatter_adam(plan, g, tok, hp, w, m, v, [p])
                    else:
                        for b in range(plan.n_buckets):
                            dpg.dpg_reduce_scatter_adam(plan, g, tok, hp, w, m, v, [p],
                                                        b0=b, b1=b + 1)
            finally:
                dpg.dpg_set_programmatic_launch(True)
            graphs[mode] = gr
        pt = {"cap_bytes": cap, "n_buckets": plan.n_buckets, "total_padded": N,
              "bytes": (2 * R + 26) * cfg.psi}
        for mode, gr in graphs.items():
            ts = []
            for _ in range(max(3, reps)):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                gr.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            pt[mode + "_ms"] = statistics.median(ts)
            pt[mode + "_ms_range"] = [min(ts), max(ts)]
        points.append(pt)
        del graphs, g, w, m, v, p
        plan.destroy()
    torch.cuda.empty_cache()
    return points


def hockney_fit(points, key="per_bucket"):
    """Least squares T = K*alpha + beta*M over the points (K launches moving M
    bytes in all): alpha in us, 1/beta in GB/s."""
    K = np.array([q["n_buckets"] for q in points], float)
    Mb = np.array([q["bytes"] for q in points], float)
    T = np.array([q[key + "_ms"] for q in points], float) * 1e-3
    (alpha, beta), *_ = np.linalg.lstsq(np.stack([K, Mb], axis=1), T, rcond=None)
    return {"alpha_us": alpha * 1e6, "inv_beta_gbs": 1.0 / beta / 1e9}


def run_hockney(a):
    import torch
    from zero_optimizer_step_gb300 import build as _build
    _build.build()
    import zero_optimizer_step_gb300 as dpg
    cfg = CONFIGS[a.hockney_config]
    torch.cuda.set_device(torch.device("cuda", 0))
    points = hockney_points(dpg, cfg, cfg.cap_sweep, a.steps)
    fused = np.array([q["fused_ms"] for q in points]) * 1e-3
    out = {"metric": "hockney alpha-beta fit of the fused reduce-scatter+Adam kernel over bucket caps",
           "workload": f"{cfg.name}: {len(cfg.shapes)} tensors, psi={cfg.psi}, R={cfg.R}",
           "points": points, "fit": {**hockney_fit(points, "per_bucket"),
                                     "plain_launches": hockney_fit(points, "per_bucket_plain"),
                                     "model": "T_per_bucket = K*alpha + beta*M (least squares)"},
           "fused_single_launch_ms": {"median": float(np.median(fused)) * 1e3,
                                      "min": float(fused.min()) * 1e3, "max": float(fused.max()) * 1e3},
           "timing": "CUDA graph replay, L2 flushed (256 MB write) before every replay"}
    print(json.dumps(out), flush=True)


def run_launch_floor(a):
    """Single fused launches (no norm) over one bucket of n elements, R = 8,
    for n from 1M to 128M elements: least squares T = T0 + bytes / B over the
    sizes from 4M up gives the fixed cost T0 of a launch (start-up of the
    first CTAs, the drain of the last) and its streaming bandwidth B."""
    import torch
    from zero_optimizer_step_gb300 import build as _build
    _build.build()
    import zero_optimizer_step_gb300 as dpg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    R = 8
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    sizes = [1 << 20, 2 << 20, CONFIGS["sweep"].psi, 8 << 20, 16 << 20, 32 << 20, 64 << 20,
             128 << 20]
    rows = []
    for n in sizes:
        plan = dpg.dpg_plan_buckets([n], 2 * n + 1024, R)
        dpg.dpg_plan_upload(plan)
        N = plan.total_padded
        g = [flat_grads_bf16([(0, n)], N, 1e-3, stream_seed(7, KIND_GRAD, r), device=dev)
             for r in range(R)]
        w = master_f32(N, stream_seed(7, KIND_MASTER), device=dev)
        m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
        p = torch.empty(N, dtype=torch.bfloat16, device=dev)
        tok = [3500] * R
        hp = dpg.HParams(step=1)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):
                dpg.dpg_reduce_scatter_adam(plan, g, tok, hp, w, m, v, [p])
        torch.cuda.current_stream().wait_stream(s)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            dpg.dpg_reduce_scatter_adam(plan, g, tok, hp, w, m, v, [p])
        ts = []
        for _ in range(max(5, a.steps)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.median(ts)
        rows.append({"elements": n, "bytes": (2 * R + 26) * n, "ms": ms,
                     "gbs": (2 * R + 26) * n / (ms * 1e-3) / 1e9})
        del gr, g, w, m, v, p
        plan.destroy()
        torch.cuda.empty_cache()
    big = [q for q in rows if q["elements"] >= 4 << 20]
    A = np.stack([np.ones(len(big)), [q["bytes"] for q in big]], axis=1)
    (t0, inv_b), *_ = np.linalg.lstsq(A, np.array([q["ms"] * 1e-3 for q in big]), rcond=None)
    peak, peak_kind = load_peak()
    for q in rows:
        q["frac"] = q["gbs"] / peak
    print(json.dumps({"metric": "fixed cost of one fused reduce-scatter+Adam launch",
                      "R": R, "rows": rows,
                      "fit": {"t0_us": t0 * 1e6, "bandwidth_gbs": 1.0 / inv_b / 1e9,
                              "model": "T = T0 + bytes / B, least squares over n >= 4M"},
                      "peak_gbs": peak, "peak_kind": peak_kind,
                      "timing": "median CUDA graph replay, L2 flushed (256 MB write) before each"}),
          flush=True)


def hockney_compact(dpg, reps=5, name="llama1b", caps=None):
    """The alpha-beta record of the default line: a list at a few caps (the 1B
    list at its three, 1 / 25 / 100 MiB), one launch per bucket against one
    launch in all."""
    cfg = CONFIGS[name]
    caps = cfg.cap_sweep if caps is None else caps
    points = hockney_points(dpg, cfg, caps, reps, modes=("per_bucket", "fused"))
    return {"workload": f"{cfg.name}: psi={cfg.psi}, R={cfg.R}, caps "
                        + "/".join(f"{c / (1 << 20):g}" for c in caps) + " MiB",
            "model": "T_per_bucket = K*alpha + beta*M (least squares; K launches, M bytes)",
            "fit": hockney_fit(points, "per_bucket"),
            "points": [{"cap_mib": q["cap_bytes"] / (1 << 20), "n_buckets": q["n_buckets"],
                        "per_bucket_ms": q["per_bucket_ms"], "fused_ms": q["fused_ms"]}
                       for q in points],
            "timing": f"median of {max(3, reps)} CUDA graph replays per point, programmatic "
                      f"launches, L2 flushed before each"}


# --------------------------------------------------------------------------
# per-kernel table: each kernel of the path timed alone on the workload
# --------------------------------------------------------------------------
def run_kernel_table(a):
    import torch
    from zero_optimizer_step_gb300 import build as _build
    _build.build()
    import zero_optimizer_step_gb300 as dpg
    cfg = config_of(a)
    cap = cap_of(cfg, a)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    R = cfg.R
    plan = dpg.dpg_plan_buckets(cfg.numels, cap, R)
    dpg.dpg_plan_upload(plan)
    N = plan.total_padded
    segs = segments(plan.param_offset, cfg.numels)
    psi = cfg.psi
    peak, peak_kind = load_peak()
    g = [flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r), device=dev)
         for r in range(R)]
    w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
    p = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(plan.n_buckets, device=dev)
    acc = torch.empty(N, device=dev)
    tok = token_counts(cfg)
    # parameter-shaped gradients for pack/unpack (one replica)
    pgrads = [g[0][int(o):int(o) + int(n)].clone() for o, n in zip(plan.param_offset, cfg.numels)]
    flat = torch.empty(N, dtype=torch.bfloat16, device=dev)
    state = {"t": 0}

    def hp():
        state["t"] += 1
        return dpg.HParams(step=state["t"])

    def plain_launches(fn):
        dpg.dpg_set_programmatic_launch(False)
        try:
            fn()
        finally:
            dpg.dpg_set_programmatic_launch(True)

    cases = [
        ("k_pack (dpg_pack, one replica)", 4, lambda: dpg.dpg_pack(plan, pgrads, flat)),
        ("k_pack unpack (dpg_unpack, one replica)", 4, lambda: dpg.dpg_unpack(plan, flat, pgrads)),
        ("k_accumulate<first> (one replica)", 6, lambda: dpg.dpg_accumulate(plan, g[0], acc, True)),
        ("k_accumulate (one replica)", 10, lambda: dpg.dpg_accumulate(plan, g[0], acc, False)),
        ("k_accumulate_pair<first> (one replica)", 8,
         lambda: dpg.dpg_accumulate_pair(plan, g[0], g[1 % R], acc, True)),
        ("k_accumulate_pair (one replica)", 12,
         lambda: dpg.dpg_accumulate_pair(plan, g[0], g[1 % R], acc, False)),
        ("k_allgather (one view)", 6, lambda: dpg.dpg_allgather_params(plan, w, [p])),
        (f"k_rs_adam_chunk<R={R}> (dpg_reduce_scatter_adam, no norm)", 2 * R + 26,
         lambda: dpg.dpg_reduce_scatter_adam(plan, g, tok, hp(), w, m, v, [p])),
        (f"k_rs_adam_chunk<R={R}> + k_chunk_finalize (dpg_step)", 2 * R + 26,
         lambda: dpg.dpg_step(plan, g, tok, hp(), w, m, v, [p], bucket_sqnorm=sq)),
        (f"k_rs_adam_staged<R={R}> (dpg_step_staged, bulk-copy staging)", 2 * R + 26,
         lambda: dpg.dpg_step_staged(plan, g, tok, hp(), w, m, v, [p], bucket_sqnorm=sq)),
        (f"k_rs_adam_chunk<R={R}> distinct views (n_views=R)", 4 * R + 24,
         lambda: dpg.dpg_step(plan, g, tok, hp(), w, m, v, views)),
        ("dpg_step_clipped, g stored (norm pass + update pass)", 2 * R + 34,
         lambda: dpg.dpg_step_clipped(plan, g, tok, hp(), 1e-6, w, m, v, [p], reduced_grad=acc)),
        ("dpg_step_clipped, replicas re-read", 4 * R + 26,
         lambda: dpg.dpg_step_clipped(plan, g, tok, hp(), 1e-6, w, m, v, [p])),
        ("k_gather_bf16 (dpg_gather_params_bf16, one view, one launch)", 4,
         lambda: dpg.dpg_gather_params_bf16(plan, p, views[:1])),
        (f"k_gather_bf16 (dpg_gather_params_bf16, {R} views, one launch)", 2 + 2 * R,
         lambda: dpg.dpg_gather_params_bf16(plan, p, views)),
        (f"k_gather_bf16 ({R} views, one launch per bucket)", 2 + 2 * R,
         lambda: [dpg.dpg_gather_params_bf16(plan, p, views, b0=b, b1=b + 1)
                  for b in range(plan.n_buckets)]),
        (f"k_gather_bf16 ({R} views, one launch per bucket, plain launches)", 2 + 2 * R,
         lambda: plain_launches(lambda: [dpg.dpg_gather_params_bf16(plan, p, views, b0=b, b1=b + 1)
                                         for b in range(plan.n_buckets)])),
        # calibration (torch's own kernels, not this library): the mix of reads
        # and writes sets the ceiling; the denominator is a 1:1 copy
        ("calibration: torch fill_ (write only, 4 B/param)", 4, lambda: acc.fill_(0.5)),
        ("calibration: torch copy_ (fp32 1:1 copy, 8 B/param)", 8, lambda: acc.copy_(w)),
        ("calibration: torch sum (read only, 4 B/param)", 4, lambda: torch.sum(w)),
        ("calibration: torch add (2 reads : 1 write, 12 B/param)", 12,
         lambda: torch.add(w, m, out=acc)),
    ]
    views = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    rows = []
    for name, bpp, fn in cases:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ms = statistics.median(device_times_ms(fn, max(5, min(a.steps, 20))))
        gbs = bpp * psi / (ms * 1e-3) / 1e9
        rows.append({"kernel": name, "bytes_per_param": bpp, "ms": ms, "achieved_gbs": gbs,
                     "frac": gbs / peak})
    print(json.dumps({"metric": "per-kernel HBM roofline", "config": workload_desc(cfg, cap, plan.n_buckets, N),
                      "peak_gbs": peak, "peak_kind": peak_kind, "rows": rows,
                      "timing": "median of CUDA-event intervals around one call each, a GPU spin "
                                "queued before the start event so that the host's call overhead "
                                "is not in the interval; no L2 flush (every operand > L2)"}),
          flush=True)


# --------------------------------------------------------------------------
# DDP against ZeRO-1/2 ("Parallelisms" -- ZeRO-1, ZeRO-2, FSDP NO_SHARD)
# --------------------------------------------------------------------------
def run_schedules(a):
    import torch
    from zero_optimizer_step_gb300 import build as _build
    _build.build()
    import zero_optimizer_step_gb300 as dpg
    cfg = config_of(a)
    cap = cap_of(cfg, a)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    R, psi = cfg.R, cfg.psi
    plan = dpg.dpg_plan_buckets(cfg.numels, cap, R)
    dpg.dpg_plan_upload(plan)
    N = plan.total_padded
    segs = segments(plan.param_offset, cfg.numels)
    g = [flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r), device=dev)
         for r in range(R)]
    tok = token_counts(cfg)[:R]
    w0 = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    peak, peak_kind = load_peak()
    state = {"t": 0}

    def hp():
        state["t"] += 1
        return dpg.HParams(step=state["t"])

    def timed(fn, reps=7):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        return statistics.median(device_times_ms(fn, reps))

    rows = []
    z = [w0.clone(), torch.zeros(N, device=dev), torch.zeros(N, device=dev)]
    zp = torch.empty(N, dtype=torch.bfloat16, device=dev)
    ms = timed(lambda: dpg.dpg_step(plan, g, tok, hp(), *z, [zp]))
    for name, mem in (("ZeRO-2", 2 + 14 / R), ("ZeRO-1", 4 + 12 / R)):
        rows.append({"schedule": name, "ms": ms, "bytes_per_param": 2 * R + 26,
                     "achieved_gbs": (2 * R + 26) * psi / (ms * 1e-3) / 1e9,
                     "model_state_bytes_per_param_per_replica": mem,
                     "note": "same fused pass; ZeRO-1 also keeps the full bf16 gradients"})
    del z
    reps = [[w0.clone(), torch.zeros(N, device=dev), torch.zeros(N, device=dev)] for _ in range(R)]
    rp = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    red = torch.empty(N, device=dev)

    def ddp():
        h = hp()
        dpg.dpg_allreduce_grads(plan, g, tok, red)
        for r in range(R):
            dpg.dpg_adam_from_reduced(plan, red, h, *reps[r], [rp[r]])

    ms = timed(ddp)
    bpp = 2 * R + 4 + R * 30
    rows.append({"schedule": "DDP (NO_SHARD)", "ms": ms, "bytes_per_param": bpp,
                 "achieved_gbs": bpp * psi / (ms * 1e-3) / 1e9,
                 "model_state_bytes_per_param_per_replica": 16,
                 "note": "all-reduce, then each of the R replicas updates its own full state"})
    del reps
    # ZeRO-3: the step writes only the sharded bf16 parameters; every layer is
    # all-gathered from the shards before forward and again before backward
    z = [w0.clone(), torch.zeros(N, device=dev), torch.zeros(N, device=dev)]
    shards = torch.empty(N, dtype=torch.bfloat16, device=dev)
    ms_step = timed(lambda: dpg.dpg_step(plan, g, tok, hp(), *z, [shards]))

    def gathers():
        for _ in range(2):
            for b in range(plan.n_buckets):
                dpg.dpg_gather_params_bf16(plan, shards, rp, b0=b, b1=b + 1)

    ms_gather = timed(gathers)
    bpp = 2 * R + 26 + 2 * (2 + 2 * R)
    rows.append({"schedule": "ZeRO-3", "ms": ms_step + ms_gather, "ms_step": ms_step,
                 "ms_gathers": ms_gather, "bytes_per_param": bpp,
                 "achieved_gbs": bpp * psi / ((ms_step + ms_gather) * 1e-3) / 1e9,
                 "gather_gbs": 2 * (2 + 2 * R) * psi / (ms_gather * 1e-3) / 1e9,
                 "model_state_bytes_per_param_per_replica": 16 / R,
                 "note": "same fused pass writing one sharded bf16 buffer, then two "
                         "layer-by-layer parameter all-gathers (forward, backward)"})
    print(json.dumps({"metric": "DDP vs ZeRO-1/2/3 schedules", "config": workload_desc(cfg, cap, plan.n_buckets, N),
                      "peak_gbs": peak, "peak_kind": peak_kind, "rows": rows,
                      "timing": "median of CUDA-event intervals around one call each, a GPU spin "
                                "queued before the start event"}), flush=True)


# --------------------------------------------------------------------------
# Overlap of bucket updates with backward ("Parallelisms" -- Critical path,
# Gradient bucketing; "Distributed Training and Parallelism" -- DDP buckets:
# small buckets start early but pay more startup, large ones leave a tail)
# --------------------------------------------------------------------------
def make_gemm_backward(cfg, plan, grad0, weight, tokens, dev):
    """A stand-in backward made of real GEMMs: for every weight, in
    backward-ready order, dW = dY^T X written straight into replica 0's flat
    gradient slice (gradients produced in the communication buffers) and
    dX = dY W into scratch; 1-D weights get a token reduction.  Returns a
    function that issues bucket b's work on the current stream."""
    import torch
    shapes = [tuple(s) for _, s in cfg.shapes]
    rows = max(s[0] for s in shapes)
    cols = max(s[-1] for s in shapes)
    gen = torch.Generator(device=dev).manual_seed(7)
    dy_all = (torch.randn(tokens, rows, device=dev, generator=gen) * 1e-3).to(torch.bfloat16)
    x_all = torch.randn(tokens, cols, device=dev, generator=gen).to(torch.bfloat16)
    dx_flat = torch.empty(tokens * cols, dtype=torch.bfloat16, device=dev)
    by_bucket = [[] for _ in range(plan.n_buckets)]
    for q in range(len(shapes) - 1, -1, -1):            # backward-ready order
        if shapes[q] and math.prod(shapes[q]) > 0:
            by_bucket[int(plan.param_bucket[q])].append(q)

    def run(b):
        for q in by_bucket[b]:
            off = int(plan.param_offset[q])
            shp = shapes[q]
            if len(shp) == 2:
                o, i = shp
                dw = grad0[off:off + o * i].view(o, i)
                torch.mm(dy_all[:, :o].t(), x_all[:, :i], out=dw)
                torch.mm(dy_all[:, :o], weight[off:off + o * i].view(o, i),
                         out=dx_flat[:tokens * i].view(tokens, i))
            else:
                n = int(math.prod(shp))
                grad0[off:off + n].copy_((dy_all[:, :n].float() * x_all[:, :n].float()).sum(0))
    return run


def run_overlap(a):
    import torch
    from zero_optimizer_step_gb300 import build as _build
    _build.build()
    import zero_optimizer_step_gb300 as dpg
    cfg = config_of(a)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    R, psi = cfg.R, cfg.psi
    sm_mhz = 2070.0       # the spin kernel counts SM clocks; the measured time is reported
    caps = [int(float(c) * (1 << 20)) for c in a.overlap_caps_mib.split(",")]
    grid_caps = [int(x) for x in a.overlap_max_ctas.split(",")]
    rows = []
    lo_pri, hi_pri = torch.cuda.Stream.priority_range()   # (lowest, greatest)
    bwd_stream = torch.cuda.Stream(priority=hi_pri if a.backward_priority else 0)
    upd_stream = torch.cuda.Stream(priority=lo_pri if a.backward_priority else 0)
    for cap in caps:
        plan = dpg.dpg_plan_buckets(cfg.numels, cap, R)
        dpg.dpg_plan_upload(plan)
        N = plan.total_padded
        segs = segments(plan.param_offset, cfg.numels)
        g = [flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r), device=dev)
             for r in range(R)]
        w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
        m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
        p = torch.empty(N, dtype=torch.bfloat16, device=dev)
        tok = token_counts(cfg)[:R]
        # backward of bucket b takes a share of the backward time proportional
        # to its parameters; buckets are produced in plan order (last layers first)
        cycles = [int(a.backward_ms * 1e3 * sm_mhz * float(pb) / N) for pb in plan.bucket_padded]
        gemm_bucket = make_gemm_backward(cfg, plan, g[0], p, a.tokens, dev) \
            if a.backward_kind == "gemm" else None

        def one(overlap: bool):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            eb = torch.cuda.Event(enable_timing=True)
            eu = torch.cuda.Event(enable_timing=True)
            e0.record(bwd_stream)
            upd_stream.wait_event(e0)
            evs = []
            with torch.cuda.stream(bwd_stream):
                for b in range(plan.n_buckets):
                    if gemm_bucket is None:
                        torch.cuda._sleep(cycles[b])
                    else:
                        gemm_bucket(b)
                    ev = torch.cuda.Event()
                    ev.record(bwd_stream)
                    evs.append(ev)
            eb.record(bwd_stream)
            if not overlap:
                upd_stream.wait_event(eb)
            # bucket b's update waits on its ready event, issued by the library
            dpg.dpg_reduce_scatter_adam_when_ready(plan, g, tok, dpg.HParams(step=1), w, m, v, [p],
                                                   ready_events=evs, stream=upd_stream)
            eu.record(upd_stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(eb), e0.elapsed_time(eu)

        for gc in grid_caps:
            dpg.dpg_set_fused_max_ctas(gc)
            try:
                one(True)
                res = {}
                for mode in (True, False):
                    ts = sorted(one(mode) for _ in range(5))
                    res[mode] = ts[len(ts) // 2]
            finally:
                dpg.dpg_set_fused_max_ctas(0)
            bwd, tot = res[True]
            _, serial = res[False]
            bwd_alone = res[False][0]
            rows.append({"cap_bytes": cap, "n_buckets": plan.n_buckets, "fused_max_ctas": gc,
                         "backward_ms": bwd_alone, "backward_ms_overlapped": bwd,
                         "overlapped_total_ms": tot, "exposed_tail_ms": tot - bwd,
                         "serial_total_ms": serial, "update_alone_ms": serial - bwd_alone,
                         "saved_vs_serial_ms": serial - tot})
        del g, w, m, v, p, gemm_bucket
        plan.destroy()
    backward = (f"{a.backward_ms} ms of spin kernels (one CTA), split over buckets in proportion "
                f"to their parameters, in backward-ready order" if a.backward_kind == "spin" else
                f"bf16 GEMMs per weight in backward-ready order: dW = dY^T X written into replica "
                f"0's flat gradient slice, dX = dY W, {a.tokens} tokens (4 * tokens * psi flops); "
                f"the other replicas' gradients are resident synthetic data")
    print(json.dumps({"metric": "exposed update tail behind a simulated backward",
                      "workload": f"{cfg.name}: psi={psi}, R={R}", "backward": backward,
                      "streams": "backward high priority, updates low" if a.backward_priority
                                 else "equal priority",
                      "rows": rows}), flush=True)


def main():
    a = parse()
    if a.overlap:
        run_overlap(a)
        return
    if a.traffic_from:
        write_traffic(a)
        return
    if a.schedules:
        run_schedules(a)
        return
    if a.kernels:
        run_kernel_table(a)
        return
    if a.hockney:
        run_hockney(a)
        return
    if a.launch_floor:
        run_launch_floor(a)
        return
    if a.impl == "reference":
        run_reference(a)
    elif a.sharded:
        run_sharded(a)
    else:
        run_dpg(a)


if __name__ == "__main__":
    main()
