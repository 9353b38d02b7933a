#!/usr/bin/env python
"""Bench of the resident brute-force top-K search on one GPU.

Headline workload: N = 1,000,000 corpus rows, D = 1024, fp32, unit-norm
Gaussian rows (seed 1), 1,000 unit-norm queries (seed 2), 10 planted
near-duplicates per query (seed 3), inner product, K = 8, with K = 32 and
K = 100 timed in their own regions. One step = one query = one launch of the
fused scoring kernel (scores, per-CTA selection, and the merge in its last
CTA). The corpus (4.1 GB) is larger than L2, so no flush is needed.

Prints one JSON line. ``value`` is the achieved corpus-read rate in GB/s over
the K = 8 timed steps (algorithmic bytes N*D*4 per step / device time). The
line also carries the other workloads of the configuration table, each in its
own block: ``config1`` (10k x 384, K = 8, 16 queries), ``sweep`` (the pages'
N x D x K grid, 200 queries per cell), ``batched`` / ``batched_tf32``
(256 queries x 1M x 768 on the tensor cores), ``int32`` (1e8 values, K = 20
and 50), ``cosine`` and ``views``.

--impl reference times the oracle (the CPU reference of this tier) on the
same workload, whole queries over all rows, on the host cores.

--case NAME runs one small workload for a profiler capture instead (see
run_case: single, small, batch, batch_full, int32).

Under torchrun (N > 1 ranks) every rank holds one contiguous row shard of a
corpus N times as large and a step is a sharded search: the local search, an
exchange of the K best (index, score) pairs of every shard, and the merge of
the N lists on every rank.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "search p50 µs & achieved HBM GB/s (vs 8 TB/s) at N=1M D=1024 K=8/32/100"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("single-query resident search: N=1,000,000 x D=1024 fp32 unit-norm Gaussian corpus "
            "(4.1 GB resident), 1,000 queries with 10 planted near-duplicates each, inner product, K=8")
SWEEP_N = (10_000, 50_000, 100_000, 500_000, 1_000_000)
SWEEP_D = (384, 768, 1024)
SWEEP_K = (8, 32, 100)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--n", type=int, default=1_000_000)
    ap.add_argument("--d", type=int, default=1024)
    ap.add_argument("--queries", type=int, default=1000)
    ap.add_argument("--extra-k", default="32,100")
    ap.add_argument("--sweep-queries", type=int, default=200)
    ap.add_argument("--case", default=None, help="run one profiling case instead of the bench")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-gate", action="store_true")
    ap.add_argument("--no-batched", action="store_true")
    ap.add_argument("--no-int32", action="store_true")
    ap.add_argument("--no-cosine", action="store_true")
    ap.add_argument("--no-views", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-config1", action="store_true")
    ap.add_argument("--sharded", action="store_true",
                    help="run the row-sharded step (local search, all-gather, merge) even on one rank")
    ap.add_argument("--schedule", type=int, default=None)
    ap.add_argument("--ctas-per-sm", type=int, default=None)
    ap.add_argument("--stage-bytes", type=int, default=None)
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's).
    A CPU tensor under gloo, a device tensor under NCCL."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def device_info(gpu=0):
    """GPU name, driver version and CUDA runtime of the run (nvidia-smi for the driver)."""
    import torch
    info = {"name": torch.cuda.get_device_name(gpu), "cuda_runtime": torch.version.cuda, "driver": None}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().splitlines()
        info["driver"] = out[0].strip() if out else None
    except (OSError, subprocess.SubprocessError):
        pass
    return info


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except Exception:
        return None


def hbm_peak():
    pk = _peaks()
    if pk and "hbm_gbs" in pk:
        return float(pk["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    pk = _peaks()
    if pk and "bf16_tflops" in pk:
        return float(pk["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the files that define the scoring kernel's code."""
    h = hashlib.sha256()
    for f in ("score_select.cu", "rbf_device.cuh", "merge_core.cuh"):
        with open(os.path.join(ROOT, "resident_brute_force_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the scoring kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "score_select_f32_N100k_D1024_K8_ncu.md")
    rec = {}
    try:
        with open(p) as f:
            for line in f:
                if ":" in line and not line.startswith(("|", "#", " ")):
                    key, _, val = line.partition(":")
                    rec[key.strip()] = val.strip()
    except OSError:
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    try:
        return int(rec["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks

# Clock-event reason bits of NVML (nvmlClocksEventReason*).
_REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
                0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
_BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock-event
    reasons, power) for the device torch calls `gpu`."""

    def __init__(self, gpu: int):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(gpu).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [x.strip() for x in vis.split(",") if x.strip()]
            idx = int(parts[gpu]) if gpu < len(parts) and parts[gpu].isdigit() else gpu
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle for the device")
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_sm = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None

    def sample(self):
        sm = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        pw = ctypes.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(sm)) != 0:
            return None
        self._reasons(self.h, ctypes.byref(rs))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        return float(sm.value), int(rs.value), pw.value / 1000.0


class ClockSampler:
    """SM clock and clock-event reasons sampled every 2 ms (NVML through ctypes;
    nvidia-smi every 100 ms if NVML cannot be loaded) for the whole run; each
    timed region is bracketed with `region(name)` and reported with the
    samples that fall inside it."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []  # (t, sm_mhz, reasons set, watts)
        self.regions = []  # (name, t0, t1)
        self.max_sm = None
        self.source = None
        self._stop = threading.Event()
        self._proc = None

    def start(self):
        try:
            nv = _Nvml(self.gpu)
            self.max_sm = nv.max_sm
            self.source = "nvml, 2 ms"
            threading.Thread(target=self._poll_nvml, args=(nv,), daemon=True).start()
            return self
        except Exception:
            pass
        try:
            fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                      "clocks_event_reasons.sw_power_cap")
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 100 ms"
            threading.Thread(target=self._read_smi, daemon=True).start()
        except Exception:
            self._proc = None
        return self

    def _poll_nvml(self, nv):
        while not self._stop.is_set():
            s = nv.sample()
            if s is not None:
                sm, bits, w = s
                self.samples.append((time.perf_counter(), sm, {n for b, n in _REASON_BITS.items() if bits & b}, w))
            time.sleep(0.002)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.strip().split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
                w = float(parts[2]) if parts[2].replace(".", "", 1).isdigit() else None
            except ValueError:
                continue
            self.max_sm = mx
            reasons = {nm for nm, v in zip(names, parts[3:7]) if v.lower().startswith("active")}
            self.samples.append((time.perf_counter(), sm, reasons, w))

    class _Region:
        def __init__(self, owner, name):
            self.owner, self.name = owner, name

        def __enter__(self):
            self.t0 = time.perf_counter()
            return self

        def __exit__(self, *exc):
            self.owner.regions.append((self.name, self.t0, time.perf_counter()))

    def region(self, name: str):
        return ClockSampler._Region(self, name)

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()

    def _stats(self, windows):
        xs = [s for s in list(self.samples) if any(t0 <= s[0] <= t1 for t0, t1 in windows)]
        reasons = sorted(set().union(*[s[2] for s in xs])) if xs else []
        return {"sm_mhz": statistics.median([s[1] for s in xs]) if xs else None, "sm_max_mhz": self.max_sm,
                "reasons": reasons, "samples": len(xs),
                "sm_mhz_min": min(s[1] for s in xs) if xs else None,
                "rejectable": bool(set(reasons) & _BAD_REASONS)}

    def report(self, headline_prefix: str):
        """Top level: the samples of every region whose name starts with
        headline_prefix; `regions`: each region's own."""
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        head = [(t0, t1) for n, t0, t1 in self.regions if n.startswith(headline_prefix)]
        out = self._stats(head)
        out["source"] = self.source
        out["regions"] = {}
        for n, t0, t1 in self.regions:
            r = self._stats([(t0, t1)])
            out["regions"][n] = {"samples": r["samples"], "sm_mhz": r["sm_mhz"], "reasons": r["reasons"],
                                 "seconds": round(t1 - t0, 4)}
        return out


# ---------------------------------------------------------------- workloads

_CORPORA = {}


def pristine_corpus(n, d):
    """unit_corpus(n, d, seed 1), generated once per (n, d) and never modified."""
    import workloads
    key = (n, d)
    if key not in _CORPORA:
        _CORPORA[key] = workloads.unit_corpus(n, d, seed=1)
    return _CORPORA[key]


def make_workload(n, d, nq):
    import workloads
    c = pristine_corpus(n, d).copy()
    qs = workloads.unit_queries(nq, d, seed=2)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    return c, qs, planted


def result_d2h_bytes(k: int, eb: int = 4) -> int:
    """Bytes of a host-buffer call's result block: the error word and padding,
    then K int32, then K elements of `eb` bytes."""
    a_off = 16
    b_off = (a_off + 4 * k + 15) // 16 * 16
    return b_off + eb * k


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_oracle_rate(c, qs, k, budget_s=12.0, max_queries=200):
    """Time the oracle as it stands on this host. Returns (GB/s, cores, sample text, per-query seconds)."""
    import oracle
    o = oracle.get()
    cores = o.num_threads()
    n, d = c.shape
    times = []
    t_start = time.perf_counter()
    j = 0
    while j < max_queries and (time.perf_counter() - t_start) < budget_s:
        t0 = time.perf_counter()
        o.topk(c, qs[j % len(qs)], k)
        times.append(time.perf_counter() - t0)
        j += 1
    total = sum(times)
    rate = len(times) * n * d * 4 / total / 1e9
    sample = (f"{len(times)} queries x {n} rows x D={d} (K={k}; double scoring + full sort of all rows), "
              f"{total:.1f} s of CPU work")
    return rate, cores, sample, total / len(times)


def headline_config(args, world):
    return {"workload": WORKLOAD, "n": args.n, "d": args.d, "k": 8, "queries": args.queries,
            "parallelism": f"row shards x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (4.1 GB corpus), no flush"}


def run_reference(args):
    """The oracle on the headline workload: each step is one whole query (all
    N rows scored in double, all N pairs sorted), timed on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    n, d = args.n, args.d
    c, qs, _ = make_workload(n, d, args.queries)
    o = oracle.get()
    for j in range(args.warmup):
        o.topk(c, qs[j % len(qs)], 8)
    t0 = time.perf_counter()
    for j in range(args.steps):
        o.topk(c, qs[j % len(qs)], 8)
    dt = time.perf_counter() - t0
    rate = args.steps * n * d * 4 / dt / 1e9
    sample = f"{args.steps} whole queries x {n} rows x D={d} (K=8; double scoring + full sort of all rows)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(rate, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(args, 1),
        "cpu_baseline": {"value": round(rate, 3), "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(rate, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ timing

def percentile(xs, p):
    s = sorted(xs)
    if not s:
        return None
    i = min(len(s) - 1, max(0, int(round(p / 100.0 * (len(s) - 1)))))
    return s[i]


HOST_AHEAD_S_PER_CALL = 40e-6  # host time to enqueue one call (Python binding + launch), generous


def hold_stream(stream, calls):
    """Keep `stream` busy (a GPU spin kernel, outside every timed event) for
    longer than the host needs to enqueue `calls` calls, so that the timed
    calls then run back to back on the device: device time per call, not the
    host's issue rate."""
    import torch
    cycles = int(2.2e9 * max(1e-3, calls * HOST_AHEAD_S_PER_CALL))
    with torch.cuda.stream(stream):
        torch.cuda._sleep(cycles)


def time_device(stream, fn, steps, warmup, back_to_back=False):
    """Per-call device times (ms) of fn() on `stream`, events at call boundaries,
    with the calls enqueued ahead of the device (hold_stream). With
    back_to_back, also the mean per call (ms) of a second pass of `steps`
    calls with events only at its two ends: an event record between two
    launches costs ~2 us of device time, which matters for short calls."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    hold_stream(stream, steps)
    with torch.cuda.stream(stream):
        for j in range(steps):
            ev[j].record(stream)
            fn()
        ev[steps].record(stream)
    torch.cuda.synchronize()
    per_call = [ev[j].elapsed_time(ev[j + 1]) for j in range(steps)]
    if not back_to_back:
        return per_call
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream, steps)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return per_call, a.elapsed_time(b) / steps


def time_device_flushed(stream, fn, steps, warmup, flush):
    """Per-call device times (ms) of fn() with L2 flushed before every call:
    events around the call only, the flush (a write larger than L2) outside."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    hold_stream(stream, 2 * steps)
    with torch.cuda.stream(stream):
        for j in range(steps):
            flush.fill_(j & 0xFF)
            ev[j][0].record(stream)
            fn()
            ev[j][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_host(fn, steps, warmup):
    """Per-call host wall times (s) of a synchronous call."""
    for _ in range(warmup):
        fn()
    out = []
    for _ in range(steps):
        t0 = time.perf_counter()
        fn()
        out.append(time.perf_counter() - t0)
    return out


def l2_bytes():
    import torch
    return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)


TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates


# ------------------------------------------------------------- the blocks

def run_batched(rbf, clocks, steps, warmup, tf32=False):
    """Batched queries: B=256 x N=1,000,000 x D=768, K=32 (tensor-core scoring
    + fused select + merge), fp32 accumulate; bf16 corpus copy, or with
    tf32=True the resident fp32 corpus itself (kind::tf32). Device-timed
    through search_resident_batch_dev; end to end through the host-buffer
    search_resident_batch (B x D floats up, B x K indices and scores down)."""
    import torch
    n, d, b, k = 1_000_000, 768, 256, 32
    c, qs, _ = make_workload(n, d, b)
    st = torch.cuda.Stream()
    e = rbf.Engine(n, d, 100, max_batch=b, flags=0 if tf32 else rbf.RBF_FLAG_BF16_CORPUS, stream=st)
    e.upload_corpus_rowmajor(c)
    del c
    dq = torch.from_numpy(qs).cuda()
    di = torch.empty((b, k), dtype=torch.int32, device="cuda")
    ds = torch.empty((b, k), dtype=torch.float32, device="cuda")
    tag = "batched_tf32" if tf32 else "batched"
    with clocks.region(f"{tag}.k32"):
        ms, mean = time_device(st, lambda: e.search_resident_batch_dev(dq, k, di, ds), steps, warmup,
                               back_to_back=True)
    launches = e.last_launches
    # The other K buckets: 8 (register lists, like 32) and 100 (per-thread
    # lists in the partials buffer, one merge per 256-query group).
    other = {}
    for kk in (8, 100):
        dik = torch.empty((b, kk), dtype=torch.int32, device="cuda")
        dsk = torch.empty((b, kk), dtype=torch.float32, device="cuda")
        with clocks.region(f"{tag}.k{kk}"):
            other[kk] = time_device(st, lambda: e.search_resident_batch_dev(dq, kk, dik, dsk), steps, warmup)
    # A small batch (16 queries, K = 32): the same corpus pass for fewer queries.
    di16 = torch.empty((16, k), dtype=torch.int32, device="cuda")
    ds16 = torch.empty((16, k), dtype=torch.float32, device="cuda")
    with clocks.region(f"{tag}.b16"):
        ms16 = time_device(st, lambda: e.search_resident_batch_dev(dq[:16], k, di16, ds16), steps, warmup)
    with clocks.region(f"{tag}.e2e"):
        host = time_host(lambda: e.search_resident_batch(qs, k), steps, min(warmup, 3))
    e.close()
    p50 = percentile(ms, 50) * 1e-3
    flops = 2.0 * b * n * d
    peak, src = bf16_peak()
    if tf32:
        peak, src = round(peak * TF32_OVER_BF16, 1), src + " bf16 x nominal tf32/bf16 ratio"
    hbm, hsrc = hbm_peak()
    corpus_bytes = n * d * (4 if tf32 else 2)
    # Both rooflines: the tensor work at the bf16 peak and the one pass over
    # the bf16 corpus at the HBM peak; the slower of the two bounds the call.
    bound = "hbm" if corpus_bytes / (hbm * 1e9) > flops / (peak * 1e12) else "tensor"
    corpus = "fp32 corpus as tf32" if tf32 else "bf16 corpus"
    e2e_p50 = percentile(host, 50)
    return {"workload": f"B=256 x N=1,000,000 x D=768 {corpus} (fp32 accumulate), K=32, 10 planted rows/query",
            "p50_us": round(p50 * 1e6, 1), "p99_us": round(percentile(ms, 99) * 1e3, 1),
            "tflops": round(flops / p50 / 1e12, 1), "tensor_peak_tflops": peak, "peak_source": src,
            "tensor_frac": round(flops / p50 / 1e12 / peak, 4),
            "corpus_gbs": round(corpus_bytes / p50 / 1e9, 1), "hbm_peak_gbs": hbm, "hbm_peak_source": hsrc,
            "hbm_frac": round(corpus_bytes / p50 / 1e9 / hbm, 4), "bound": bound,
            "queries_per_s": round(b / p50, 1), "mean_us_back_to_back": round(mean * 1e3, 1),
            "k8_p50_us": round(percentile(other[8], 50) * 1e3, 1),
            "k100_p50_us": round(percentile(other[100], 50) * 1e3, 1),
            "b16_p50_us": round(percentile(ms16, 50) * 1e3, 1),
            "launches_per_call": launches,
            "e2e": {"p50_us": round(e2e_p50 * 1e6, 1), "p99_us": round(percentile(host, 99) * 1e6, 1),
                    "queries_per_s": round(b / e2e_p50, 1), "h2d_bytes_per_call": b * d * 4,
                    "d2h_bytes_per_call": result_d2h_bytes(b * k), "api": "search_resident_batch (host buffers)"},
            "steps": len(ms)}


def run_cosine(rbf, clocks, c, qs, planted, steps, warmup):
    """Cosine mode on the headline workload (N=1M, D=1024, K=8): rows made
    unit length at upload; each step is the scoring kernel (which scales the
    query to unit length first) + the merge, through search_resident_dev."""
    import torch
    n, d = c.shape
    st = torch.cuda.Stream()
    e = rbf.Engine(n, d, 8, stream=st, flags=rbf.RBF_FLAG_COSINE)
    e.upload_corpus_rowmajor(c)
    for j in range(0, len(qs), max(1, len(qs) // 10)):
        idx, _ = e.search_resident(qs[j], 8)
        assert set(idx.tolist()) <= set(planted[j].tolist()), f"cosine: planted rows missing for query {j}"
    dq = torch.from_numpy(qs).cuda()
    di = torch.empty(8, dtype=torch.int32, device="cuda")
    ds = torch.empty(8, dtype=torch.float32, device="cuda")
    nq = len(qs)
    it = iter(range(10 ** 9))
    with clocks.region("cosine"):
        ms = time_device(st, lambda: e.search_resident_dev(dq[next(it) % nq], 8, di, ds), steps, warmup)
    e.close()
    p50 = percentile(ms, 50) * 1e-3
    hbm, _ = hbm_peak()
    gbs = n * d * 4 / p50 / 1e9
    return {"workload": "cosine mode, N=1,000,000 x D=1024 fp32 (rows unit length at upload), K=8",
            "p50_us": round(p50 * 1e6, 1), "p99_us": round(percentile(ms, 99) * 1e3, 1),
            "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4), "launches_per_step": 1, "steps": len(ms)}


def run_views(rbf, clocks, reps=6):
    """Concurrent single-query searches through views (rbf_create_view):
    N=100,000 x D=768 fp32 (307 MB, larger than L2), K=8, 256 device-resident
    queries per round issued round-robin over 1 or 4 handles, each on its own
    stream; throughput = queries / host wall time of whole rounds (the calls
    are asynchronous; one synchronisation per round)."""
    import torch
    import workloads
    n, d, k, nq = 100_000, 768, 8, 256
    c = pristine_corpus(1_000_000, d)[:n]
    dq = torch.from_numpy(workloads.unit_queries(nq, d, seed=2)).cuda()
    oi = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    osc = torch.empty((nq, k), dtype=torch.float32, device="cuda")
    hbm, _ = hbm_peak()
    out = {"workload": "N=100,000 x D=768 fp32, K=8, 256 queries per round, round-robin over handles"}
    for nh in (1, 4):
        streams = [torch.cuda.Stream() for _ in range(nh)]
        base = rbf.Engine(n, d, k, stream=streams[0])
        base.upload_corpus_rowmajor(c)
        hs = [base] + [base.view(stream=st) for st in streams[1:]]

        def round_():
            for j in range(nq):
                hs[j % nh].search_resident_dev(dq[j], k, oi[j], osc[j])

        for _ in range(3):
            round_()
        torch.cuda.synchronize()
        with clocks.region(f"views.h{nh}"):
            t0 = time.perf_counter()
            for _ in range(reps):
                round_()
            torch.cuda.synchronize()
            qps = reps * nq / (time.perf_counter() - t0)
        for h in hs[1:]:
            h.close()
        base.close()
        out[f"handles_{nh}"] = {"qps": round(qps, 1), "gbs": round(qps * n * d * 4 / 1e9, 1),
                                "hbm_frac": round(qps * n * d * 4 / 1e9 / hbm, 4)}
    out["speedup_4_over_1"] = round(out["handles_4"]["qps"] / out["handles_1"]["qps"], 3)
    return out


def run_int32(rbf, clocks, steps, warmup):
    """Flat int32 two-stage top-K: 100,000,000 values, K=20 and K=50; device
    time through topk_int32_dev, and the host-output topk_int32 end to end
    (the array is device-resident by the call's definition: K values and K
    positions come down)."""
    import torch
    import workloads
    n = 100_000_000
    x = torch.from_numpy(workloads.int32_uniform(n, seed=1)).cuda()
    st = torch.cuda.Stream()
    e = rbf.Engine(16, 16, 64, stream=st)
    out = {"workload": "n=100,000,000 int32 uniform over the full range",
           # The two-stage page's own kernel times for n = 1e8 (context, other hardware).
           "pages_context": {"k20_ms": 8.7, "k50_ms": 15.1, "hardware": "Tesla V100, GRID 64 x BLOCK 256"}}
    dv = torch.empty(64, dtype=torch.int32, device="cuda")
    dp = torch.empty(64, dtype=torch.int64, device="cuda")
    hbm, _ = hbm_peak()
    for k in (20, 50):
        with clocks.region(f"int32.k{k}"):
            ms, mean = time_device(st, lambda: e.topk_int32_dev(x, k, dv, dp), steps, warmup, back_to_back=True)
        with clocks.region(f"int32.k{k}.e2e"):
            host = time_host(lambda: e.topk_int32(x, k), steps, 3)
        p50 = percentile(ms, 50) * 1e-3
        out[f"k{k}"] = {"p50_us": round(p50 * 1e6, 1), "p99_us": round(percentile(ms, 99) * 1e3, 1),
                        "gbs": round(4.0 * n / p50 / 1e9, 1), "hbm_frac": round(4.0 * n / p50 / 1e9 / hbm, 4),
                        "mean_us_back_to_back": round(mean * 1e3, 1),
                        "hbm_frac_back_to_back": round(4.0 * n / (mean * 1e-3) / 1e9 / hbm, 4),
                        "e2e_p50_us": round(percentile(host, 50) * 1e6, 1),
                        "e2e_p99_us": round(percentile(host, 99) * 1e6, 1),
                        "e2e_d2h_bytes_per_call": result_d2h_bytes(k, 8)}
    # The entry point that allocates nothing (register-load stage 1 + merge
    # kernel, scratch in a fixed device array), for comparison.
    for k in (20, 50):
        cs = torch.cuda.current_stream()
        with clocks.region(f"int32.noalloc.k{k}"):
            ms = time_device(cs, lambda: rbf.topk_int32_noalloc(x, k, dv, dp, stream=cs), steps, warmup)
        out[f"noalloc_k{k}_p50_us"] = round(percentile(ms, 50) * 1e3, 1)
    e.close()
    return out


def run_config1(rbf, clocks, reps):
    """N=10,000 x D=384 unit-norm corpus (seed 1), 16 queries (seed 2), K=8.
    The corpus (15.4 MB) fits in L2: device time is reported L2-resident
    (back-to-back calls) and with L2 flushed before every call (a 256 MB
    write outside the timed events), and end to end through search_resident.
    Every query is checked against the oracle first."""
    import torch

    import oracle
    import workloads
    from tests.parity import check_float_topk
    n, d, k, nq = 10_000, 384, 8, 16
    c = pristine_corpus(1_000_000, d)[:n]
    qs = workloads.unit_queries(nq, d, seed=2)
    st = torch.cuda.Stream()
    e = rbf.Engine(n, d, k, stream=st)
    e.upload_corpus_rowmajor(c)
    for j in range(nq):
        idx, sc = e.search_resident(qs[j], k)
        check_float_topk(idx, sc, oracle.scores(c, qs[j]), k)
    dq = torch.from_numpy(qs).cuda()
    di = torch.empty(k, dtype=torch.int32, device="cuda")
    ds = torch.empty(k, dtype=torch.float32, device="cuda")
    steps = nq * reps
    it = iter(range(10 ** 9))
    with clocks.region("config1.l2"):
        warm, warm_mean = time_device(st, lambda: e.search_resident_dev(dq[next(it) % nq], k, di, ds), steps, 20,
                                      back_to_back=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    with clocks.region("config1.flushed"):
        cold = time_device_flushed(st, lambda: e.search_resident_dev(dq[next(it) % nq], k, di, ds), steps, 20,
                                   flush)
    del flush
    launches = e.last_launches
    with clocks.region("config1.e2e"):
        host = time_host(lambda: e.search_resident(qs[next(it) % nq], k), steps, 20)
    e.close()
    hbm, _ = hbm_peak()
    p50 = percentile(warm, 50) * 1e-3
    p50c = percentile(cold, 50) * 1e-3
    return {"workload": "N=10,000 x D=384 fp32 unit-norm corpus, 16 queries, K=8, inner product",
            "queries": nq, "calls": steps, "l2": "corpus 15.4 MB < L2: L2-resident unless flushed",
            "p50_us": round(p50 * 1e6, 2), "p99_us": round(percentile(warm, 99) * 1e3, 2),
            "qps": round(1.0 / p50, 1), "gbs_l2": round(n * d * 4 / p50 / 1e9, 1),
            "mean_us_back_to_back": round(warm_mean * 1e3, 2),
            "flushed_p50_us": round(p50c * 1e6, 2), "flushed_p99_us": round(percentile(cold, 99) * 1e3, 2),
            "flushed_gbs": round(n * d * 4 / p50c / 1e9, 1),
            "flushed_hbm_frac": round(n * d * 4 / p50c / 1e9 / hbm, 4),
            "e2e_p50_us": round(percentile(host, 50) * 1e6, 2), "e2e_p99_us": round(percentile(host, 99) * 1e6, 2),
            "e2e_h2d_bytes_per_call": d * 4, "e2e_d2h_bytes_per_call": result_d2h_bytes(k),
            "oracle_checked_queries": nq, "launches_per_call": launches}


def run_sweep(rbf, clocks, queries):
    """The pages' sweep: N in {10k, 50k, 100k, 500k, 1M} x D in {384, 768,
    1024} x K in {8, 32, 100}, unit-norm Gaussian rows (seed 1) and queries
    (seed 2). Per cell: `queries` device calls (search_resident_dev, events at
    call boundaries) and as many host calls (search_resident, wall clock). One
    query per (N, D) is checked against the oracle at every K first. A corpus
    under twice the L2 stays in L2 between calls and is flagged, not flushed."""
    import torch

    import oracle
    import workloads
    from tests.parity import check_float_topk
    hbm, hsrc = hbm_peak()
    l2 = l2_bytes()
    cells = []
    for d in SWEEP_D:
        full = pristine_corpus(max(SWEEP_N), d)
        dfull = torch.from_numpy(full).cuda()  # one host-to-device copy; every upload is then on the device
        qs = workloads.unit_queries(queries, d, seed=2)
        dq = torch.from_numpy(qs).cuda()
        st = torch.cuda.Stream()
        eng = rbf.Engine(max(SWEEP_N), d, max(SWEEP_K), stream=st)
        for n in SWEEP_N:
            eng.upload_corpus_rowmajor(dfull[:n])
            sigma = oracle.scores(full[:n], qs[0])
            for k in SWEEP_K:
                check_float_topk(*eng.search_resident(qs[0], k), sigma, k)
            nbytes = n * d * 4
            for k in SWEEP_K:
                di = torch.empty(k, dtype=torch.int32, device="cuda")
                dsc = torch.empty(k, dtype=torch.float32, device="cuda")
                it = iter(range(10 ** 9))
                with clocks.region(f"sweep.n{n}.d{d}.k{k}"):
                    dev, b2b = time_device(st, lambda: eng.search_resident_dev(dq[next(it) % queries], k, di, dsc),
                                           queries, 10, back_to_back=True)
                    it2 = iter(range(10 ** 9))
                    host = time_host(lambda: eng.search_resident(qs[next(it2) % queries], k), queries, 10)
                p50 = percentile(dev, 50) * 1e-3
                mean = statistics.mean(dev) * 1e-3
                cells.append({
                    "n": n, "d": d, "k": k, "queries": queries,
                    "p50_us": round(p50 * 1e6, 1), "p99_us": round(percentile(dev, 99) * 1e3, 1),
                    "mean_us_back_to_back": round(b2b * 1e3, 1),
                    "qps": round(1.0 / mean, 1), "gbs": round(nbytes / mean / 1e9, 1),
                    "hbm_frac": round(nbytes / mean / 1e9 / hbm, 4),
                    "e2e_p50_us": round(percentile(host, 50) * 1e6, 1),
                    "e2e_p99_us": round(percentile(host, 99) * 1e6, 1),
                    "l2_resident": nbytes < 2 * l2})
        eng.close()
        del dfull, dq
    return {"grid": "N x D x K = {10k,50k,100k,500k,1M} x {384,768,1024} x {8,32,100}", "hbm_peak_gbs": hbm,
            "hbm_peak_source": hsrc, "l2_bytes": l2, "oracle_gate": "1 query per (N, D), every K",
            "cells": cells}


# ------------------------------------------------------------- row shards

def run_sharded(rbf, args, rank: int, world: int) -> dict:
    """The step on `world` ranks: each rank holds args.n rows (weak
    scaling: a corpus of world * args.n rows), a step is one sharded search
    (local search, exchange, merge). value = all ranks' rows x D x 4 bytes per
    step / the slowest rank's time."""
    import torch
    import torch.distributed as dist

    import workloads
    from resident_brute_force_gb300.sharded import ShardedSearch
    n_total, d, nq = args.n * world, args.d, args.queries
    s = ShardedSearch(rbf, n_total, d, 256, world, rank)
    shard = workloads.unit_corpus_rows(s.row0, s.rows, d, seed=1)
    qs = workloads.unit_queries(nq, d, seed=2)
    planted = workloads.plant_near_duplicates_shard(shard, s.row0, n_total, qs, per_query=10, noise=0.05, seed=3)
    s.upload(shard)
    del shard
    dq = torch.from_numpy(qs).cuda()
    di = torch.empty(256, dtype=torch.int32, device="cuda")
    ds = torch.empty(256, dtype=torch.float32, device="cuda")
    if not args.no_gate:
        for j in range(0, nq, max(1, nq // 20)):
            idx, _ = s.search(qs[j], 32)
            assert set(idx[:10].tolist()) == set(planted[j].tolist()), f"planted rows missing for query {j}"
    per_k = {}
    headline = None
    ks = [8] + [int(x) for x in args.extra_k.split(",") if x]
    for k in ks:
        for j in range(args.warmup):
            s.search_dev(dq[j % nq], k, di, ds)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        dist.barrier()
        torch.cuda.synchronize()
        for j in range(args.steps):
            ev[j].record(s.stream)
            s.search_dev(dq[j % nq], k, di, ds)
        ev[args.steps].record(s.stream)
        torch.cuda.synchronize()
        dist.barrier()
        step_ms = [ev[j].elapsed_time(ev[j + 1]) for j in range(args.steps)]
        total_ms = max_over_ranks(ev[0].elapsed_time(ev[args.steps]), world)
        per_k[str(k)] = {"p50_us": round(percentile(step_ms, 50) * 1e3, 2),
                         "p99_us": round(percentile(step_ms, 99) * 1e3, 2),
                         "gbs": round(world * args.steps * args.n * d * 4 / (total_ms * 1e-3) / 1e9, 1),
                         "launch_us_mean": round(statistics.mean(step_ms) * 1e3, 2)}
        if k == 8:
            headline = total_ms
    for j in range(args.warmup):
        s.search(qs[j % nq], 8)
    dist.barrier()
    t0 = time.perf_counter()
    for j in range(args.steps):
        s.search(qs[j % nq], 8)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    s.close()
    value = world * args.steps * args.n * d * 4 / (headline * 1e-3) / 1e9
    peak, src = hbm_peak()
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(headline / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(headline_config(args, world), n=n_total, rows_per_rank=args.n),
        "per_k": per_k, "p50_us": per_k["8"]["p50_us"],
        "roofline": {"kernel": "score_select_f32 (per rank)", "bound": "hbm",
                     "achieved": round(value / world, 1), "peak": peak, "peak_source": src, "unit": "GB/s",
                     "frac": round(value / world / peak, 4), "traffic": None},
        "cpu_baseline": None,
        "e2e": {"value": round(world * args.steps * args.n * d * 4 / e2e_s / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": d * 4, "d2h_bytes_per_step": 8 * 8},
        # Per step and rank: the scoring kernel, the shard-list encoding and
        # the merge kernel (the collective's own kernels are NCCL's).
        "gpu_launches": 3 * args.steps,
    }


# ------------------------------------------------------------ profiling cases

def run_case(part: str) -> int:
    """One small workload per kernel for profiler captures: each holds a few
    hundred MB on the device (batch_full: about 4.6 GB, for one-pass launch
    lists only) and makes a handful of launches."""
    import torch

    import resident_brute_force_gb300 as rbf
    import workloads
    if rbf._build.is_stale():
        rbf._build.build()
    if part == "single":  # scoring (+ merge kernel), 100k x 1024, K=8
        n, d = 100_000, 1024
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(4, d, seed=2)
        e = rbf.Engine(n, d, 256)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        di = torch.empty(256, dtype=torch.int32, device="cuda")
        ds = torch.empty(256, dtype=torch.float32, device="cuda")
        for j in range(4):
            e.search_resident_dev(dq[j], 8, di, ds)  # one launch each (merge in the last CTA)
        for j in range(3):
            e.score_select_partials_dev(dq[j], 8)  # the two-step calls: the merge kernel
            e.merge_partial_topk_dev(8, di, ds)
    elif part == "small":  # the 10k x 384 corpus, K=8 (launch latency)
        n, d = 10_000, 384
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(16, d, seed=2)
        e = rbf.Engine(n, d, 8)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        di = torch.empty(8, dtype=torch.int32, device="cuda")
        ds = torch.empty(8, dtype=torch.float32, device="cuda")
        for j in range(16):
            e.search_resident_dev(dq[j], 8, di, ds)
    elif part == "batch":  # batched, 256 queries x 200k x 768, K=32
        n, d, b = 200_000, 768, 256
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(b, d, seed=2)
        e = rbf.Engine(n, d, 32, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        di = torch.empty((b, 32), dtype=torch.int32, device="cuda")
        ds = torch.empty((b, 32), dtype=torch.float32, device="cuda")
        for _ in range(2):
            e.search_resident_batch_dev(dq, 32, di, ds)
    elif part == "batch_full":  # 256 x 1M x 768, K=8/32/100 (one-pass launch lists only)
        n, d, b = 1_000_000, 768, 256
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(b, d, seed=2)
        e = rbf.Engine(n, d, 100, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        for k in (8, 32, 100):
            di = torch.empty((b, k), dtype=torch.int32, device="cuda")
            ds = torch.empty((b, k), dtype=torch.float32, device="cuda")
            for _ in range(3):
                e.search_resident_batch_dev(dq, k, di, ds)
    elif part == "int32":  # int32 top-K, 5e7 values, K=20
        x = torch.from_numpy(workloads.int32_uniform(50_000_000, seed=1)).cuda()
        e = rbf.Engine(16, 16, 64)
        dv = torch.empty(64, dtype=torch.int32, device="cuda")
        dp = torch.empty(64, dtype=torch.int64, device="cuda")
        for _ in range(2):
            e.topk_int32_dev(x, 20, dv, dp)
    else:
        raise SystemExit(f"unknown case {part!r}: single | small | batch | batch_full | int32")
    torch.cuda.synchronize()
    print("ok", part)
    return 0


# -------------------------------------------------------------------- main

def main(argv=None):
    args = parse(argv)
    if args.case:
        return run_case(args.case)
    if args.impl == "reference":
        return run_reference(args)

    import torch

    rank, world, local = dist_env()
    sharded = world > 1 or args.sharded
    if sharded:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29531")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", rank=rank, world_size=world)
    torch.cuda.set_device(local)

    import resident_brute_force_gb300 as rbf
    if rbf._build.is_stale():
        rbf._build.build()
    if sharded:
        line = run_sharded(rbf, args, rank, world)
        import torch.distributed as dist
        dist.destroy_process_group()
        # NCCL may print to stdout through C stdio (buffered until exit): flush
        # it first so that the result is the last line.
        try:
            ctypes.CDLL(None).fflush(None)
        except Exception:
            pass
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0

    clocks = ClockSampler(local).start()
    n, d, nq = args.n, args.d, args.queries
    c, qs, planted = make_workload(n, d, nq)
    stream = torch.cuda.Stream()
    eng = rbf.Engine(n, d, 256, stream=stream)
    if args.schedule is not None:
        eng.set_option(rbf.RBF_OPT_SCHEDULE, args.schedule)
    if args.ctas_per_sm is not None:
        eng.set_option(rbf.RBF_OPT_CTAS_PER_SM, args.ctas_per_sm)
    if args.stage_bytes is not None:
        eng.set_option(rbf.RBF_OPT_STAGE_BYTES, args.stage_bytes)
    eng.upload_corpus_rowmajor(c)
    dq = torch.from_numpy(qs).cuda()
    d_idx = torch.empty(256, dtype=torch.int32, device="cuda")
    d_sc = torch.empty(256, dtype=torch.float32, device="cuda")

    # Correctness gate before any timing: planted rows lead for a sample of
    # queries, and one query matches the oracle under the parity rule.
    if not args.no_gate:
        for j in range(0, nq, max(1, nq // 20)):
            idx, _ = eng.search_resident(qs[j], 32)
            assert set(idx[:10].tolist()) == set(planted[j].tolist()), f"planted rows missing for query {j}"
        import oracle
        from tests.parity import check_float_topk
        sigma = oracle.scores(c, qs[0])
        for k in (8, 32, 100):
            idx, sc = eng.search_resident(qs[0], k)
            check_float_topk(idx, sc, sigma, k)

    bytes_per_step = n * d * 4
    ks = [8] + [int(x) for x in args.extra_k.split(",") if x]
    per_k = {}
    headline = None
    for k in ks:
        with torch.cuda.stream(stream):
            for j in range(args.warmup):
                eng.search_resident_dev(dq[j % nq], k, d_idx, d_sc)
        # One step is one search_resident_dev call: a single launch of the
        # scoring kernel, whose last CTA also merges the per-CTA lists. The
        # timed region is exactly `steps` back-to-back calls between two events
        # on the launching stream (throughput, mean launch duration); a second
        # pass with an event at every step boundary gives the per-call p50/p99.
        qv = [dq[j % nq] for j in range(args.steps)]
        t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        bounds = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        torch.cuda.synchronize()
        with clocks.region(f"headline.k{k}"):
            hold_stream(stream, args.steps)
            with torch.cuda.stream(stream):
                t_a.record(stream)
                for j in range(args.steps):
                    eng.search_resident_dev(qv[j], k, d_idx, d_sc)
                t_b.record(stream)
            torch.cuda.synchronize()
            hold_stream(stream, args.steps)
            with torch.cuda.stream(stream):
                for j in range(args.steps):
                    bounds[j].record(stream)
                    eng.search_resident_dev(qv[j], k, d_idx, d_sc)
                bounds[args.steps].record(stream)
            torch.cuda.synchronize()
        step_ms = [bounds[j].elapsed_time(bounds[j + 1]) for j in range(args.steps)]
        total_ms = t_a.elapsed_time(t_b)
        launches_per_step = eng.last_launches
        rec = {
            "p50_us": round(percentile(step_ms, 50) * 1e3, 2),
            "p99_us": round(percentile(step_ms, 99) * 1e3, 2),
            "gbs": round(args.steps * bytes_per_step / (total_ms * 1e-3) / 1e9, 1),
            "qps": round(args.steps / (total_ms * 1e-3), 1),
            "launch_us_mean": round(total_ms / args.steps * 1e3, 2),
            "per_call_event_us_mean": round(statistics.mean(step_ms) * 1e3, 2),
            "launches_per_step": launches_per_step,
        }
        per_k[str(k)] = rec
        if k == 8:
            headline = (total_ms, step_ms)

    # End to end through the public host-buffer call: the query through the
    # pinned staging block, the kernel, the K results through the pinned
    # result block.
    e2e = None
    if not args.no_e2e:
        for j in range(args.warmup):
            eng.search_resident(qs[j % nq], 8)
        call_s = []
        with clocks.region("e2e.k8"):
            t0 = time.perf_counter()
            for j in range(args.steps):
                t1 = time.perf_counter()
                eng.search_resident(qs[j % nq], 8)
                call_s.append(time.perf_counter() - t1)
            dt = time.perf_counter() - t0
        e2e = {"value": round(args.steps * bytes_per_step / dt / 1e9, 1), "unit": "GB/s",
               "h2d_bytes_per_step": d * 4, "d2h_bytes_per_step": result_d2h_bytes(8),
               "p50_us": round(percentile(call_s, 50) * 1e6, 2), "p99_us": round(percentile(call_s, 99) * 1e6, 2),
               "ms_per_step": round(dt / args.steps * 1e3, 4)}

    total_ms, step_ms = headline
    value = args.steps * bytes_per_step / (total_ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    # The dominant (only) kernel's average launch duration: the mean step of
    # the timed back-to-back region.
    k1_mean_s = total_ms / args.steps * 1e-3
    achieved = bytes_per_step / k1_mean_s / 1e9
    roofline = {"kernel": "score_select_f32", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic(), "bytes_per_launch": bytes_per_step,
                "vs_8tbs": round(achieved / 8000.0, 4)}

    eng.close()
    blocks = {}
    if not args.no_cosine:
        blocks["cosine"] = run_cosine(rbf, clocks, c, qs, planted, 200, 5)
    del c
    if not args.no_config1:
        blocks["config1"] = run_config1(rbf, clocks, reps=20)
    if not args.no_sweep:
        blocks["sweep"] = run_sweep(rbf, clocks, args.sweep_queries)
    if not args.no_batched:
        blocks["batched"] = run_batched(rbf, clocks, 30, 3)
        blocks["batched_tf32"] = run_batched(rbf, clocks, 20, 3, tf32=True)
    if not args.no_int32:
        blocks["int32"] = run_int32(rbf, clocks, 50, 5)
    if not args.no_views:
        blocks["views"] = run_views(rbf, clocks)
    clocks.stop()

    cpu = None
    if not args.no_cpu_baseline:
        c, qs, _ = make_workload(n, d, nq)
        rate, cores, sample, _ = cpu_oracle_rate(c, qs, 8)
        cpu = {"value": round(rate, 3), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "cpu_model": cpu_model()}
        # The same oracle on one core (scoring no longer split over threads).
        import oracle
        o = oracle.get()
        o.set_num_threads(1)
        try:
            rate1, _, sample1, _ = cpu_oracle_rate(c, qs, 8, budget_s=4.0, max_queries=3)
        finally:
            o.set_num_threads(cores)
        cpu["one_core"] = {"value": round(rate1, 3), "sample": sample1}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": headline_config(args, world),
        "p50_us": per_k["8"]["p50_us"], "p99_us": per_k["8"]["p99_us"], "per_k": per_k,
        "k100_over_k8": round(per_k["100"]["p50_us"] / per_k["8"]["p50_us"], 3) if "100" in per_k else None,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps * per_k["8"]["launches_per_step"], "clocks": clocks.report("headline."), "device": device_info(local),
        # The pages' number for this workload (1M x 1024, K = 8) is end to end on a
        # GTX 1080: 114.12 ms per query = 35.9 GB/s. Context, not the target; vs_baseline
        # stays null because that figure is end to end and `value` is device time.
        "pages_context": {"e2e_gbs": 35.9, "hardware": "GTX 1080 (sm_61), end to end, mean of 3",
                          "e2e_over_pages": round(e2e["value"] / 35.9, 1) if e2e else None},
    }
    line.update(blocks)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
