#!/usr/bin/env python3
"""Benchmark of the lossless BF16 exponent codec on GB300.

Default workload: the Llama3-8B-shaped all-gather payload (one 4096x14336 BF16
tensor, i.i.d. N(0, 0.02^2), LUT from sigma = 0.02).  One step = one pass of
the codec's hot path over one batch: compress a batch, and decompress the
stream compressed one step earlier (so the stream read by decompress is not
L2-resident, as it would not be after crossing the network).  Three rotating
buffer sets, 316 MB touched per step (> 129 MB L2), keep every step's inputs
out of L2.  Within the timed region each op's K launches run back to back
between one pair of CUDA events.  After it, the same launches are timed one
at a time (each between its own events), and once more back to back with
events at six group boundaries for a spread; both are reported beside the
timed means.  Other workloads (--workload): activation_mix (compress +
decompress), moe_a2a (one batched compress of 128 static/dynamic segments),
rs_local (decompress-reduce of 8 shards), rs_local_own (the same with the rank's own shard
uncompressed), activation_mix_lut (the exponent histogram pass that measures
a LUT from the data), gauss1m, gauss268m (one stream of 268M elements, the
same distribution as the default).

Prints ONE JSON line (rank 0).  `value` = GB/s of BF16 input through the step
(2n bytes per compress and per decompress; reduce: 2 S n; histogram: 2n),
whole job.
`--impl reference` times the CPU oracle (plain C, single thread) instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="zccl", choices=["zccl", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=["llama3_8b_allgather", "activation_mix", "moe_a2a", "rs_local", "rs_local_own",
                            "activation_mix_lut", "gauss1m", "gauss268m"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="with the default workload, skip the record of the other workloads")
    return p.parse_args()


# ---------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and with runs of whitespace collapsed:
    what the hash of a kernel's sources should follow (a comment edit does
    not change the kernel)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_sha(names):
    h = hashlib.sha256()
    for n in list(names) + ["zccl_common.cuh"]:
        with open(os.path.join(ROOT, "lossless_bf16_exponent_split_gb300", "csrc", n)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


# the kernels of each op live in these sources (plus zccl_common.cuh)
KERNEL_SOURCES = {"compress": ["zccl_compress.cu"], "decompress": ["zccl_decompress.cu", "zccl_decode.cuh"],
                  "decompress_reduce": ["zccl_reduce.cu", "zccl_decompress.cu", "zccl_decode.cuh"],
                  "histogram": ["zccl_hist.cu"]}
OP_KERNELS = {"compress": "compress_kernel (one cooperative launch)",
              "decompress": "decompress_kernel (one cooperative launch)",
              "decompress_reduce": "escape_scan_kernel + reduce_kernel (PDL pair)",
              "histogram": "hist_zero_kernel + hist_kernel (PDL pair)"}
OP_LAUNCHES = {"compress": 1, "decompress": 1, "decompress_reduce": 2, "histogram": 2}
# the headline workload (the 58.7M-element Llama3-8B all-gather payload), and
# the others that its run also measures and reports under "configs"
DEFAULT_WORKLOAD = "llama3_8b_allgather"
CONFIG_WORKLOADS = ["activation_mix", "moe_a2a", "rs_local", "rs_local_own", "activation_mix_lut"]
# the committed ncu summary of each op's dominant kernel is
# profiles/<PROFILE_KERNEL[op]>_<workload>.md
PROFILE_KERNEL = {"compress": "compress_kernel", "decompress": "decompress_kernel",
                  "decompress_reduce": "reduce_kernel", "histogram": "hist_kernel"}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{PROFILE_KERNEL[kernel]}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return float(m.group(1))


class NvmlClockPoller:
    """SM clock and clock-event reasons read through NVML (ctypes) every
    ~0.5 ms from a background thread, so that a timed region of a few
    milliseconds still gets samples.  Read-only; any NVML failure leaves it
    inactive."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        import threading
        self.samples, self.max_mhz, self.reasons = [], None, set()
        self.stop = threading.Event()
        self.thread = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            self.nvml = nvml
            self.handle = ctypes.c_void_p()
            found = False
            try:  # by UUID: NVML may number the GPUs differently from CUDA
                import torch
                uuid = str(torch.cuda.get_device_properties(device_index).uuid)
                found = nvml.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.handle)) == 0
            except Exception:
                found = False
            if not found and nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index),
                                                                 ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint(0)
            if nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
                self.max_mhz = float(mx.value)
            get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.get_reasons = get_reasons
            self.thread = threading.Thread(target=self._run, daemon=True)
        except Exception:
            self.thread = None

    def _run(self):
        import ctypes
        clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self.stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if self.get_reasons(self.handle, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.0005)

    def __enter__(self):
        if self.thread is not None:
            self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)


class ClockSampler:
    """Clocks and throttle reasons during the timed region: NVML polled every
    ~0.5 ms inside it (see NvmlClockPoller), and nvidia-smi every 100 ms from
    0.3 s before to 0.2 s after it as a fallback."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        # the raw nvidia-smi record goes where ZCCL_BENCH_CLOCKS_DIR says (kept
        # for inspection), else to a temporary file removed after the summary
        keep = os.environ.get("ZCCL_BENCH_CLOCKS_DIR")
        base = keep if keep else tempfile.gettempdir()
        self.keep = bool(keep)
        self.path = os.path.join(base, f"zccl_clocks_{os.getpid()}.csv")
        self.poller = None

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        self.poller = NvmlClockPoller(self.idx).__enter__()
        return self

    def __exit__(self, *exc):
        if self.poller is not None:
            self.poller.__exit__(*exc)
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        try:
            return self._summary()
        finally:
            if not self.keep:
                try:
                    os.remove(self.path)
                except OSError:
                    pass

    def _summary(self):
        p = self.poller
        if p is not None and p.samples:
            return {"sm_mhz": statistics.median(p.samples), "sm_max_mhz": p.max_mhz, "samples": len(p.samples),
                    "reasons": sorted(p.reasons), "source": "nvml, polled during the timed region"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons), "source": "nvidia-smi, 100 ms around the timed region"}


# ---------------------------------------------------------------------------
def config_record(workload: str, m: dict) -> dict:
    """One workload's entry of the "configs" record: each op's mean time over
    the back-to-back launches, its algorithmic bytes, achieved GB/s and
    fraction of the HBM peak, the median single evented launch, the ncu
    traffic of its dominant kernel (if a summary of the current source is
    committed), and the clocks seen while it ran."""
    peak, peak_kind = hbm_peak()
    ops = {}
    for nm in m["names"]:
        ms = m["k_ms"][nm]
        a = m["alg"][nm] / (ms * 1e-3) / 1e9
        med = float(np.median(m["single"][nm]))
        ops[nm] = {"ms": round(ms, 4), "algorithmic_bytes": m["alg"][nm], "achieved_gbs": round(a, 2),
                   "frac_of_" + peak_kind: round(a / peak, 4),
                   "single_launch_evented_median_ms": round(med, 4),
                   "single_launch_frac_of_" + peak_kind: round(m["alg"][nm] / (med * 1e-3) / 1e9 / peak, 4),
                   "traffic": ncu_traffic(nm, workload)}
    keep = {k: v for k, v in m["cfg_extra"].items() if k in ("n", "shards", "segments", "stream_bytes",
                                                             "stream_bytes_total", "ratio", "top7_coverage")}
    return {"desc": workload_desc(workload), **keep, "ops": ops, "clocks": m["clocks"],
            "timing": "mean of the back-to-back launches between one event pair, as the headline"}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "zccl" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, value: float, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world: int, step_bytes: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank processes step_bytes per step; the step
    takes the slowest rank's time (weak scaling)."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


# ---------------------------------------------------------------------------
def workload_desc(name):
    from lossless_bf16_exponent_split_gb300 import workloads
    return workloads.CONFIGS[name]["desc"]


def decompress_offset(warmup: int, steps: int, R: int) -> int:
    """Rotation offset of the stream the round trip's decompress reads at
    step k: buffer (k + offset) mod R, with compress writing buffer k mod R.
    -1 (the previous step's stream) unless the timed decompress batch would
    then start on the buffer the timed compress batch wrote last, still partly
    in L2; then +1.  Never 0, which would read the stream just written in the
    interleaved single-launch timing."""
    last = (warmup + steps) % R
    return -1 if warmup % R != last else 1


def group_bounds(steps: int, groups: int = 6) -> list:
    """Launch indices bounding up to `groups` non-empty, near-equal groups of
    `steps` back-to-back launches (for the spread pass)."""
    g = min(steps, groups)
    return [round(i * steps / g) for i in range(g + 1)]


def make_inputs(name, seed):
    """Host arrays for a workload: (kind, payload(s), sigma, extra)."""
    from lossless_bf16_exponent_split_gb300 import workloads as w
    cfg = w.CONFIGS[name]
    if name in ("llama3_8b_allgather", "gauss1m", "gauss268m"):
        return "roundtrip", w.gaussian(cfg["n"], cfg["sigma"], seed=seed), cfg["sigma"], None
    if name == "activation_mix":
        return "roundtrip", w.activation_mix(seed=seed), cfg["sigma"], None
    if name == "activation_mix_lut":
        return "histogram", w.activation_mix(seed=seed), cfg["sigma"], None
    if name == "moe_a2a":
        m = w.moe_payload(tokens=cfg["tokens"], top_k=cfg["top_k"], experts=cfg["experts"],
                          hidden=cfg["hidden"], seed=seed)
        return "batched", m.payload, cfg["sigma"], m
    if name in ("rs_local", "rs_local_own"):
        return ("reduce", w.reduce_shards(cfg["S"], cfg["n"], cfg["sigma"], seed=seed), cfg["sigma"],
                cfg.get("local_pos"))
    raise ValueError(name)


def cpu_baseline(name, budget_s=12.0):
    """The oracle as it stands (single-threaded C), on a bounded sample."""
    import oracle
    from lossless_bf16_exponent_split_gb300 import workloads as w
    cfg = w.CONFIGS[name]
    sigma = cfg["sigma"]
    lut = oracle.lut_from_sigma(sigma)
    if name in ("rs_local", "rs_local_own"):
        n = 1 << 21
        shards = w.reduce_shards(cfg["S"], n, sigma, seed=0)
        lp = cfg.get("local_pos")
        streams = [None if s == lp else oracle.compress(x, lut) for s, x in enumerate(shards)]
        t0 = time.perf_counter()
        reps = 0
        while True:
            if lp is None:
                oracle.decompress_reduce(streams, n)
            else:
                oracle.decompress_reduce_local(streams, n, local=shards[lp], local_pos=lp)
            reps += 1
            if time.perf_counter() - t0 > budget_s / 2:
                break
        dt = (time.perf_counter() - t0) / reps
        return {"value": round(2 * cfg["S"] * n / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"decompress_reduce of {cfg['S']} shards x {n} elements, {reps} reps"}
    if name == "activation_mix_lut":
        x = w.activation_mix(2048, 4096)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.lut_from_histogram(oracle.exponent_histogram(x))
            reps += 1
            if time.perf_counter() - t0 > budget_s / 2:
                break
        dt = (time.perf_counter() - t0) / reps
        return {"value": round(2 * x.size / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"exponent histogram + LUT of the first {x.size} elements of the workload, {reps} reps"}
    n = 1 << 23
    x = w.gaussian(n, sigma, seed=0) if not name.startswith("activation_mix") else w.activation_mix(2048, 4096)
    n = x.size
    t0 = time.perf_counter()
    reps = 0
    while True:
        s = oracle.compress(x, lut)
        oracle.decompress(s, n)
        reps += 1
        if time.perf_counter() - t0 > budget_s / 2:
            break
    dt = (time.perf_counter() - t0) / reps
    op = "compress (as batched segments) + decompress" if name == "moe_a2a" else "compress + decompress"
    return {"value": round(2 * 2 * n / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{op} of the first {n} elements of the workload's distribution, {reps} reps"}


def _oracle_slice_worker(name, k, budget_s):
    """One process of cpu_baseline_all_cores: slice k of the workload's
    distribution, generated here, run through the oracle for budget_s."""
    sys.path.insert(0, ROOT)
    import oracle
    from lossless_bf16_exponent_split_gb300 import workloads as w
    cfg = w.CONFIGS[name]
    lut = oracle.lut_from_sigma(cfg["sigma"])
    if name in ("rs_local", "rs_local_own"):
        per = 1 << 18
        streams = [oracle.compress(x, lut) for x in w.reduce_shards(cfg["S"], per, cfg["sigma"], seed=k)]
        step, unit = (lambda: oracle.decompress_reduce(streams, per)), 2 * cfg["S"] * per
    elif name == "activation_mix_lut":
        x = w.activation_mix(256, 4096, seed=k)
        step, unit = (lambda: oracle.exponent_histogram(x)), 2 * x.size
    else:
        x = w.gaussian(1 << 20, cfg["sigma"], seed=k) if not name.startswith("activation_mix") else \
            w.activation_mix(256, 4096, seed=k)
        step, unit = (lambda: oracle.decompress(oracle.compress(x, lut), x.size)), 2 * 2 * x.size
    step()
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        step()
        reps += 1
    return reps * unit, time.perf_counter() - t0


def cpu_baseline_all_cores(name, budget_s=6.0):
    """The same oracle, unchanged, run by one process per host core at once,
    each on its own slice of the workload's distribution: the chunk-parallel
    CPU figure.  Processes start by spawn (this runs after GPU work)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    with cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as pool:
        res = list(pool.map(_oracle_slice_worker, [name] * cores, range(cores), [budget_s] * cores))
    total_bytes = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    what = {"rs_local": "decompress_reduce of 8 shards x 262,144",
            "rs_local_own": "decompress_reduce of 8 shards x 262,144",
            "activation_mix_lut": "exponent histogram of 1,048,576"}.get(name, "compress + decompress of 1,048,576")
    return {"value": round(total_bytes / wall / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle, one process per core", "sample": f"{what} elements per process, {budget_s:.0f} s each"}


# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0, None
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg_name = args.workload
    from lossless_bf16_exponent_split_gb300 import workloads as w
    cfg = w.CONFIGS[cfg_name]
    lut = oracle.lut_from_sigma(cfg["sigma"])
    # each step: a bounded sample of the workload (oracle speed ~0.1-0.3 GB/s)
    if cfg_name in ("rs_local", "rs_local_own"):
        n = 1 << 20
        shards = w.reduce_shards(cfg["S"], n, cfg["sigma"], seed=0)
        lp = cfg.get("local_pos")
        streams = [None if s == lp else oracle.compress(x, lut) for s, x in enumerate(shards)]
        if lp is None:
            step = lambda: oracle.decompress_reduce(streams, n)
        else:
            step = lambda: oracle.decompress_reduce_local(streams, n, local=shards[lp], local_pos=lp)
        unit_bytes = 2 * cfg["S"] * n
        sample = f"decompress_reduce of {cfg['S']} shards x {n} elements per step"
    elif cfg_name == "activation_mix_lut":
        x = w.activation_mix(1024, 4096)
        step = lambda: oracle.lut_from_histogram(oracle.exponent_histogram(x))
        unit_bytes = 2 * x.size
        sample = f"exponent histogram + LUT of {x.size} elements of the workload per step"
    else:
        n = 1 << 21
        x = w.gaussian(n, cfg["sigma"], seed=0)

        def step():
            s = oracle.compress(x, lut)
            oracle.decompress(s, n)
        unit_bytes = 2 * 2 * n
        sample = f"compress + decompress of {n} elements of the workload's distribution per step"
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = unit_bytes / dt / 1e9
    line = {"metric": "compress/decompress GB/s of BF16 input", "value": round(v, 4), "unit": "GB/s",
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": cfg_name, "desc": cfg["desc"]},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import lossless_bf16_exponent_split_gb300 as z
    from lossless_bf16_exponent_split_gb300 import build
    build.build()
    z.lib()

    def measure(workload, steps, warmup, with_e2e):
        """Sets up one workload, times its ops (the timed region, single
        evented launches, the spread pass) and, if asked and the workload has
        one, the end-to-end leg; returns what the JSON line reports."""
        kind, host, sigma, extra = make_inputs(workload, seed=rank)
        lut = z.zccl_lut_from_sigma(sigma)
        stream = torch.cuda.current_stream()
        h = int(stream.cuda_stream)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        st_ptr = status.data_ptr()

        def tdev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

        if kind == "roundtrip":
            n = host.size
            R = 3
            xs = [tdev(host) for _ in range(R)]
            cap = z.zccl_max_compressed_bytes(n)
            outs = [torch.empty(cap, dtype=torch.uint8, device=dev) for _ in range(R)]
            nbs = [torch.zeros(1, dtype=torch.int64, device=dev) for _ in range(R)]
            y = torch.empty(n, dtype=torch.int16, device=dev)
            wsb = z.zccl_workspace_bytes(z.OP_COMPRESS, n)
            ws_c = torch.zeros(wsb, dtype=torch.uint8, device=dev)
            ws_d = torch.zeros(wsb, dtype=torch.uint8, device=dev)

            def comp(r):
                z.check(z.zccl_compress(xs[r].data_ptr(), n, lut, outs[r].data_ptr(), cap, nbs[r].data_ptr(),
                                        ws_c.data_ptr(), wsb, st_ptr, h), "compress")

            def decomp(r):
                z.check(z.zccl_decompress(outs[r].data_ptr(), cap, y.data_ptr(), n, ws_d.data_ptr(), wsb, st_ptr, h),
                        "decompress")

            for r in range(R):
                comp(r)
            torch.cuda.synchronize()
            stream_bytes = int(nbs[0].item())
            names = ["compress", "decompress"]
            alg = {"compress": 2 * n + stream_bytes, "decompress": stream_bytes + 2 * n}
            step_input_bytes = 2 * 2 * n

            # decompress reads a stream compressed one launch before or after in
            # the rotation, never the one just written (part of it is still in L2):
            # not in the interleaved single-launch timing, nor at the start of the
            # decompress batch, which follows the whole compress batch
            off = decompress_offset(warmup, steps, R)
            ops = [("compress", lambda k: comp(k % R)), ("decompress", lambda k: decomp((k + off) % R))]
            cfg_extra = {"n": n, "stream_bytes": stream_bytes, "ratio": round(stream_bytes / (2 * n), 5),
                         "step": "compress batch k + decompress the stream of batch k-1 (k+1 in the rotation "
                                 "when k-1's buffer is the one the compress batch wrote last)",
                         "l2": f"3 rotating buffer sets, {(4 * n + stream_bytes) / 1e6:.0f} MB touched per step "
                               "(> 129 MB L2)"}
        elif kind == "batched":
            m = extra
            payload = tdev(host)
            segs = []
            hid = m.hidden
            outs = []
            for (r0, rows) in m.segments:
                nn = rows * hid
                cap = z.zccl_max_compressed_bytes(nn)
                o = torch.empty(cap, dtype=torch.uint8, device=dev)
                outs.append(o)
                segs.append((payload[r0 * hid:(r0 + rows) * hid], o))
            codec = z.Codec(dev)
            table = codec.segment_table(segs)
            total_n = host.size
            nb = torch.zeros(len(segs), dtype=torch.int64, device=dev)
            wsb = z.zccl_workspace_bytes(z.OP_COMPRESS_BATCHED, total_n, len(segs))
            ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)

            def comp():
                z.check(z.zccl_compress_batched(table.data_ptr(), len(segs), total_n, lut, nb.data_ptr(),
                                                ws.data_ptr(), wsb, st_ptr, h), "compress_batched")
            comp()
            torch.cuda.synchronize()
            sb = int(nb.sum().item())
            names = ["compress"]
            alg = {"compress": 2 * total_n + sb}
            step_input_bytes = 2 * total_n

            ops = [("compress", lambda k: comp())]
            cfg_extra = {"n": total_n, "segments": len(segs), "stream_bytes": sb,
                         "step": "one batched compress of all static+dynamic segments",
                         "l2": "input 537 MB > 129 MB L2"}
        elif kind == "histogram":
            n = host.size
            R = 5
            xs = [tdev(host) for _ in range(R)]
            hist = torch.empty(256, dtype=torch.int64, device=dev)

            def hist_call(r):
                z.check(z.zccl_exponent_histogram(xs[r].data_ptr(), n, hist.data_ptr(), 0, h), "exponent_histogram")
            names = ["histogram"]
            alg = {"histogram": 2 * n + 256 * 8}
            step_input_bytes = 2 * n

            ops = [("histogram", lambda k: hist_call(k % R))]
            hist_call(0)
            hh0 = hist.cpu().numpy().view(np.uint64).astype(np.float64)
            lut_data = z.zccl_lut_from_histogram(hist.cpu().numpy().view(np.uint64))
            coverage = {"sigma_lut": round(float(hh0[list(lut)].sum() / n), 6),
                        "data_lut": round(float(hh0[list(lut_data)].sum() / n), 6),
                        "sigma": sigma, "data_lut_exponents": list(lut_data)}
            cfg_extra = {"n": n, "step": "one exponent histogram pass (zeroing + counting kernel, PDL pair)",
                         "top7_coverage": coverage,
                         "l2": f"5 rotating inputs; {4 * 2 * n >> 20} MiB read between two reads of one (> 129 MB L2)"}
        else:  # reduce (with the rank's own shard uncompressed at local_pos, if given)
            shards = host
            local_pos = extra
            S = len(shards)
            n = shards[0].size
            codec = z.Codec(dev)
            # three copies of the step's inputs (streams, local shard) and outputs,
            # used in rotation: two other calls (442 MB) run between two reads of one
            R = 3
            sets = []
            for _ in range(R):
                streams, sizes = [], []
                for s_, x in enumerate(shards):
                    if s_ == local_pos:
                        streams.append(None)
                        sizes.append(None)
                        continue
                    o, nbt = codec.compress(tdev(x), lut)
                    streams.append(o)
                    sizes.append(nbt)
                torch.cuda.synchronize()
                sizes_h = [0 if v is None else int(v.item()) for v in sizes]
                ptrs = torch.tensor([0 if o is None else o.data_ptr() for o in streams], dtype=torch.int64, device=dev)
                inb = torch.tensor(sizes_h, dtype=torch.int64, device=dev)
                local_x = tdev(shards[local_pos]) if local_pos is not None else None
                y = torch.empty(n, dtype=torch.int16, device=dev)
                sets.append((streams, ptrs, inb, local_x, y))
            wsb = z.zccl_workspace_bytes(z.OP_DECOMPRESS_REDUCE, n, S)
            ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)

            def red(k):
                _, ptrs, inb, local_x, y = sets[k % R]
                if local_x is None:
                    z.check(z.zccl_decompress_reduce(ptrs.data_ptr(), inb.data_ptr(), S, y.data_ptr(), n,
                                                     ws.data_ptr(), wsb, st_ptr, h), "decompress_reduce")
                else:
                    z.check(z.zccl_decompress_reduce_local(ptrs.data_ptr(), inb.data_ptr(), S, local_x.data_ptr(),
                                                           local_pos, 0, y.data_ptr(), n, ws.data_ptr(), wsb, st_ptr,
                                                           h), "decompress_reduce_local")
            names = ["decompress_reduce"]
            alg = {"decompress_reduce": sum(sizes_h) + (2 * n if local_pos is not None else 0) + 2 * n}
            step_input_bytes = 2 * S * n
            ops = [("decompress_reduce", red)]
            cfg_extra = {"n": n, "shards": S, "stream_bytes_total": sum(sizes_h),
                         "step": "one fused decompress+reduce of S shards"
                                 + (f" (shard {local_pos} uncompressed)" if local_pos is not None else ""),
                         "l2": f"{R} rotating copies of the inputs and output; "
                               f"{(R - 1) * (sum(sizes_h) + 2 * n + (2 * n if local_pos is not None else 0)) >> 20} MiB "
                               "touched between two reads of one (> 129 MB L2)"}

        # ---- warm-up, then K timed steps ----
        for k in range(warmup):
            for _, fn in ops:
                fn(k + 1)
        torch.cuda.synchronize()
        status.zero_()
        op_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ops]
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        barrier(pg, dev)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            wall0 = time.perf_counter()
            # a ~1 ms GPU sleep before the start event gives the host a head start,
            # so no event brackets time the GPU spends waiting for the host to
            # enqueue (the sleep itself is outside the timed region)
            torch.cuda._sleep(2_000_000)
            t_start.record(stream)
            # the K steps' work op by op: each op's K launches run back to back
            # between one pair of events, so a launch's time is its share of that
            # span (an event pair around every launch would also time the event's
            # wait for the previous kernel to drain)
            for (nm, fn), (e0, e1) in zip(ops, op_ev):
                e0.record(stream)
                for k in range(steps):
                    fn(warmup + 1 + k)
                e1.record(stream)
            t_end.record(stream)
            torch.cuda.synchronize()
            wall = time.perf_counter() - wall0
        barrier(pg, dev)
        st = int(status.item())
        if st != 0:
            raise SystemExit(f"device status {st} ({z.status_string(st)}) during the timed region")
        k_ms = {nm: e0.elapsed_time(e1) / steps for (nm, _), (e0, e1) in zip(ops, op_ev)}
        region_ms = t_start.elapsed_time(t_end)
        ms_per_step = max_over_ranks(pg, region_ms / steps, dev)
        value = aggregate_gbs(world, step_input_bytes, ms_per_step)

        # ---- the same launches one at a time, each between its own events ----
        # (outside the timed region: what a caller timing a single call sees)
        S1 = min(steps, 10)
        sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(S1)]
        torch.cuda.synchronize()
        torch.cuda._sleep(2_000_000)
        for k in range(S1):
            sev[k][0].record(stream)
            for i, (_, fn) in enumerate(ops):
                fn(warmup + steps + 1 + k)
                sev[k][i + 1].record(stream)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise SystemExit(f"device status {int(status.item())} after the single-launch timing")
        single = {nm: [sev[k][i].elapsed_time(sev[k][i + 1]) for k in range(S1)] for i, (nm, _) in enumerate(ops)}

        # ---- spread: the same back-to-back runs again, with events at the
        # boundaries of up to 6 groups (each inner event adds a drain, so these
        # group means are a little above the timed region's) ----
        bounds = group_bounds(steps)
        n_groups = len(bounds) - 1
        gev = [[torch.cuda.Event(enable_timing=True) for _ in bounds] for _ in ops]
        torch.cuda.synchronize()
        torch.cuda._sleep(2_000_000)
        for (nm, fn), evs in zip(ops, gev):
            evs[0].record(stream)
            for g in range(n_groups):
                for k in range(bounds[g], bounds[g + 1]):
                    fn(warmup + steps + S1 + 1 + k)
                evs[g + 1].record(stream)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise SystemExit(f"device status {int(status.item())} after the spread pass")
        k_groups = {nm: [evs[g].elapsed_time(evs[g + 1]) / (bounds[g + 1] - bounds[g]) for g in range(n_groups)]
                    for (nm, _), evs in zip(ops, gev)}

        # ---- end to end through the C ABI with host buffers ----
        e2e = None
        if kind == "roundtrip" and not (not with_e2e):
            # Pipelined as a user would: step k's upload (pinned host -> device)
            # runs on one copy stream and step k-1's download on another while
            # step k-1's compress + decompress run, with two buffer slots.  Every
            # step's copies are inside the timed region.
            hx = torch.from_numpy(host.view(np.int16)).pin_memory()
            hy = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(2)]
            hnb = [torch.empty(1, dtype=torch.int64).pin_memory() for _ in range(2)]
            ys = [y, torch.empty(n, dtype=torch.int16, device=dev)]
            s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            in_done = [torch.cuda.Event() for _ in range(2)]
            comp_done = [torch.cuda.Event() for _ in range(2)]
            out_done = [torch.cuda.Event() for _ in range(2)]
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)

            def e2e_step(k):
                i = k % 2
                with torch.cuda.stream(s_in):
                    s_in.wait_event(comp_done[i])  # step k-2 has finished reading slot i
                    xs[i].copy_(hx, non_blocking=True)
                    in_done[i].record(s_in)
                stream.wait_event(in_done[i])
                stream.wait_event(out_done[i])  # step k-2's download has read ys[i]
                comp(i)
                z.check(z.zccl_decompress(outs[i].data_ptr(), cap, ys[i].data_ptr(), n, ws_d.data_ptr(), wsb, st_ptr,
                                          h), "decompress")
                comp_done[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[i])
                    hy[i].copy_(ys[i], non_blocking=True)
                    hnb[i].copy_(nbs[i], non_blocking=True)
                    out_done[i].record(s_out)
            for k in range(2):
                e2e_step(k)
            torch.cuda.synchronize()
            ev0.record(stream)
            s_in.wait_event(ev0)
            s_out.wait_event(ev0)
            for k in range(steps):
                e2e_step(k)
            stream.wait_event(out_done[0])
            stream.wait_event(out_done[1])
            ev1.record(stream)
            torch.cuda.synchronize()
            e2e_ms = ev0.elapsed_time(ev1) / steps
            e2e_ms = max_over_ranks(pg, e2e_ms, dev)
            for i in range(min(2, steps)):
                assert np.array_equal(hy[i].numpy().view(np.uint16), host), "e2e round trip not bit-exact"
            e2e = {"value": round(world * 2 * 2 * n / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                   "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": 2 * n, "d2h_bytes_per_step": 2 * n + 8,
                   "path": "pinned host -> H2D -> zccl_compress -> zccl_decompress -> D2H, "
                           "uploads and downloads of neighbouring steps overlapped on two copy streams"}

        if kind == "histogram" and not (not with_e2e):
            hx = torch.from_numpy(host.view(np.int16)).pin_memory()
            hh = torch.empty(256, dtype=torch.int64).pin_memory()
            luts = []

            def e2e_step():
                xs[0].copy_(hx, non_blocking=True)
                hist_call(0)
                hh.copy_(hist, non_blocking=True)
                torch.cuda.current_stream().synchronize()
                luts.append(z.zccl_lut_from_histogram(hh.numpy().view(np.uint64)))
            for _ in range(2):
                e2e_step()
            torch.cuda.synchronize()
            barrier(pg, dev)
            t0 = time.perf_counter()
            for _ in range(steps):
                e2e_step()
            e2e_ms = (time.perf_counter() - t0) * 1e3 / steps
            e2e_ms = max_over_ranks(pg, e2e_ms, dev)
            assert len(set(luts)) == 1
            e2e = {"value": round(world * 2 * n / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                   "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": 2 * n, "d2h_bytes_per_step": 256 * 8,
                   "path": "pinned host -> H2D -> zccl_exponent_histogram -> D2H -> zccl_lut_from_histogram",
                   "lut": list(luts[0])}

        return {"kind": kind, "names": names, "alg": alg, "k_ms": k_ms, "single": single, "k_groups": k_groups,
                "clocks": clk.summary(), "wall": wall, "ms_per_step": ms_per_step, "value": value,
                "cfg_extra": cfg_extra, "e2e": e2e, "step_input_bytes": step_input_bytes}

    m = measure(args.workload, args.steps, args.warmup, not args.no_e2e)
    names, alg, k_ms, single, k_groups = m["names"], m["alg"], m["k_ms"], m["single"], m["k_groups"]
    ms_per_step, value, cfg_extra, e2e, wall = m["ms_per_step"], m["value"], m["cfg_extra"], m["e2e"], m["wall"]
    step_input_bytes = m["step_input_bytes"]
    # every other workload, measured the same way (fewer steps) and reported
    # beside the headline, when the default workload runs on one GPU
    configs = None
    if args.workload == DEFAULT_WORKLOAD and world == 1 and not args.no_configs:
        configs = {}
        for w in CONFIG_WORKLOADS:
            mm = measure(w, min(args.steps, 20), min(args.warmup, 3), False)
            configs[w] = config_record(w, mm)
            del mm
            torch.cuda.synchronize()
            torch.cuda.empty_cache()

    if rank != 0:
        return
    peak, peak_kind = hbm_peak()
    dom = max(k_ms, key=k_ms.get)
    achieved = alg[dom] / (k_ms[dom] * 1e-3) / 1e9
    kernels = {}
    for nm in names:
        a = alg[nm] / (k_ms[nm] * 1e-3) / 1e9
        inp = (step_input_bytes / len(names)) / (k_ms[nm] * 1e-3) / 1e9
        q = np.percentile(single[nm], [10, 50, 90])
        a1 = alg[nm] / (float(q[1]) * 1e-3) / 1e9
        qg = np.percentile(k_groups[nm], [10, 50, 90])
        kernels[nm] = {"ms": round(k_ms[nm], 4),
                       "timing": f"{args.steps} launches back to back, one event pair",
                       "spread_pass_group_ms_p10_median_p90": [round(float(x), 4) for x in qg],
                       "bf16_input_gbs": round(inp, 2), "algorithmic_bytes": alg[nm], "achieved_gbs": round(a, 2),
                       "frac_of_" + peak_kind: round(a / peak, 4),
                       "single_launch_evented": {"launches": len(single[nm]),
                                                 "ms_p10_median_p90": [round(float(x), 4) for x in q],
                                                 "achieved_gbs_median": round(a1, 2),
                                                 "frac_of_" + peak_kind: round(a1 / peak, 4)}}
    line = {
        "metric": "compress/decompress GB/s of BF16 input",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
        "config": {"workload": args.workload, "desc": workload_desc(args.workload), **cfg_extra,
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": dom, "launches": OP_KERNELS[dom],
                     "duration": f"mean of {args.steps} back-to-back launches in the timed region "
                                 "(CUDA events on the launching stream)",
                     "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": ncu_traffic(dom, args.workload),
                     "algorithmic_bytes_per_launch": alg[dom]},
        "kernels": kernels,
        "gpu_launches": sum(OP_LAUNCHES[nm] for nm in names) * args.steps,
        "clocks": m["clocks"],
        "wall_s_timed_region": round(wall, 4),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if configs is not None:
        line["configs"] = configs
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(args.workload)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
