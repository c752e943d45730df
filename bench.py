"""Benchmark of the layout-folded bf16 -> fp32 reduce-scatter fold and the
all-gather placement.

One step = one pass of the hot path over one gradient group: the fused
reduce-scatter fold of W virtual ranks (tide_rs_fold) followed by the
all-gather placement of W bf16 shard slots into the group's full parameter
tensors (tide_ag_place).  Default workload: the largest group that fits one
GPU, one Qwen3-30B-A3B-style MoE layer with W = 32 (389 parameters,
623,116,288 elements per gradient set, 42.37 GB of algorithmic reduce-scatter
bytes).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``value`` is the reduce-scatter's effective
bandwidth, the metric: W*N*2 bytes read + N*4 written (+N*4 read when
accumulating) per fold, summed over all GPUs, over the slowest rank's mean
fold time (CUDA events around every fold of the timed steps).  The whole
step (fold + placement, whose bytes are N*2 read + N*2 written) is reported
under ``step``; ``per_config`` times the fold, the step and the two-pass
baseline on all five workloads.  Inputs are larger than L2 (no flush
needed); timing uses CUDA events on the launching stream.

``--impl reference`` times the CPU oracle (the plain two-pass definition) on
a bounded sample of the same workload, on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import os

os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")  # before CUDA starts: separate queues per stream
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused bf16→fp32 reduce-scatter effective GB/s and % of GB300 HBM roofline"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "qwen3_30b_a3b_moe_layer"


ORDERS = {"rank": 0, "staged": 1, "nodes": 2, "tree": 3}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--ag-mode", choices=["sm", "ce2d", "ce1d"], default="sm")
    ap.add_argument("--kernel", choices=["auto", "direct", "bulk"], default="auto")
    ap.add_argument("--sched", choices=["auto", "static", "dynamic", "per_item"], default="auto",
                    help="fold schedule (auto: the library default, dynamic)")
    ap.add_argument("--cta-budget", type=int, default=0)
    ap.add_argument("--chunk-bytes", type=int, default=0)
    ap.add_argument("--fill-bytes", type=int, default=0, help="bulk kernel: bytes per rank per stage fill")
    ap.add_argument("--fill-ranks", type=int, default=0, help="bulk kernel: ranks per stage fill")
    ap.add_argument("--ce-streams", type=int, default=0, help="copy-engine placement: internal streams")
    ap.add_argument("--order", choices=list(ORDERS), default="rank",
                    help="summation order of the fold (rank order is the bit-exact contract)")
    ap.add_argument("--node-size", type=int, default=0, help="two-level order: ranks per node (0: half the world)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-baseline", action="store_true", help="skip the two-pass GPU baseline")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--no-interference", action="store_true", help="skip the concurrent-GEMM harness")
    ap.add_argument("--no-variants", action="store_true", help="skip timing the other placement variants")
    ap.add_argument("--no-per-config", action="store_true", help="skip timing the five workloads one by one")
    ap.add_argument("--interference-rs", type=int, default=10, help="reduce-scatters per interference co-run")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU baseline: seconds of single-threaded oracle work (half that on all cores)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The maximum of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, world: int, ms_per_step: float) -> float:
    """Effective GB/s of the whole job: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


def alg_bytes(w, numel: int):
    rs = w.world * numel * 2 + numel * 4 + (numel * 4 if w.accumulate else 0)
    ag = numel * 2 + numel * 2
    return rs, ag


def nvml_device(cuda_index: int):
    """(NVML library, device handle) of the CUDA device, matched by UUID
    (read-only use: nothing is set through it)."""
    import ctypes
    lib = ctypes.CDLL("libnvidia-ml.so.1")
    if lib.nvmlInit_v2() != 0:
        raise OSError("nvmlInit failed")
    count = ctypes.c_uint(0)
    lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
    want = ""
    try:
        import torch
        want = str(torch.cuda.get_device_properties(cuda_index).uuid).lower().replace("gpu-", "")
    except Exception:
        pass
    for i in range(count.value):
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
            continue
        buf = ctypes.create_string_buffer(96)
        lib.nvmlDeviceGetUUID(h, buf, 96)
        if want and want in buf.value.decode().lower():
            return lib, h
    h = ctypes.c_void_p()
    if lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
        raise OSError("no NVML handle")
    return lib, h


def gpu_local_cpus(cuda_index: int):
    """The CPUs NVML names as closest to the GPU (its NUMA-local cores), or
    None when NVML cannot tell."""
    import ctypes
    import os
    try:
        lib, h = nvml_device(cuda_index)
        words = (os.cpu_count() or 64) // 64 + 1
        mask = (ctypes.c_ulong * words)()
        if lib.nvmlDeviceGetCpuAffinity(h, words, mask) != 0:
            return None
    except (OSError, AttributeError):
        return None
    bits = ctypes.sizeof(ctypes.c_ulong) * 8
    cpus = {w * bits + b for w in range(words) for b in range(bits) if (mask[w] >> b) & 1}
    return cpus or None


def cpu_ranges(cpus) -> str:
    """Compact text of a CPU set: 0-71,144-215."""
    out, xs = [], sorted(cpus)
    i = 0
    while i < len(xs):
        j = i
        while j + 1 < len(xs) and xs[j + 1] == xs[j] + 1:
            j += 1
        out.append(f"{xs[i]}-{xs[j]}" if j > i else f"{xs[i]}")
        i = j + 1
    return ",".join(out)


class ClockSampler:
    """SM clock, max clock, power and clock-event (throttle) reasons sampled
    every ~2 ms while the timed region runs.  Reads NVML through ctypes (read
    only: no setting is changed); falls back to `nvidia-smi -lms 100`."""
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []  # (time, sm_mhz, max_mhz, power_w, reasons_mask)
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None

    def _nvml(self):
        lib, chosen = nvml_device(self.cuda_index)
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, chosen, reasons_fn

    def start(self):
        import ctypes
        try:
            lib, h, reasons_fn = self._nvml()
        except (OSError, AttributeError):
            return self._start_smi()
        self.source = "nvml"
        clk, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

        def loop():
            while not self._stop.is_set():
                lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
                lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
                lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                reasons_fn(h, ctypes.byref(rs))
                self.samples.append((time.time(), clk.value, mx.value, pw.value / 1000.0, rs.value))
                time.sleep(0.002)
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def _start_smi(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self._smi = subprocess.Popen(["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            return
        self.source = "nvidia-smi"
        bits = [0x8, 0x40, 0x20, 0x4]

        def loop():
            for line in self._smi.stdout:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    mask = sum(b for b, v in zip(bits, parts[3:7]) if v.lower() == "active")
                    self.samples.append((time.time(), float(parts[0]), float(parts[1]), float(parts[2]), mask))
                except ValueError:
                    continue
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._smi:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
        if self._thread:
            self._thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        window = "timed"
        if not inside:
            inside = [x for x in self.samples if t0 - 1.0 <= x[0] <= t1 + 1.0]
            window = "timed+-1s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        sm = sorted(x[1] for x in inside)
        mask = 0
        for x in inside:
            mask |= int(x[4])
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(x[2] for x in inside),
                "reasons": sorted(name for bit, name in self.REASONS.items() if mask & bit),
                "samples": len(inside), "window": window, "source": self.source,
                "power_w_max": round(max(x[3] for x in inside), 1)}


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_digest() -> str:
    """sha256 (16 hex digits) of the fold kernels' code: rs_fold.cu without
    its // comments and blank lines, so that comment edits keep profiles valid."""
    import hashlib
    import re
    with open(os.path.join(ROOT, "all_gather_gb300", "csrc", "rs_fold.cu")) as f:
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in f]
    code = "\n".join(ln for ln in lines if ln.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def _profile_kv(name: str):
    """key: value lines of a committed profile summary, or None if missing or
    if the fold kernels' code changed since the summary was taken."""
    try:
        digest = kernel_digest()
        kv = {}
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
    except OSError:
        return None
    return kv if kv.get("rs_fold_cu_sha256_16") == digest else None


SM_TIME_CASE = "llama3.1_8b_attn"  # the reduced case whose two-pass kernels fit a narrow capture


def profile_sm_time(workload: str):
    """SM time of one reduce-scatter, fused vs two-pass, from the committed ncu
    summary of this workload or else of the reduced case (named in the record)."""
    for name in (workload, SM_TIME_CASE):
        kv = _profile_kv(f"sm_time_{name}.txt")
        if kv:
            break
    else:
        return None
    try:
        f, b = float(kv["fused_sm_ms_per_rs"]), float(kv["two_pass_sm_ms_per_rs"])
        return {"workload": name, "fused_sm_ms_per_rs": f, "two_pass_sm_ms_per_rs": b, "ratio": round(b / f, 2),
                "fused_sm_ms_per_gb": float(kv["fused_sm_ms_per_gb"]),
                "two_pass_sm_ms_per_gb": float(kv["two_pass_sm_ms_per_gb"]),
                "fused_dram_gb_per_rs": float(kv["fused_dram_gb_per_rs"]),
                "two_pass_dram_gb_per_rs": float(kv["two_pass_dram_gb_per_rs"]),
                "source": f"profiles/sm_time_{name}.txt (ncu sm__cycles_active.sum)"}
    except (KeyError, ValueError):
        return None


def profile_traffic(workload: str):
    """Per-launch DRAM bytes of the fold kernel from the committed ncu summary,
    or None if there is none or the kernel code changed since it was taken."""
    kv = _profile_kv(f"rs_fold_{workload}_traffic.txt")
    try:
        return float(kv["traffic_bytes_per_launch"]) if kv else None
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
def sample_params(w):
    """The CPU sample of a workload: one parameter of each distinct shape, in
    the group's order (every kind of tensor the group holds, each once)."""
    seen, idx = set(), []
    for p, shape in enumerate(w.shapes):
        if shape not in seen:
            seen.add(shape)
            idx.append(p)
    return idx


def sample_text(w, idx) -> str:
    numel = sum(w.numels()[i] for i in idx)
    return (f"one parameter of each of the {len(idx)} distinct shapes of {w.name} "
            f"({', '.join(w.names[i] for i in idx)}), all {w.world} ranks, {numel} elements per gradient set")


def cpu_grads(w, idx):
    """host_grads[j][u]: bf16 bits (uint16) of sample parameter idx[j] on rank u,
    generated on the CPU with the same recipe as on the GPU."""
    import numpy as np
    import torch

    import workloads
    return [[workloads.normal_fp32(w.numels()[i], workloads.grad_seed(w, u, i), w.sigma, "cpu", w.outlier_rate,
                                   w.outlier_scale).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
             for u in range(w.world)] for i in idx]


def rs_alg_bytes(w, numel: int) -> int:
    """The metric's bytes: W*N*2 read + N*4 written (+N*4 read when accumulating)."""
    return alg_bytes(w, numel)[0]


def cpu_oracle_sample(w, host_grads, idx, min_seconds=10.0, max_reps=50):
    """Time the CPU oracle's reduce-scatter (the metric) on the sample
    parameters, single-threaded.  host_grads[j][u]: uint16 bf16 bits."""
    import numpy as np

    import oracle
    dims_all = w.dim0_rownumel()
    dims = [dims_all[i] for i in idx]
    orc = oracle.load()
    _, _, S = orc.geometry(w.world, dims)
    out = np.zeros((w.world, S), np.float32)
    numel = sum(d * k for d, k in dims)
    reps, t0 = 0, time.perf_counter()
    while True:
        orc.rs(w.world, dims, host_grads, w.alpha, w.accumulate, out)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return {"value": round(rs_alg_bytes(w, numel) * reps / el / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle", "sample": f"{sample_text(w, idx)}; reduce-scatter, {reps} reps in {el:.1f} s"}


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model"):
        for line in info.splitlines():
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    impl = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")]
    part = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")]
    if not (impl and part):
        return "unknown"
    arm_parts = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2", "0xd4f": "Neoverse-V2"}
    name = arm_parts.get(part[0].lower(), "") if impl[0].lower() == "0x41" else ""
    return f"{name} (implementer {impl[0]} part {part[0]})" if name else f"implementer {impl[0]} part {part[0]}"


def cpu_oracle_all_cores(w, host_grads, idx, min_seconds=5.0, max_reps=50):
    """The same oracle sample on every core this process may use: the
    unchanged oracle function runs on independent windows (slices of one
    (parameter, rank) piece, at most 2^20 elements) in a thread pool; ctypes
    releases the GIL inside each call.  The windows are first checked to
    reassemble the single-threaded result bit for bit."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    dims_all = w.dim0_rownumel()
    dims = [dims_all[i] for i in idx]
    orc = oracle.load()
    W = w.world
    R, o, S = orc.geometry(W, dims)
    out = np.zeros((W, S), np.float32)
    jobs = []
    for p, (d, k) in enumerate(dims):
        for r in range(W):
            v = orc.valid_rows(d, R[p], r) * k
            base = r * R[p] * k
            for a in range(0, R[p] * k, 1 << 20):
                b = min(a + (1 << 20), R[p] * k)
                nv, npad = max(0, min(b, v) - a), (b - a) - max(0, min(b, v) - a)
                srcs = [host_grads[p][u][base + a:base + a + nv] for u in range(W)]
                jobs.append((srcs, nv, npad, r, o[p] + a))

    def rs_job(j, dst):
        srcs, nv, npad, r, pos = j
        old = dst[r, pos:pos + nv + npad] if w.accumulate else None
        dst[r, pos:pos + nv + npad] = orc.rs_window(srcs, nv, npad, w.alpha, w.accumulate, old)

    threads = len(os.sched_getaffinity(0))
    numel = sum(d * k for d, k in dims)
    with ThreadPoolExecutor(max_workers=threads) as pool:
        chk, want = np.zeros((W, S), np.float32), np.zeros((W, S), np.float32)
        list(pool.map(lambda j: rs_job(j, chk), jobs))
        orc.rs(W, dims, host_grads, w.alpha, w.accumulate, want)
        if not np.array_equal(chk.view(np.uint32), want.view(np.uint32)):
            raise AssertionError("parallel oracle windows differ from the single-threaded oracle")
        del chk, want
        reps, t0 = 0, time.perf_counter()
        while True:
            list(pool.map(lambda j: rs_job(j, out), jobs))
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or reps >= max_reps:
                break
    return {"value": round(rs_alg_bytes(w, numel) * reps / el / 1e9, 4), "unit": UNIT, "cores": threads,
            "cpu": cpu_model(), "matches_single_thread": True,
            "sample": f"same sample, {len(jobs)} reduce-scatter windows per rep over {threads} threads, "
                      f"{reps} reps in {el:.1f} s"}


def run_reference(args):
    """The reference arm: the CPU oracle's reduce-scatter (the metric) on the
    sample parameters of the same workload, single-threaded on this host, each
    step one reduce-scatter of the sample."""
    world, rank, _ = dist_env()
    import workloads
    w = workloads.get(args.workload)
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    idx = sample_params(w)
    dims_all = w.dim0_rownumel()
    dims = [dims_all[i] for i in idx]
    host = cpu_grads(w, idx)
    orc = oracle.load()
    _, _, S = orc.geometry(w.world, dims)
    out = np.zeros((w.world, S), np.float32)
    numel = sum(d * k for d, k in dims)

    def step():
        orc.rs(w.world, dims, host, w.alpha, w.accumulate, out)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = rs_alg_bytes(w, numel) * args.steps / el / 1e9
    sample = f"{sample_text(w, idx)}; one reduce-scatter per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": w.name, "world": w.world, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                             "cpu": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def pct(xs, q):
    ys = sorted(xs)
    return round(ys[min(len(ys) - 1, int(q * len(ys)))], 4)


def thirds(xs):
    """Medians of the first, middle and last third of the timed steps, the
    median of those, and their spread (max - min) relative to it: drift or a
    co-tenant on the shared GPU shows up here."""
    n = len(xs) // 3
    if n < 1:
        return None
    meds = [pct(xs[i * n:(i + 1) * n], 0.5) for i in range(3)]
    mid = sorted(meds)[1]
    return {"medians_ms": meds, "median_of_medians_ms": mid,
            "spread_pct": round(100.0 * (max(meds) - min(meds)) / mid, 2) if mid > 0 else None}


def timed_steps(plan, w, out, slots, full_b, ag_mode, K, stream):
    """K steps of fold + placement with CUDA events around each part; returns
    per-step fold and placement times (ms) and the whole region's time."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        plan.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)
        ev[i][1].record(stream)
        plan.ag_place(slots, full_b, mode=ag_mode)
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    rs_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ag_ms = [e[1].elapsed_time(e[2]) for e in ev]
    return rs_ms, ag_ms, start.elapsed_time(end)


def fold_record(w, rs_ms, peak):
    numel = w.total_numel()
    rs_b = rs_alg_bytes(w, numel)
    mean = sum(rs_ms) / len(rs_ms)
    gbs = rs_b / (mean * 1e-3) / 1e9
    return {"ms": round(mean, 4), "gbs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
            "frac_of_8tbs_nominal": round(gbs / 8000.0, 4), "alg_bytes": rs_b, "p10_ms": pct(rs_ms, 0.1),
            "p50_ms": pct(rs_ms, 0.5), "p90_ms": pct(rs_ms, 0.9), "thirds": thirds(rs_ms)}


def graph_step(plan, w, out, slots, full_b, steps, step_bytes, overlap=False):
    """The step (fold + placement) captured once in a CUDA graph and replayed:
    the time of the two kernels without the host's per-call enqueue, which
    bounds small groups when launched one call at a time.  overlap: the
    placement runs on a second stream of the graph, beside the fold (the two
    touch disjoint buffers, as a layer's reduce-scatter and the next layer's
    all-gather do)."""
    import torch
    side, side2 = torch.cuda.Stream(), torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        plan.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)
        plan.ag_place(slots, full_b, mode="sm")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        if overlap:
            side2.wait_stream(side)
        plan.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)
        with torch.cuda.stream(side2 if overlap else side):
            plan.ag_place(slots, full_b, mode="sm")
        if overlap:
            side.wait_stream(side2)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        g.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    mean = sum(ms) / steps
    del g
    what = "tide_rs_fold + tide_ag_place captured once, graph replayed"
    return {"ms": round(mean, 4), "p50_ms": pct(ms, 0.5), "gbs": round(step_bytes / (mean * 1e-3) / 1e9, 1),
            "what": what + (", placement on a second stream beside the fold" if overlap else "")}


def measure_config(w, dev, steps, peak, gs=None, baseline=True):
    """Fold, placement and step times of one workload in the benchmark's launch
    configuration (default flags, SM placement), plus the two-pass baseline's
    reduce-scatter.  Builds (and frees) the workload's inputs unless given."""
    import torch

    import all_gather_gb300 as tide
    import workloads
    from all_gather_gb300 import baselines
    own = gs is None
    gs = workloads.make_grads(w, device=dev) if own else gs
    plan = tide.Plan(gs.views)
    S = plan.slot_numel
    out = workloads.make_out_init(w, S, device=dev) if w.accumulate else torch.zeros(w.world, S, device=dev)
    slots = workloads.make_slots(w, S, device=dev)
    full = [torch.empty(s, dtype=torch.bfloat16, device=dev) for s in w.shapes]
    full_b = plan.bind_full(full)
    stream = torch.cuda.current_stream()
    timed_steps(plan, w, out, slots, full_b, "sm", 3, stream)
    rs_ms, ag_ms, _ = timed_steps(plan, w, out, slots, full_b, "sm", steps, stream)
    # the step alone, events only around the whole region (per-part events cost
    # host time that small groups would otherwise measure)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        plan.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)
        plan.ag_place(slots, full_b, mode="sm")
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    numel = w.total_numel()
    rs_b, ag_b = alg_bytes(w, numel)
    ag_mean = sum(ag_ms) / steps
    rec = {"world": w.world, "params": w.num_params, "elements": numel, "accumulate": w.accumulate,
           "alpha": w.alpha, "steps": steps, "fold": fold_record(w, rs_ms, peak),
           "placement": {"ms": round(ag_mean, 4), "gbs": round(ag_b / (ag_mean * 1e-3) / 1e9, 1), "alg_bytes": ag_b,
                         "p50_ms": pct(ag_ms, 0.5)},
           "step": {"ms": round(total / steps, 4), "gbs": round((rs_b + ag_b) / (total / steps * 1e-3) / 1e9, 1)}}
    rec["step_graph"] = graph_step(plan, w, out, slots, full_b, steps, rs_b + ag_b)
    rec["step_graph_overlapped"] = graph_step(plan, w, out, slots, full_b, steps, rs_b + ag_b, overlap=True)
    if baseline:
        b = baselines.time_two_pass(w, gs.views, S, out, slots, full, steps=min(steps, 5))
        b["fused_speedup_rs"] = round(b["rs_ms"] / rec["fold"]["p50_ms"], 3)
        rec["two_pass_baseline"] = {k: b[k] for k in ("rs_ms", "rs_gbs", "fused_speedup_rs", "pack_buffer_bytes")}
    plan.close()
    del out, slots, full, full_b
    if own:
        del gs
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import all_gather_gb300 as tide
    import workloads
    from all_gather_gb300 import baselines
    from all_gather_gb300 import build as _build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    w = workloads.get(args.workload)
    numel = w.total_numel()
    rs_b, ag_b = alg_bytes(w, numel)
    step_bytes = rs_b + ag_b

    gs = workloads.make_grads(w, device=dev)
    flags = tide.make_flags(cta_budget=args.cta_budget, chunk_bytes=args.chunk_bytes, fill_bytes=args.fill_bytes,
                            fill_ranks=args.fill_ranks, ce_streams=args.ce_streams,
                            sched={"auto": 0, "dynamic": 1, "per_item": 2, "static": 3}[args.sched],
                            kernel={"auto": 0, "direct": 1, "bulk": 2}[args.kernel], order=ORDERS[args.order],
                            node_size=(args.node_size or max(1, w.world // 2)) if args.order == "nodes" else 0)
    plan = tide.Plan(gs.views, flags)
    S = plan.slot_numel
    cfg = plan.fold_config()
    out = workloads.make_out_init(w, S, device=dev) if w.accumulate else torch.zeros(w.world, S, device=dev)
    slots = workloads.make_slots(w, S, device=dev)
    full = [torch.empty(s, dtype=torch.bfloat16, device=dev) for s in w.shapes]
    full_b = plan.bind_full(full)  # checked once, as a training loop would
    stream = torch.cuda.current_stream()
    W_UP = max(args.warmup, 3)
    timed_steps(plan, w, out, slots, full_b, args.ag_mode, W_UP, stream)

    clocks = ClockSampler(local)
    clocks.start()
    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = tide.tide_launch_count()
    switch = sys.getswitchinterval()
    sys.setswitchinterval(1e-4)  # let the clock sampler thread run while this thread launches
    t_wall0 = time.time()
    rs_ms, ag_ms, total_ms = timed_steps(plan, w, out, slots, full_b, args.ag_mode, K, stream)
    t_wall1 = time.time()
    sys.setswitchinterval(switch)
    if world > 1:
        dist.barrier()
    launches = tide.tide_launch_count() - launches0
    clocks.stop()
    rs_mean = sum(rs_ms) / K
    ag_mean = sum(ag_ms) / K
    total_ms = max_over_ranks(total_ms, world, dev)
    rs_mean_max = max_over_ranks(rs_mean, world, dev)
    ms_per_step = total_ms / K
    value = whole_job_gbs(rs_b, world, rs_mean_max)  # the metric: the fold's effective bandwidth
    peak, peak_kind = measured_peak_gbs()
    achieved = rs_b / (rs_mean * 1e-3) / 1e9
    clk = clocks.summary(t_wall0, t_wall1)
    traffic = profile_traffic(w.name) if (args.order == "rank" and args.sched == "auto" and args.cta_budget == 0
                                          and args.kernel in ("auto", "bulk")) else None

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W_UP, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "world": w.world, "params": w.num_params, "elements": numel,
                   "alpha": w.alpha, "accumulate": w.accumulate, "ag_mode": args.ag_mode, "order": args.order,
                   "fold_grid": cfg["grid"], "fold_block": cfg["block"], "fold_items": cfg["items"],
                   "chunk_elems": cfg["chunk_elems"], "l2": "inputs larger than L2 (no flush)",
                   "value": "reduce-scatter fold: world * (W*N*2 + N*4 [+ N*4]) / max-over-ranks mean fold time",
                   "step": "tide_rs_fold + tide_ag_place", "parallelism": f"weak: {world} independent replicas"},
        "step": {"ms": round(ms_per_step, 4), "gbs": round(whole_job_gbs(step_bytes, world, ms_per_step), 2),
                 "alg_bytes": step_bytes, "what": "tide_rs_fold + tide_ag_place, bytes of both"},
        "parts": {"rs_fold": fold_record(w, rs_ms, peak),
                  "ag_place": {"ms": round(ag_mean, 4), "gbs": round(ag_b / (ag_mean * 1e-3) / 1e9, 1),
                               "alg_bytes": ag_b, "p10_ms": pct(ag_ms, 0.1), "p50_ms": pct(ag_ms, 0.5),
                               "p90_ms": pct(ag_ms, 0.9), "thirds": thirds(ag_ms)}},
        "device": {"name": torch.cuda.get_device_name(dev),
                   "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "tide_rs_fold (fold_bulk_kernel)",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "frac_of_8tbs_nominal": round(achieved / 8000.0, 4)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "sm_time": profile_sm_time(w.name) if args.order == "rank" else None,
    }

    # the per-GPU extras at N = 1 only: with N > 1 every rank is an
    # independent replica of the same GPU work
    single = world == 1
    if single and not args.no_variants:
        result["variants"] = time_variants(plan, w, S, slots, full, dev, gs.views, steps=min(K, 20))
        result["host_issue_us"] = host_issue_us({
            "tide_rs_fold": lambda: plan.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate),
            "tide_ag_place sm": lambda: plan.ag_place(slots, full_b, mode="sm"),
            "tide_ag_place sm, full tensors checked per call": lambda: plan.ag_place(slots, full, mode="sm"),
            "tide_ag_place ce2d": lambda: plan.ag_place(slots, full_b, mode="ce2d"),
            "tide_ag_place ce1d": lambda: plan.ag_place(slots, full_b, mode="ce1d")})

    # two-pass stock-FSDP2-style baseline (chunk_cat pack to fp32, then reduce), timed alone
    if not args.no_baseline and single:
        result["baseline_two_pass"] = baselines.time_two_pass(w, gs.views, S, out, slots, full, steps=min(K, 10))
        b = result["baseline_two_pass"]
        b["fused_speedup_rs"] = round(b["rs_ms"] / rs_mean, 3)
        b["fused_speedup_ag"] = round(b["ag_ms"] / ag_mean, 3)

    # concurrent-compute interference (victim GEMMs / elementwise vs the RS arms)
    if not args.no_interference and single:
        from all_gather_gb300 import interference
        result["interference"] = interference.summarize(
            interference.measure(w.name, budgets=(0, 128, 64, 32, 16, 8), n_rs=args.interference_rs, device=local,
                                 grads=gs))
        result["interference"]["sm_probe"] = interference.sm_probe(w.name, budgets=(0, 152, 64, 32, 16, 8), windows=20,
                                                                   device=local, grads=gs)
        result["interference"]["target"] = interference.corun_target(w.name, device=local, grads=gs,
                                                                     n_rs=args.interference_rs)

    # end to end through the public API: pinned host gradients -> device -> fold -> host shards
    if not args.no_e2e:
        result["e2e"] = e2e(args, w, gs, plan, S, out, dev, world)

    if single and not args.no_cpu_baseline:
        idx = sample_params(w)
        host = [[gs.views[u][i].reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16) for u in range(w.world)]
                for i in idx]
        result["cpu_baseline"] = cpu_oracle_sample(w, host, idx, min_seconds=args.cpu_seconds)
        result["cpu_baseline"]["cpu"] = cpu_model()
        result["cpu_baseline"]["all_cores"] = cpu_oracle_all_cores(w, host, idx, min_seconds=args.cpu_seconds / 2)

    plan.close()
    del out, slots, full, full_b
    torch.cuda.empty_cache()

    # every workload in the benchmark's launch configuration (N = 1 only)
    if single and not args.no_per_config:
        per = {}
        for cw in workloads.WORKLOADS:
            same = cw.name == w.name
            per[cw.name] = measure_config(cw, dev, steps=min(K, 20), peak=peak, gs=gs if same else None,
                                          baseline=not args.no_baseline)
        result["per_config"] = per

    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def host_issue_us(calls: dict, reps: int = 30) -> dict:
    """Host time to enqueue each call (from the Python call to its return,
    ctypes marshalling included; the device is idle before every call, so no
    call waits for queue space): median and p90 in microseconds."""
    import torch
    res = {}
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            ts.append((time.perf_counter() - t0) * 1e6)
        torch.cuda.synchronize()
        ts.sort()
        res[name] = {"p50": round(ts[len(ts) // 2], 1), "p90": round(ts[int(0.9 * (len(ts) - 1))], 1)}
    return res


def time_variants(plan, w, S, slots, full, dev, gs_views, steps: int = 20) -> dict:
    """Mean event time of each placement and fold variant over `steps` launches."""
    import torch

    import all_gather_gb300 as tide
    import workloads
    N = w.total_numel()
    slots32 = torch.stack([workloads.normal_fp32(S, workloads.slot_seed(w, r), 0.02, dev) for r in range(w.world)])
    stream = torch.cuda.current_stream()
    full_b = plan.bind_full(full)
    calls = {
        "ag_place_f32 (fp32 master shards -> bf16, fused cast)": (lambda: plan.ag_place_f32(slots32, full_b), 6 * N),
        "ag_place ce2d (copy engines, one 2D copy per parameter)": (lambda: plan.ag_place(slots, full_b, "ce2d"),
                                                                    4 * N),
        "ag_place ce1d (copy engines, one copy per piece)": (lambda: plan.ag_place(slots, full_b, "ce1d"), 4 * N),
    }
    # the fold in the other Section 4.3 orders, the tree order, and with fp32 gradients
    out_v = torch.zeros(w.world, S, device=dev)
    rs_b = w.world * N * 2 + N * 4 + (N * 4 if w.accumulate else 0)
    L = max(1, w.world // 2)
    plans = {
        "rs_fold order=staged_own (one-node Level 1 order)": tide.Plan(
            gs_views, tide.make_flags(order=tide.TIDE_ORDER_STAGED_OWN)),
        f"rs_fold order=nodes node_size={L} (two-level order)": tide.Plan(
            gs_views, tide.make_flags(order=tide.TIDE_ORDER_NODES, node_size=L)),
        "rs_fold order=tree (pairwise)": tide.Plan(gs_views, tide.make_flags(order=tide.TIDE_ORDER_TREE)),
    }
    for name, pl in plans.items():
        calls[name] = ((lambda pl=pl: pl.rs_fold(out_v, alpha=w.alpha, accumulate=w.accumulate)), rs_b)
    grads32 = [[v.float() for v in vs] for vs in gs_views]
    plan32 = tide.Plan(grads32, tide.make_flags(grad_dtype=tide.TIDE_DTYPE_F32))
    calls["rs_fold fp32 gradients (b_grad = 4)"] = (
        lambda: plan32.rs_fold(out_v, alpha=w.alpha, accumulate=w.accumulate),
        w.world * N * 4 + N * 4 + (N * 4 if w.accumulate else 0))
    # the copy-engine placement captured once and replayed from a CUDA graph:
    # no per-step host issue of the copy list
    graphs = {}
    for mode in ("ce2d", "ce1d"):
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            plan.ag_place(slots, full_b, mode)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            plan.ag_place(slots, full_b, mode)
        graphs[mode] = g
    calls["ag_place ce2d from a CUDA graph (replay)"] = (graphs["ce2d"].replay, 4 * N)
    calls["ag_place ce1d from a CUDA graph (replay)"] = (graphs["ce1d"].replay, 4 * N)
    res = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record(stream)
        for _ in range(steps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / steps
        res[name] = {"ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "alg_bytes": nbytes}
    del graphs
    for pl in list(plans.values()) + [plan32]:
        pl.close()
    del slots32, grads32, out_v
    torch.cuda.empty_cache()
    return res


def e2e(args, w, gs, plan, S, out, dev, world):
    """The metric end to end through the public API with host buffers.  Every
    step's W gradient sets start in pinned host memory and its fp32 shards end
    there.  Main form: a plan built on the host gradients folds them in place,
    reading them over the host link (NVLink-C2C on Grace), and each step's
    shards are read back while the next step folds (two device output
    buffers).  For comparison (`staged`): the copy engines upload the
    gradients to device buffers every step and the device-resident plan folds
    them (two device buffer sets on upload / fold / read-back streams).  The
    value is the reduce-scatter's algorithmic bytes over the time per step."""
    import os

    import torch
    # Host buffers on the GPU's own NUMA node: pinned pages are placed where
    # the allocating thread runs, and a GB300 tray has two Grace CPUs, each
    # attached to its own GPUs; buffers on the far one cross the CPU-to-CPU
    # link on every copy.
    def pow2(n):  # torch's pinned-memory allocator rounds each block up to a power of two
        return 1 << max(0, int(n - 1).bit_length())
    grad_bytes = sum(pow2(a.numel() * a.element_size()) for a in gs.arenas)
    out_bytes = pow2(out.numel() * 4)
    need = grad_bytes + 3 * out_bytes  # pinned: the gradients, the old shards, two read-back buffers
    avail = host_mem_available() // max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    if need * 1.25 > avail:
        return {"skipped": f"host memory: the pinned buffers need {need / 1e9:.1f} GB, "
                           f"{avail / 1e9:.1f} GB available to this rank", "unit": UNIT}
    saved = os.sched_getaffinity(0)
    local = gpu_local_cpus(torch.device(dev).index or 0)
    use = (local & saved) if local else None
    if use:
        os.sched_setaffinity(0, use)
    try:
        h_arenas = [_pinned_copy(a) for a in gs.arenas]  # every step's inputs: the same bytes
        res = _e2e_in_place(args, w, gs, h_arenas, S, out, dev, world)
        if world == 1:  # the comparison needs a second device copy of the gradients: one GPU only
            res["staged"] = _e2e_staged(args, w, gs, h_arenas, plan, S, out, dev, world)
        del h_arenas
    finally:
        os.sched_setaffinity(0, saved)
    res["host_cpus"] = {"gpu_local": cpu_ranges(local) if local else None,
                        "used": cpu_ranges(use) if use else cpu_ranges(saved)}
    return res


def host_mem_available() -> int:
    """MemAvailable of /proc/meminfo in bytes (0 if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return 0


def _pinned_copy(t):
    """A pinned host copy of a device tensor (allocated pinned, no pageable staging)."""
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def _e2e_in_place(args, w, gs, h_arenas, S, out, dev, world):
    import torch
    import torch.distributed as dist

    import all_gather_gb300 as tide
    K = max(2, args.e2e_steps)
    # the host gradients as per-parameter views into the pinned arenas (the device layout)
    h_views = [[h[o:o + v.numel()].view(v.shape) for o, v in zip(gs.offsets, gs.views[u])]
               for u, h in enumerate(h_arenas)]
    plan_h = tide.Plan(h_views)  # gradients in host memory: folded in place over the host link
    h_out0 = _pinned_copy(out)
    outs = [torch.empty_like(out) for _ in range(2)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(a.numel() * a.element_size() for a in h_arenas) + (h_out0.numel() * 4 if w.accumulate else 0)
    d2h = h_out0.numel() * 4
    s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("comp", "out")}

    def step(i, first):
        b = i % 2
        with torch.cuda.stream(s_comp):
            if not first[b]:
                s_comp.wait_event(ev["out"][b])  # the shards of set b were read back
            if w.accumulate:
                outs[b].copy_(h_out0, non_blocking=True)
            plan_h.rs_fold(outs[b], alpha=w.alpha, accumulate=w.accumulate, stream=s_comp)
            ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            h_outs[b].copy_(outs[b], non_blocking=True)
            ev["out"][b].record(s_out)
        first[b] = False

    first = [True, True]
    for i in range(2):
        step(i, first)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_comp)
    for i in range(K):
        step(i, first)
    s_out.wait_stream(s_comp)
    end.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / K, world, dev)
    last = (K - 1) % 2
    ok = torch.equal(h_outs[last], outs[last].cpu())  # read-back == on-device result
    plan_h.close()
    del outs, h_outs, h_out0, h_views
    torch.cuda.empty_cache()
    return {"value": round(whole_job_gbs(rs_alg_bytes(w, w.total_numel()), world, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "steps": K,
            "readback_matches_device": ok,
            "mode": "gradients read in place from pinned host memory by tide_rs_fold (over the host link, no "
                    "staging copy); fp32 shards -> pinned host every step",
            "note": "h2d bytes: the gradients the fold reads from host memory each step (+ old shards when "
                    "accumulating)"}


def _e2e_staged(args, w, gs, h_arenas, plan, S, out, dev, world):
    import torch
    import torch.distributed as dist

    import all_gather_gb300 as tide
    import workloads
    K = max(2, args.e2e_steps)
    h_out0 = _pinned_copy(out)
    h_outs = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    gs2 = workloads.make_grads(w, device=dev)  # the second device buffer set has its own arenas and plan
    plan2 = tide.Plan(gs2.views)
    sets = [(gs.arenas, plan, out), (gs2.arenas, plan2, torch.empty_like(out))]
    h2d = sum(a.numel() * a.element_size() for a in h_arenas) + (h_out0.numel() * 4 if w.accumulate else 0)
    d2h = h_out0.numel() * 4
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}

    def step(i, first):
        b = i % 2
        arenas, pl, o = sets[b]
        with torch.cuda.stream(s_in):
            if not first[b]:
                s_in.wait_event(ev["comp"][b])  # device inputs of set b are free again
                s_in.wait_event(ev["out"][b])   # and its shards were read back
            for a, h in zip(arenas, h_arenas):
                a.copy_(h, non_blocking=True)
            if w.accumulate:
                o.copy_(h_out0, non_blocking=True)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["in"][b])
            pl.rs_fold(o, alpha=w.alpha, accumulate=w.accumulate, stream=s_comp)
            ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            h_outs[b].copy_(o, non_blocking=True)
            ev["out"][b].record(s_out)
        first[b] = False

    first = [True, True]
    for i in range(2):  # warm-up, one step on each buffer set
        step(i, first)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(K):
        step(i, first)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    end.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / K, world, dev)
    ok = torch.equal(h_outs[(K - 1) % 2], sets[(K - 1) % 2][2].cpu())
    plan2.close()
    del gs2, sets, h_outs, h_out0
    torch.cuda.empty_cache()
    return {"value": round(whole_job_gbs(rs_alg_bytes(w, w.total_numel()), world, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "steps": K,
            "readback_matches_device": ok,
            "mode": "pinned host gradients -> device by the copy engines, tide_rs_fold on the device copies, "
                    "fp32 shards -> pinned host; two device buffer sets, upload / fold / read-back streams"}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
