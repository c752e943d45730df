"""Concurrent-compute interference of the reduce-scatter (measurement harness).

Follows the method of the TIDE paper's Table 4 / Section 2.2: a victim kernel
runs back to back on one stream while the reduce-scatter runs on another;
the slowdown is the median duration of the victims that ran entirely inside
the reduce-scatter window over the median duration of the victim alone,
minus one.  Victims: a bf16 GEMM of 256 x 8192 x 8192 (the page's one-wave
GEMM), a large 8192^3 bf16 GEMM, and a 256 MiB bf16 elementwise kernel.
Arms: the fused fold at several CTA budgets and with one short-lived CTA per
work item, the two-pass stock-FSDP2 baseline, and the all-gather placement on
SMs and on the copy engines (issued per call, or replayed from a CUDA graph).
Each pair runs twice: on streams of equal priority (the page's method) and
with the victim's stream at the higher priority.  Set CUDA_DEVICE_MAX_CONNECTIONS=32
before CUDA starts (the page's setting) so the two streams get separate
hardware queues.

    python -m all_gather_gb300.interference [--workload NAME] [--budgets 0,16,64]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
from typing import Callable, Dict

os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")


def _victims(dev) -> Dict[str, Callable[[], None]]:
    import torch
    g = torch.Generator(device=dev).manual_seed(1234)
    a1 = torch.randn(256, 8192, device=dev, generator=g).to(torch.bfloat16)
    b1 = torch.randn(8192, 8192, device=dev, generator=g).to(torch.bfloat16)
    c1 = torch.empty(256, 8192, device=dev, dtype=torch.bfloat16)
    a2 = torch.randn(8192, 8192, device=dev, generator=g).to(torch.bfloat16)
    c2 = torch.empty(8192, 8192, device=dev, dtype=torch.bfloat16)
    x = torch.randn(128 * 1024 * 1024, device=dev, generator=g).to(torch.bfloat16)  # 256 MiB
    y = torch.empty_like(x)
    return {
        "gemm_256x8192x8192": lambda: torch.matmul(a1, b1, out=c1),
        "gemm_8192x8192x8192": lambda: torch.matmul(a2, b1, out=c2),
        "elementwise_256MiB": lambda: torch.mul(x, 1.0009765625, out=y),
    }


def _time_alone(fn, n: int, stream) -> float:
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
        for s, e in ev:
            s.record(stream)
            fn()
            e.record(stream)
    torch.cuda.synchronize()
    return statistics.median(s.elapsed_time(e) for s, e in ev)


def _co_run(rs_call: Callable[[], None], n_rs: int, victim, victim_ms: float, rs_ms_est: float,
            victim_high: bool = False) -> dict:
    """victim_high: the victim runs on a higher-priority stream than the
    reduce-scatter (compute first, communication in the background), so the
    block scheduler gives free SMs to the victim's CTAs first.  A persistent
    grid holds its SMs either way; short-lived CTAs yield them as they retire."""
    import torch
    s_rs, s_v = torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-1 if victim_high else 0)
    n_v = int((rs_ms_est * n_rs) / max(victim_ms, 1e-3) * 1.5) + 20
    n_v = min(n_v, 4000)
    start = torch.cuda.Event(enable_timing=True)
    rs0, rs1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_v)]
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    start.record(cur)
    s_rs.wait_event(start)
    s_v.wait_event(start)
    with torch.cuda.stream(s_v):
        for s, e in ev:
            s.record(s_v)
            victim()
            e.record(s_v)
    with torch.cuda.stream(s_rs):
        rs0.record(s_rs)
        for _ in range(n_rs):
            rs_call()
        rs1.record(s_rs)
    torch.cuda.synchronize()
    w0, w1 = start.elapsed_time(rs0), start.elapsed_time(rs1)
    inside = [s.elapsed_time(e) for s, e in ev if start.elapsed_time(s) >= w0 and start.elapsed_time(e) <= w1]
    return {"rs_window_ms": round(w1 - w0, 4), "rs_ms": round((w1 - w0) / n_rs, 4), "victims_inside": len(inside),
            "victim_ms": round(statistics.median(inside), 5) if inside else None}


def measure(workload: str = "llama3.1_8b_block", budgets=(0, 64, 16), n_rs: int = 20, device: int = 0,
            grads=None, with_placement: bool = True) -> dict:
    import torch

    import all_gather_gb300 as tide
    import workloads
    from all_gather_gb300 import baselines

    torch.cuda.set_device(device)
    dev = torch.device("cuda", device)
    w = workloads.get(workload)
    gs = grads if grads is not None else workloads.make_grads(w, device=dev)
    victims = _victims(dev)
    plans = {}
    for b in budgets:
        plans[f"fused_cta{b}" if b else "fused_full_wave"] = tide.Plan(gs.views, tide.make_flags(cta_budget=b))
    plans["fused_per_item"] = tide.Plan(gs.views, tide.make_flags(sched=tide.TIDE_SCHED_PER_ITEM))
    S = next(iter(plans.values())).slot_numel
    out = torch.zeros(w.world, S, device=dev)
    pack = torch.empty(w.world, w.world * S, device=dev)
    arms = {name: (lambda p=p: p.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)) for name, p in plans.items()}
    arms["two_pass_baseline"] = lambda: baselines.two_pass_rs(gs.views, pack, out, w.alpha, w.accumulate)
    if with_placement:
        # the all-gather side: placement on SMs vs on the copy engines (no SMs)
        slots = workloads.make_slots(w, S, device=dev)
        full = [torch.empty(s_, dtype=torch.bfloat16, device=dev) for s_ in w.shapes]
        pl = next(iter(plans.values()))
        full_b = pl.bind_full(full)
        arms["placement_sm_kernel"] = lambda: pl.ag_place(slots, full_b, mode="sm")
        arms["placement_copy_engines"] = lambda: pl.ag_place(slots, full_b, mode="ce2d")
        # the same copies replayed from a CUDA graph (no host issue per call)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            pl.ag_place(slots, full_b, mode="ce2d")
        torch.cuda.synchronize()
        ce_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ce_graph, stream=side):
            pl.ag_place(slots, full_b, mode="ce2d")
        arms["placement_copy_engines_graph"] = ce_graph.replay

    quiet = torch.cuda.Stream()
    rs_alone = {name: _time_alone(fn, 10, quiet) for name, fn in arms.items()}
    res = {"workload": w.name, "cuda_device_max_connections": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS"),
           "rs_alone_ms": {k: round(v, 4) for k, v in rs_alone.items()}, "victims": {}}
    for vname, vfn in victims.items():
        alone = _time_alone(vfn, 50, quiet)
        entry = {"alone_ms": round(alone, 5), "arms": {}, "arms_victim_high": {}}
        for name, fn in arms.items():
            for key, high in (("arms", False), ("arms_victim_high", True)):
                r = _co_run(fn, n_rs, vfn, alone, rs_alone[name], victim_high=high)
                r["slowdown"] = round(r["victim_ms"] / alone - 1.0, 4) if r["victim_ms"] else None
                entry[key][name] = r
        res["victims"][vname] = entry
    arms.clear()  # the captured graph goes before the plans it reads
    for p in plans.values():
        p.close()
    del pack, out
    torch.cuda.empty_cache()
    return res


PROBE_SMEM = 213 * 1024   # the one-wave GEMM's per-CTA footprint on the page: one CTA fills an SM
PROBE_CLUSTERS = 32       # 256x8192x8192 GEMM: 128 CTAs in 32 four-CTA clusters


BLOCKED_NS = 5000  # a probe CTA entering later than this after its stream reached it was blocked


def _probe_once(tide, ctas, cluster, hold_ns, bufs, stream):
    smid, tin, tout, ready = bufs
    tide.tide_sm_probe(ctas, cluster, PROBE_SMEM, hold_ns, smid.data_ptr(), tin.data_ptr(), tout.data_ptr(),
                       ready.data_ptr(), stream.cuda_stream)


def _displaced(tin, tout, n):
    """Probe CTAs that entered after the first probe CTA left (second wave)."""
    a, b = tin[:n].cpu(), tout[:n].cpu()
    return int((a > b.min()).sum())


def _blocked(tin, ready, n):
    """Probe CTAs that entered more than BLOCKED_NS after the probe was reached."""
    return int(((tin[:n].cpu() - ready[0].cpu()) > BLOCKED_NS).sum())


def sm_probe(workload: str = "llama3.1_8b_block", budgets=(0, 152, 64, 16), windows: int = 30, device: int = 0,
             grads=None, hold_us: float = 30.0) -> dict:
    """Table 5 / Figure 3 measurement on this GPU: (1) the cluster slots of the
    one-wave GEMM's shape; (2) per reduce-scatter arm, over `windows` probe
    launches at random points of the reduce-scatter, the displaced probe CTAs
    (mode) and the share of windows with any; (3) with one SM-filling probe
    CTA per SM, the mean number of SMs the reduce-scatter held."""
    import random

    import torch

    import all_gather_gb300 as tide
    import workloads
    from all_gather_gb300 import baselines

    torch.cuda.set_device(device)
    dev = torch.device("cuda", device)
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    slots = tide.tide_sm_probe_max_clusters(4, PROBE_SMEM)
    res = {"sms": n_sm, "cluster_slots_4cta_213KB": slots, "probe": f"{PROBE_CLUSTERS} x 4-CTA clusters, "
           f"{PROBE_SMEM // 1024} KB smem per CTA, hold {hold_us} us; resident probe: {n_sm} single CTAs", "arms": {}}
    if slots < 1:
        res["skipped"] = "the device cannot hold one probe cluster"
        return res
    w = workloads.get(workload)
    gs = grads if grads is not None else workloads.make_grads(w, device=dev)
    nmax = max(PROBE_CLUSTERS * 4, n_sm)
    bufs = (torch.zeros(nmax, dtype=torch.int32, device=dev), torch.zeros(nmax, dtype=torch.int64, device=dev),
            torch.zeros(nmax, dtype=torch.int64, device=dev), torch.zeros(1, dtype=torch.int64, device=dev))
    s_rs, s_pr = torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-1)  # the probe stands for compute
    hold = int(hold_us * 1000)
    # the probe alone: no displacement expected when it fits in one wave (the
    # first launch also loads the kernel, so it is a warm-up)
    _probe_once(tide, PROBE_CLUSTERS * 4, 4, hold, bufs, s_pr)
    torch.cuda.synchronize()
    _probe_once(tide, PROBE_CLUSTERS * 4, 4, hold, bufs, s_pr)
    torch.cuda.synchronize()
    res["alone_displaced"] = _displaced(bufs[1], bufs[2], PROBE_CLUSTERS * 4)
    res["alone_blocked"] = _blocked(bufs[1], bufs[3], PROBE_CLUSTERS * 4)
    plans = {(f"fused_cta{b}" if b else "fused_full_wave"): tide.Plan(gs.views, tide.make_flags(cta_budget=b))
             for b in budgets}
    plans["fused_per_item"] = tide.Plan(gs.views, tide.make_flags(sched=tide.TIDE_SCHED_PER_ITEM))
    S = next(iter(plans.values())).slot_numel
    out = torch.zeros(w.world, S, device=dev)
    pack = torch.empty(w.world, w.world * S, device=dev)
    arms = {name: (lambda p=p: p.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)) for name, p in plans.items()}
    arms["two_pass_baseline"] = lambda: baselines.two_pass_rs(gs.views, pack, out, w.alpha, w.accumulate)
    rnd = random.Random(5)
    clock_hz = 1.9e9  # nominal SM clock: only sets the random start delay of a probe window
    for name, fn in arms.items():
        # reduce-scatter duration alone, to place the probes inside it
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        rs_ms = e0.elapsed_time(e1)
        disp, blocked, resident = [], [], []
        for kind, ctas, cluster in (("gemm", PROBE_CLUSTERS * 4, 4), ("resident", n_sm, 1)):
            for _ in range(windows):
                torch.cuda.synchronize()
                with torch.cuda.stream(s_rs):
                    fn()
                delay = int(rnd.random() * 0.8 * rs_ms * 1e-3 * clock_hz)
                with torch.cuda.stream(s_pr):
                    if delay > 0:
                        torch.cuda._sleep(delay)
                    _probe_once(tide, ctas, cluster, hold, bufs, s_pr)
                torch.cuda.synchronize()
                if kind == "gemm":
                    disp.append(_displaced(bufs[1], bufs[2], ctas))
                    blocked.append(_blocked(bufs[1], bufs[3], ctas))
                else:
                    resident.append(_blocked(bufs[1], bufs[3], ctas))
        mode = max(set(disp), key=disp.count)
        res["arms"][name] = {"rs_ms": round(rs_ms, 4), "displaced_mode": mode,
                             "windows_hit_pct": round(100.0 * sum(b > 0 for b in blocked) / len(blocked), 1),
                             "blocked_gemm_ctas_mean": round(sum(blocked) / len(blocked), 1),
                             "resident_sms_mean": round(sum(resident) / len(resident), 2)}
    for p in plans.values():
        p.close()
    del pack, out
    torch.cuda.empty_cache()
    return res


GEMM_CTAS, GEMM_CLUSTER = 128, 4  # the one-wave GEMM's launch: 32 four-CTA clusters of 213 KB CTAs


def corun_budget() -> dict:
    """The fold's CTA budget next to the one-wave GEMM on this device:
    Equation (4)'s spare cluster slots (tide_corun_cta_budget) from the slots
    the probe shape gets here (tide_sm_probe_max_clusters)."""
    import all_gather_gb300 as tide
    slots = tide.tide_sm_probe_max_clusters(GEMM_CLUSTER, PROBE_SMEM)
    budget = tide.tide_corun_cta_budget(slots, GEMM_CTAS, GEMM_CLUSTER) if slots > 0 else -1
    return {"cluster_slots": slots, "gemm_clusters": -(-GEMM_CTAS // GEMM_CLUSTER), "cta_budget": budget}


def corun_target(workload: str, device: int = 0, grads=None, n_rs: int = 10, reps: int = 3) -> dict:
    """One stated configuration against the two-pass baseline: the fused fold
    at the co-run CTA budget (corun_budget) must finish at least 1.5x sooner
    than the two-pass reduce-scatter and slow the one-wave GEMM less than the
    two-pass reduce-scatter does, on streams of equal priority (Table 4's
    method).  Each co-run is repeated `reps` times; the medians are reported."""
    import torch

    import all_gather_gb300 as tide
    import workloads
    from all_gather_gb300 import baselines

    torch.cuda.set_device(device)
    dev = torch.device("cuda", device)
    w = workloads.get(workload)
    gs = grads if grads is not None else workloads.make_grads(w, device=dev)
    cb = corun_budget()
    res = {"workload": w.name, "victim": "gemm_256x8192x8192 (bf16, one wave)", "priority": "equal", **cb}
    if cb["cta_budget"] < 1:
        res["met"] = False
        res["why"] = "no spare cluster slot on this device: every resident fold CTA can displace GEMM CTAs"
        return res
    plans = {"fused_corun_budget": tide.Plan(gs.views, tide.make_flags(cta_budget=cb["cta_budget"])),
             "fused_full_wave": tide.Plan(gs.views)}
    S = plans["fused_full_wave"].slot_numel
    out = torch.zeros(w.world, S, device=dev)
    pack = torch.empty(w.world, w.world * S, device=dev)
    arms = {name: (lambda p=p: p.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)) for name, p in plans.items()}
    arms["two_pass_baseline"] = lambda: baselines.two_pass_rs(gs.views, pack, out, w.alpha, w.accumulate)
    victim = _victims(dev)["gemm_256x8192x8192"]
    quiet = torch.cuda.Stream()
    gemm_alone = _time_alone(victim, 50, quiet)
    rs_alone = {name: _time_alone(fn, 3, quiet) for name, fn in arms.items()}
    slow, rs_co = {}, {}
    for name, fn in arms.items():
        runs = [_co_run(fn, n_rs, victim, gemm_alone, rs_alone[name]) for _ in range(reps)]
        sd = [r["victim_ms"] / gemm_alone - 1.0 for r in runs if r["victim_ms"]]
        slow[name] = round(statistics.median(sd), 4) if sd else None
        rs_co[name] = round(statistics.median(r["rs_ms"] for r in runs), 4)
    for p in plans.values():
        p.close()
    del pack, out
    torch.cuda.empty_cache()
    speedup = rs_alone["two_pass_baseline"] / rs_alone["fused_corun_budget"]
    lower = (slow["fused_corun_budget"] is not None and slow["two_pass_baseline"] is not None
             and slow["fused_corun_budget"] < slow["two_pass_baseline"])
    res.update({"gemm_alone_ms": round(gemm_alone, 5), "rs_alone_ms": {k: round(v, 4) for k, v in rs_alone.items()},
                "rs_ms_while_corunning": rs_co, "gemm_slowdown": slow,
                "speedup_vs_two_pass": round(speedup, 3), "speedup_at_least_1_5x": bool(speedup >= 1.5),
                "slowdown_below_two_pass": bool(lower), "met": bool(speedup >= 1.5 and lower),
                "method": f"median of {reps} co-runs of {n_rs} reduce-scatters each; slowdown = median GEMM time "
                          "fully inside the reduce-scatter window / GEMM alone - 1"})
    return res


def summarize(res: dict) -> dict:
    """victim -> {arm: slowdown} (equal stream priorities, and the victim on a
    higher-priority stream) plus the RS times per arm."""
    def table(key, field):
        return {v: {a: r[field] for a, r in e[key].items()} for v, e in res["victims"].items()}
    return {"slowdown": table("arms", "slowdown"),
            "slowdown_victim_high_priority": table("arms_victim_high", "slowdown"),
            "victim_alone_ms": {v: e["alone_ms"] for v, e in res["victims"].items()},
            "rs_alone_ms": res["rs_alone_ms"],
            "rs_ms_while_corunning": table("arms", "rs_ms"),
            "rs_ms_while_corunning_victim_high_priority": table("arms_victim_high", "rs_ms"),
            "method": "median victim duration fully inside the RS window / median alone - 1; "
                      "CUDA_DEVICE_MAX_CONNECTIONS=" + str(res["cuda_device_max_connections"])}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3.1_8b_block")
    ap.add_argument("--budgets", default="0,64,16")
    ap.add_argument("--n-rs", type=int, default=20)
    ap.add_argument("--probe", action="store_true", help="run the SM-id probe (Table 5) instead")
    ap.add_argument("--windows", type=int, default=30)
    a = ap.parse_args(argv)
    budgets = tuple(int(x) for x in a.budgets.split(","))
    res = sm_probe(a.workload, budgets, a.windows) if a.probe else measure(a.workload, budgets, a.n_rs)
    print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    sys.exit(main())
