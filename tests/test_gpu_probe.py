"""The SM-id probe (Table 5 / Figure 3's measurement) and the interference
harness (Table 4's method), on small cases.

Probe records: one per launched CTA, SM ids below the SM count, entry before
exit and at least the hold apart, at most one SM-filling CTA per SM at a
time, and a device that holds at least one cluster of the one-wave GEMM's
shape (which alone then runs in one wave).  Harness: a co-run of a fold with
the one-wave GEMM counts victims inside the fold's window and gives finite
times, and the co-run target's record is consistent with its inputs.
"""
import math

import pytest
import torch

import all_gather_gb300 as tide
import workloads
from all_gather_gb300 import interference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from all_gather_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _bufs(n):
    return (torch.full((n,), -1, dtype=torch.int32, device="cuda"), torch.zeros(n, dtype=torch.int64, device="cuda"),
            torch.zeros(n, dtype=torch.int64, device="cuda"), torch.zeros(1, dtype=torch.int64, device="cuda"))


@pytest.mark.parametrize("ctas,cluster", [(1, 1), (7, 1), (152, 1), (128, 4), (200, 1)])
def test_probe_records(ctas, cluster):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    smid, tin, tout, ready = _bufs(ctas)
    hold = 20_000
    s = torch.cuda.current_stream()
    tide.tide_sm_probe(ctas, cluster, interference.PROBE_SMEM, hold, smid.data_ptr(), tin.data_ptr(),
                       tout.data_ptr(), ready.data_ptr(), s.cuda_stream)
    torch.cuda.synchronize()
    sm, a, b, t0 = smid.cpu(), tin.cpu(), tout.cpu(), int(ready.cpu()[0])
    assert (sm >= 0).all() and (sm < n_sm).all(), "an SM id outside the device (or a CTA that left no record)"
    assert (a > 0).all() and (b >= a + hold).all(), "exit before entry + hold"
    assert (a >= t0).all(), "a probe CTA entered before its stream reached the probe"
    # an SM-filling CTA has its SM alone: CTAs on the same SM never overlap in time
    for m in set(sm.tolist()):
        idx = (sm == m).nonzero().flatten().tolist()
        spans = sorted((int(a[i]), int(b[i])) for i in idx)
        assert all(spans[i + 1][0] >= spans[i][1] for i in range(len(spans) - 1)), f"two probe CTAs shared SM {m}"
    assert len(set(sm.tolist())) <= min(ctas, n_sm)


def test_cluster_slots_and_corun_budget():
    slots = tide.tide_sm_probe_max_clusters(4, interference.PROBE_SMEM)
    assert slots >= 1
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert slots * 4 <= n_sm
    cb = interference.corun_budget()
    assert cb["cluster_slots"] == slots
    assert cb["cta_budget"] == max(0, slots - 32) * 4 == tide.tide_corun_cta_budget(slots, 128, 4)
    if slots >= 32:  # the GEMM's 32 clusters fit: the probe alone runs in one wave
        smid, tin, tout, ready = _bufs(128)
        for _ in range(2):  # the first launch also loads the kernel
            tide.tide_sm_probe(128, 4, interference.PROBE_SMEM, 30_000, smid.data_ptr(), tin.data_ptr(),
                               tout.data_ptr(), ready.data_ptr(), torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
        assert interference._displaced(tin, tout, 128) == 0


def test_co_run_counts_victims_inside_the_window():
    w = workloads.get("llama3.1_8b_attn")
    gs = workloads.make_grads(w, device="cuda")
    plan = tide.Plan(gs.views, tide.make_flags(cta_budget=16))
    out = torch.zeros(w.world, plan.slot_numel, device="cuda")
    fold = lambda: plan.rs_fold(out, alpha=1.0)  # noqa: E731
    victim = interference._victims(torch.device("cuda", 0))["gemm_256x8192x8192"]
    quiet = torch.cuda.Stream()
    alone = interference._time_alone(victim, 20, quiet)
    rs_ms = interference._time_alone(fold, 3, quiet)
    assert 0 < alone < 10 and 0 < rs_ms < 1000
    r = interference._co_run(fold, 10, victim, alone, rs_ms)
    assert r["victims_inside"] > 0
    assert math.isfinite(r["victim_ms"]) and r["victim_ms"] > 0
    assert r["rs_window_ms"] >= 10 * r["rs_ms"] * 0.999 and r["rs_ms"] > 0
    plan.close()


def test_corun_target_record():
    w = workloads.get("llama3.1_8b_attn")
    res = interference.corun_target(w.name, n_rs=5, reps=1)
    cb = interference.corun_budget()
    assert res["cta_budget"] == cb["cta_budget"]
    if cb["cta_budget"] < 1:
        assert res["met"] is False
        return
    for arm in ("fused_corun_budget", "fused_full_wave", "two_pass_baseline"):
        assert res["rs_alone_ms"][arm] > 0
        assert res["gemm_slowdown"][arm] is None or math.isfinite(res["gemm_slowdown"][arm])
    sp = res["rs_alone_ms"]["two_pass_baseline"] / res["rs_alone_ms"]["fused_corun_budget"]
    assert abs(res["speedup_vs_two_pass"] - sp) <= 1e-3 * sp + 1e-3
    assert res["met"] == (res["speedup_at_least_1_5x"] and res["slowdown_below_two_pass"])
