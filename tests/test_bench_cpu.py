"""Host legs of bench.py that need no GPU: the all-cores run of the oracle
(independent windows in a thread pool) reassembles the single-threaded
oracle's reduce-scatter bit for bit, with and without accumulation and on
ragged shapes whose pieces end in padding."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402


@pytest.mark.parametrize("accumulate", [False, True])
def test_cpu_oracle_all_cores_matches_single_thread(accumulate):
    import bench
    shapes = [(5497, 1000), (333, 17), (7, 5), (3000,)]  # the first: pieces of more than one 2^20 window
    w = workloads.custom(5, shapes, index=41, alpha=0.5, accumulate=accumulate)
    host = [[workloads.normal_fp32(w.numels()[p], workloads.grad_seed(w, u, p), w.sigma)
             .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for u in range(w.world)]
            for p in range(len(shapes))]
    rec = bench.cpu_oracle_all_cores(w, host, [0, 1, 2, 3], min_seconds=0.0, max_reps=1)
    assert rec["matches_single_thread"] and rec["cores"] >= 1 and rec["value"] > 0
    assert "windows" in rec["sample"]
    one = bench.cpu_oracle_sample(w, host, [0, 1, 2, 3], min_seconds=0.0, max_reps=1)
    assert one["cores"] == 1 and one["value"] > 0 and one["kind"] == "oracle"


def test_cpu_sample_takes_each_distinct_shape_once():
    import bench
    moe = workloads.get("qwen3_30b_a3b_moe_layer")
    idx = bench.sample_params(moe)
    assert [moe.names[i] for i in idx] == ["experts.0.gate_proj", "experts.0.down_proj", "router", "q_proj",
                                           "k_proj", "o_proj"]
    assert len({moe.shapes[i] for i in idx}) == len(idx) == len(set(moe.shapes))
    toy = workloads.get(1)
    assert bench.sample_params(toy) == list(range(toy.num_params))
    assert "6 distinct shapes" in bench.sample_text(moe, idx)
    # the metric's bytes: W*N*2 read + N*4 written (+ N*4 read when accumulating)
    l70 = workloads.get("llama3.1_70b_block")
    assert bench.rs_alg_bytes(l70, 10) == 8 * 10 * 2 + 10 * 4 + 10 * 4


def test_cpu_ranges_and_model():
    import bench
    assert bench.cpu_ranges({0, 1, 2, 3, 5, 7, 8, 9}) == "0-3,5,7-9"
    assert bench.cpu_ranges({4}) == "4"
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_profile_readers_follow_the_kernel_source():
    """The committed traffic and SM-time summaries are reported while their
    recorded digest matches the fold source (comments excluded), and not at
    all once the source has changed."""
    import bench
    digest = bench.kernel_digest()
    traffic = bench.profile_traffic("qwen3_30b_a3b_moe_layer")
    sm_time = bench.profile_sm_time("qwen3_30b_a3b_moe_layer")  # falls back to the reduced case
    for name, value in (("rs_fold_qwen3_30b_a3b_moe_layer_traffic.txt", traffic),
                        ("sm_time_llama3.1_8b_attn.txt", sm_time)):
        recorded = (bench._profile_kv(name) or {}).get("rs_fold_cu_sha256_16")
        assert (value is not None) == (recorded == digest), name
    if traffic is not None:
        assert 40.0e9 < traffic < 45.0e9  # algorithmic bytes per launch: 42.37 GB
    if sm_time is not None:
        assert sm_time["workload"] == "llama3.1_8b_attn" and sm_time["ratio"] > 5


REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference (the CPU oracle's reduce-scatter on a sample
    of the workload) prints one JSON line with the contract's keys."""
    import json
    import subprocess
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "toy",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in REQUIRED:
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "toy" and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_host_memory_probe():
    """The e2e leg sizes its pinned buffers against MemAvailable before pinning them."""
    import bench
    avail = bench.host_mem_available()
    assert avail > 0 and avail % 1024 == 0


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched as the multi-GPU bench is (torchrun, 2 ranks, 127.0.0.1), the
    reference arm runs on rank 0 only and prints exactly one JSON line; the
    other rank exits 0 without work."""
    import json
    import socket
    import subprocess
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "toy", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
