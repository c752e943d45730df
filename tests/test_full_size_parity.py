"""Every output element of the full-size workloads against the oracle.

Section 4, Equation (5) in rank order is the contract on all five workloads:
the fold of each full-size group, launched exactly as the benchmark launches
it (default flags: the persistent bulk-copy kernel at full wave), is
compared bit for bit with the oracle over every element of every rank slot,
padding included.  The oracle runs unchanged on independent windows on all
host cores (gpu_helpers.full_rs_check), one parameter at a time.  The
Llama-3.1-70B block folds in accumulate mode (its benchmark setting), so the
accumulate epilogue is covered at full size too; the Llama-3.1-8B block is
also folded with alpha = 1/W.
"""
import pytest
import torch

import all_gather_gb300 as tide
import oracle
import workloads
from gpu_helpers import full_rs_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from all_gather_gb300 import build
    build.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("index,scale", [(2, "bench"), (2, "1/W"), (3, "bench"), (4, "bench"), (5, "bench")])
def test_full_size_every_element(index, scale):
    w = workloads.get(index)
    dims = w.dim0_rownumel()
    alpha = w.alpha if scale == "bench" else 1.0 / w.world
    gs = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, dims)
    with tide.Plan(gs.views) as plan:  # default flags: the benchmark's launch configuration
        assert plan.slot_numel == S
        if w.accumulate:
            out = workloads.make_out_init(w, S, device="cuda")
            before = out.clone()
        else:
            out = torch.full((w.world, S), float("nan"), device="cuda")  # every element must be written
            before = None
        plan.rs_fold(out, alpha=alpha, accumulate=w.accumulate)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    n = full_rs_check(w.world, dims, gs.views, before, out, alpha, w.accumulate,
                      what=f"{w.name} alpha={alpha} acc={w.accumulate}")
    assert n == w.world * S
    del gs, out, before
    torch.cuda.empty_cache()
