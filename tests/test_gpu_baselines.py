"""The stock-FSDP2-style baselines the benchmark times, checked against the oracle.

The fused fold's speed-up is quoted against these arms, so they must compute
the same collective:

* ``baselines.two_pass_rs`` packs each virtual rank's gradients with
  ``torch._chunk_cat`` into fp32 (Section 2.1, Equation (3)) and reduces the
  pack over ranks with ``sum(dim=0)``, then scales and accumulates
  (Equation (5)).  torch does not fix the summation order of that sum, so it
  is held to the reordered-variant tolerance: within 1e-6 of the rank-order
  oracle in the max-norm over each parameter tensor (tensors of 1,024 or more
  elements) and, for every element, within the textbook bound
  gamma_{W+1} (|alpha| sum_u |G^(u)| + |old|) of the exact sum.
* ``baselines.copy_out_ag`` (``split_with_sizes_copy`` of the rank-major
  all-gather output into padded per-parameter storage) is a bitwise copy:
  every real row must equal the oracle's placement (Equation (2)).

Cases: a ragged group with padding rows and empty ranks, the toy group, and
the full-size Llama-3.1-8B block.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from all_gather_gb300 import baselines
from bits import assert_same_u16, bf16_bits_to_f32
from gpu_helpers import bits16

pytestmark = pytest.mark.gpu

CASES = [("ragged", lambda: workloads.custom(5, [(1003, 17), (3,), (64, 64), (2, 5), (4097,)], index=301,
                                            alpha=0.2)),
         ("ragged_acc", lambda: workloads.custom(7, [(700, 33), (13, 1), (129, 128)], index=302, alpha=0.5,
                                                accumulate=True)),
         ("toy", lambda: workloads.get(1)),
         ("llama3.1_8b_block", lambda: workloads.get(2))]


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_two_pass_rs_matches_oracle_within_tolerance(name, make):
    w = make()
    W, dims = w.world, w.dim0_rownumel()
    R, o, S = oracle.geometry(W, dims)
    gs = workloads.make_grads(w, device="cuda")
    init = workloads.make_out_init(w, S, device="cuda") if w.accumulate else torch.zeros(W, S, device="cuda")
    pack = torch.empty(W, W * S, dtype=torch.float32, device="cuda")
    out = init.clone()
    baselines.two_pass_rs(gs.views, pack, out, w.alpha, w.accumulate)
    torch.cuda.synchronize()
    del pack
    got = out.cpu().numpy()
    old = init.cpu().numpy()
    want = old.copy()
    host = [[bits16(gs.views[u][p]) for u in range(W)] for p in range(len(dims))]
    oracle.rs(W, dims, host, w.alpha, w.accumulate, want)
    gamma = (W + 1) * 2.0 ** -24 / (1 - (W + 1) * 2.0 ** -24)
    for p, (d, k) in enumerate(dims):
        n = R[p] * k
        a = got[:, o[p]:o[p] + n].reshape(-1)
        b = want[:, o[p]:o[p] + n].reshape(-1)
        if d * k >= 1024:
            assert np.abs(a - b).max() <= 1e-6 * np.abs(b).max(), f"{name} p={p}: beyond the 1e-6 max-norm tolerance"
        # every element, padding included: the bound around the exact fp64 sum
        vals = np.zeros((W, W * n))  # [u][r * n + j]: rank u's contribution to rank r's element j
        for u in range(W):
            g = bf16_bits_to_f32(host[p][u]).astype(np.float64)
            vals[u, :d * k] = g
        exact = w.alpha * vals.sum(0).reshape(W, n)
        mag = abs(w.alpha) * np.abs(vals).sum(0).reshape(W, n)
        base = old[:, o[p]:o[p] + n].astype(np.float64)
        if w.accumulate:
            exact, mag = exact + base, mag + np.abs(base)
        err = np.abs(got[:, o[p]:o[p] + n].astype(np.float64) - exact)
        assert (err <= gamma * mag + 1e-45).all(), f"{name} p={p}: beyond gamma_(W+1) of the exact sum"
    del gs, out, init
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_copy_out_ag_is_bitwise(name, make):
    w = make()
    W, dims = w.world, w.dim0_rownumel()
    R, o, S = oracle.geometry(W, dims)
    slots = workloads.make_slots(w, S, device="cuda")
    sizes = [R[p] * k for p, (_, k) in enumerate(dims)]
    padded = [torch.full((W * n,), float("nan"), dtype=torch.bfloat16, device="cuda") for n in sizes]
    baselines.copy_out_ag(slots[:, :S], padded, sizes)
    torch.cuda.synchronize()
    want = oracle.ag(W, dims, bits16(slots).reshape(W, -1))
    for p, (d, k) in enumerate(dims):
        # the padded storage holds rank r's R_p rows at r R_p; the real rows are the parameter
        assert_same_u16(bits16(padded[p])[:d * k], want[p], f"{name} copy-out p={p}")
    del slots, padded
    torch.cuda.empty_cache()
