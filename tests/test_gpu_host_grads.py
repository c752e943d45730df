"""Gradients in page-locked host memory, folded in place over the host link.

A plan whose gradient pointers are page-locked host memory (mapped into the
device's address space) folds them with the direct-load kernel, reading every
rank's rows over the host link without a staging copy.  The result must be
Equation (5) in rank order bit for bit, as for device-resident gradients:
toy group, a ragged accumulating group, ranks in different 16-byte phases, and
the full-size Llama-3.1-8B block (every element).  Pageable host memory, the
bulk-copy kernel, other orders and a rebind between host and device memory
are refused with the documented status codes.
"""
import pytest
import torch

import all_gather_gb300 as tide
import oracle
import workloads
from all_gather_gb300 import _binding
from bits import assert_same_f32
from gpu_helpers import full_rs_check, oracle_rs_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from all_gather_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _pinned(views_uv, shift=False):
    """Page-locked host copies of grads[u][p]; shift: rank u's tensors start u % 8 elements
    into their buffer, so the ranks' rows differ in 16-byte phase."""
    out = []
    for u, vs in enumerate(views_uv):
        row = []
        for t in vs:
            off = u % 8 if shift else 0
            base = torch.empty(t.numel() + 8, dtype=t.dtype, pin_memory=True)
            h = base[off:off + t.numel()].view(t.shape)
            h.copy_(t)
            row.append(h)
        out.append(row)
    return out


def _descs(views_uv):
    W, P = len(views_uv), len(views_uv[0])
    return [([views_uv[u][p].data_ptr() for u in range(W)], views_uv[0][p].shape[0],
             views_uv[0][p].numel() // max(views_uv[0][p].shape[0], 1), -1) for p in range(P)]


@pytest.mark.parametrize("case", ["toy", "ragged_acc", "mixed_phase"])
def test_host_gradients_fold_matches_oracle(case):
    if case == "toy":
        w, acc, alpha, shift = workloads.get(1), False, 0.25, False
    elif case == "ragged_acc":
        w = workloads.custom(5, [(1003, 17), (3,), (64, 64), (2, 5), (4097,)], index=311)
        acc, alpha, shift = True, 0.5, False
    else:
        w = workloads.custom(6, [(301, 17), (64,), (40, 129)], index=312)
        acc, alpha, shift = False, 1.0, True
    dims = w.dim0_rownumel()
    _, _, S = oracle.geometry(w.world, dims)
    gs = workloads.make_grads(w, device="cuda")
    host = _pinned(gs.views, shift)
    init = torch.randn(w.world, S + 3, device="cuda") if acc else torch.zeros(w.world, S + 3, device="cuda")
    with tide.Plan(host) as plan:
        assert plan.fold_config()["block"] == 256  # the direct-load kernel
        out = init.clone()
        plan.rs_fold(out, alpha=alpha, accumulate=acc)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    want = oracle_rs_full(w.world, dims, gs.views, alpha, acc, init)
    assert_same_f32(out.cpu().numpy()[:, :S], want[:, :S], f"host gradients, {case}")
    assert torch.equal(out[:, S:], init[:, S:])
    with tide.Plan(gs.views) as dplan:  # the same bits as the device-resident fold
        ref = init.clone()
        dplan.rs_fold(ref, alpha=alpha, accumulate=acc)
        torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))


def test_host_gradients_full_size_every_element():
    w = workloads.get(2)  # Llama-3.1-8B block, W = 8, 3.5 GB of gradients in host memory
    dims = w.dim0_rownumel()
    gs = workloads.make_grads(w, device="cuda")
    host = _pinned(gs.views)
    del gs
    torch.cuda.empty_cache()
    _, _, S = oracle.geometry(w.world, dims)
    out = torch.full((w.world, S), float("nan"), device="cuda")
    with tide.Plan(host) as plan:
        plan.rs_fold(out, alpha=w.alpha)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    assert full_rs_check(w.world, dims, host, None, out, w.alpha, False, what="host gradients") == w.world * S


def test_host_gradients_refusals():
    w = workloads.custom(4, [(64, 8), (33,)], index=313)
    gs = workloads.make_grads(w, device="cuda")
    host = _pinned(gs.views)
    stream = torch.cuda.current_stream().cuda_stream
    # pageable host memory: a kernel cannot read it
    pageable = [[t.cpu() for t in vs] for vs in gs.views]
    with pytest.raises(tide.TideError) as e:
        _binding.tide_plan_build(w.world, _descs(pageable), None, stream)
    assert e.value.status == tide.TIDE_ERR_INVALID_ARG and "pageable" in e.value.detail
    # host memory takes the direct-load kernel: bulk copies, other orders and fp32 are refused
    for kw in (dict(kernel=tide.TIDE_KERNEL_BULK), dict(order=tide.TIDE_ORDER_TREE),
               dict(order=tide.TIDE_ORDER_STAGED_OWN)):
        with pytest.raises(tide.TideError) as e:
            _binding.tide_plan_build(w.world, _descs(host), tide.make_flags(**kw), stream)
        assert e.value.status == tide.TIDE_ERR_UNSUPPORTED, kw
    # a rebind may not move the gradients between host and device memory
    with tide.Plan(gs.views) as plan:
        with pytest.raises(tide.TideError) as e:
            plan.rebind(host)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        out = torch.zeros(w.world, plan.slot_numel, device="cuda")
        plan.rs_fold(out)  # the plan still holds its device gradients
        torch.cuda.synchronize()
        want = oracle_rs_full(w.world, w.dim0_rownumel(), gs.views, 1.0, False, torch.zeros_like(out))
        assert_same_f32(out.cpu().numpy(), want, "after a refused rebind")


@pytest.mark.parametrize("seed", range(20))
def test_host_gradients_random_groups(seed):
    """Seeded random ragged groups (1..40 ranks, zero-size parameters, random
    16-byte phases per rank, scale and accumulate) folded from page-locked
    host memory, bit-exact against the oracle."""
    import random
    rnd = random.Random(7000 + seed)
    world = rnd.choice([1, 2, 3, 5, 8, 16, 32, 40])
    shapes = []
    for _ in range(rnd.randint(1, 5)):
        d = rnd.choice([0, 1, world, world + 1, rnd.randint(1, 9 * world + 5)])
        shapes.append((d,) if rnd.random() < 0.2 else (d, rnd.choice([1, 3, 8, 64, 130])))
    w = workloads.custom(world, shapes, index=700 + seed)
    gs = workloads.make_grads(w, device="cuda")
    host = _pinned(gs.views, shift=rnd.random() < 0.5)
    dims = w.dim0_rownumel()
    _, _, S = oracle.geometry(world, dims)
    alpha = rnd.choice([1.0, 0.5, 1.0 / world])
    acc = rnd.random() < 0.4
    init = torch.randn(world, S + 2, device="cuda") if acc else torch.zeros(world, S + 2, device="cuda")
    out = init.clone()
    with tide.Plan(host) as plan:
        plan.rs_fold(out, alpha=alpha, accumulate=acc)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    want = oracle_rs_full(world, dims, gs.views, alpha, acc, init)
    assert_same_f32(out.cpu().numpy()[:, :S], want[:, :S], f"seed {seed}: W={world} {shapes}")
