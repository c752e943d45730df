"""The allocation-free fold (tide_rs_fold_noalloc) against the oracle and the
plan-based fold.

Some callers cannot allocate GPU memory (code running inside an allocator or
an out-of-memory handler, under a pool or cap that forbids new device
allocations), so they cannot build a plan, whose device tables come from
cudaMalloc.  tide_rs_fold_noalloc serves them from a fixed device array owned
by the library.  These tests call it through the C ABI and check:

* two calls in a row, with different groups, each equal to the oracle
  (Equation (5) in rank order) and to the plan-based tide_rs_fold bit for bit
  (the tolerance of every fold parity test: none);
* a group whose ranks' rows differ in 16-byte phase (the fold's scalar path)
  and a 32-rank group (several shared-memory stage fills per chunk);
* the full-size Llama-3.1-70B block and MoE layer, element for element equal
  to the plan-based fold, and 60 seeded random ragged groups against the oracle;
* that after a warm-up call, further calls leave the device's free memory and
  torch's allocation count unchanged, and that the entry point's device
  status word reads TIDE_OK through tide_last_device_status(NULL, stream);
* that an oversized request is refused before any GPU work.

The file sorts last so that a run stopping at the first failure has run
everything else; every test here also passes in a fresh process.
"""
import pytest
import torch

import all_gather_gb300 as tide
import workloads
from bits import assert_same_f32
from gpu_helpers import oracle_rs_full

pytestmark = pytest.mark.gpu


def _descs(grads_uv):
    W, P = len(grads_uv), len(grads_uv[0])
    out = []
    for p in range(P):
        t = grads_uv[0][p]
        d0 = t.shape[0]
        out.append(([grads_uv[u][p].data_ptr() for u in range(W)], d0, t.numel() // d0 if d0 else 0, -1))
    return out


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _noalloc(world, views, out, stride, alpha, accumulate):
    tide.tide_rs_fold_noalloc(world, _descs(views), out.data_ptr(), stride, alpha, int(accumulate), _stream())


def _check(world, views, alpha, accumulate, stride_extra=0, what=""):
    """Allocation-free result vs the plan-based fold and vs the oracle."""
    dims = [(t.shape[0], t.numel() // t.shape[0] if t.shape[0] else 0) for t in views[0]]
    with tide.Plan(views) as plan:
        S = plan.slot_numel
        stride = S + stride_extra
        init = torch.randn(world, stride, device="cuda") if accumulate else None
        ref = init.clone() if accumulate else torch.full((world, stride), 7.0, device="cuda")
        plan.rs_fold(ref, alpha=alpha, accumulate=accumulate)
    got = init.clone() if accumulate else torch.full((world, stride), 7.0, device="cuda")
    if not accumulate:
        got[:, :S] = -1.0  # every element up to S must be overwritten
    _noalloc(world, views, got, stride, alpha, accumulate)
    torch.cuda.synchronize()
    assert tide.tide_last_device_status(0, _stream()) == tide.TIDE_OK
    assert_same_f32(got.cpu().numpy(), ref.cpu().numpy(), f"{what}: allocation-free vs plan-based fold")
    before = init if accumulate else torch.zeros(world, stride, device="cuda")
    want = oracle_rs_full(world, dims, views, alpha, accumulate, before)
    assert_same_f32(got[:, :S].cpu().numpy(), want[:, :S], f"{what}: allocation-free fold vs the oracle")
    if not accumulate:
        assert (got[:, S:] == 7.0).all(), f"{what}: wrote past S"


def test_noalloc_matches_oracle_and_plan_fold_two_calls_in_a_row():
    torch.cuda.set_device(0)
    # call 1: the toy group (W = 4, ragged shapes, padding, scale 1/W; pieces
    # whose ranks share a non-zero 16-byte phase)
    w1 = workloads.get(1)
    g1 = workloads.make_grads(w1, device="cuda")
    _check(w1.world, g1.views, w1.alpha, False, stride_extra=3, what="call 1 (toy group)")
    # call 2, straight after: a different group (W = 8) in accumulate mode
    w2 = workloads.custom(8, [(1000, 33), (17,), (4096, 64), (5, 3)], index=123)
    g2 = workloads.make_grads(w2, device="cuda")
    _check(w2.world, g2.views, 0.5, True, what="call 2 (W = 8, accumulate)")


def test_noalloc_ranks_in_different_phases_and_32_ranks():
    torch.cuda.set_device(0)
    # every rank's tensors start at a different 2-byte offset: the ranks' rows
    # differ in 16-byte phase, so the fold reads them element by element
    w = workloads.custom(5, [(301, 17), (64,), (40, 129)], index=124)
    g = workloads.make_grads(w, device="cuda")
    views = []
    for u in range(w.world):
        vs = []
        for t in g.views[u]:
            base = torch.empty(t.numel() + 8, dtype=torch.bfloat16, device="cuda")
            v = base[u % 8:u % 8 + t.numel()].view(t.shape)
            v.copy_(t)
            vs.append(v)
        views.append(vs)
    _check(w.world, views, 1.0, False, what="mixed phases")
    # 32 ranks: four stage fills of eight ranks per chunk, summed in order
    w32 = workloads.custom(32, [(1000, 33), (4096,), (64, 128), (33, 7)], index=125)
    g32 = workloads.make_grads(w32, device="cuda")
    _check(w32.world, g32.views, 1.0 / 32, False, stride_extra=5, what="W = 32")
    _check(w32.world, g32.views, 1.0, True, what="W = 32, accumulate")


@pytest.mark.parametrize("index", [3, 5])
def test_noalloc_full_size_matches_plan_fold(index):
    """The full-size Llama-3.1-70B block (accumulate) and MoE layer (389
    parameters x 32 ranks: ~1.9 MB of tables, the largest benchmark request):
    every output element equal to the plan-based fold's, which the full-size
    parity tests compare with the oracle."""
    torch.cuda.set_device(0)
    w = workloads.get(index)
    g = workloads.make_grads(w, device="cuda")
    with tide.Plan(g.views) as plan:
        S = plan.slot_numel
        init = workloads.make_out_init(w, S, device="cuda") if w.accumulate else None
        ref = init.clone() if w.accumulate else torch.full((w.world, S), float("nan"), device="cuda")
        plan.rs_fold(ref, alpha=w.alpha, accumulate=w.accumulate)
    got = init.clone() if w.accumulate else torch.full((w.world, S), float("nan"), device="cuda")
    _noalloc(w.world, g.views, got, S, w.alpha, w.accumulate)
    torch.cuda.synchronize()
    assert tide.tide_last_device_status(0, _stream()) == tide.TIDE_OK
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"{w.name}: allocation-free fold differs"
    del g, got, ref, init
    torch.cuda.empty_cache()


@pytest.mark.parametrize("seed", range(60))
def test_noalloc_random_groups(seed):
    """Seeded random groups (1..40 ranks, ragged and zero-size parameters,
    trailing ranks without rows, random scale and accumulate) through the
    allocation-free fold, bit-exact against the oracle."""
    import random
    torch.cuda.set_device(0)
    rnd = random.Random(5000 + seed)
    world = rnd.choice([1, 2, 3, 5, 8, 13, 16, 32, 40])
    shapes = []
    for _ in range(rnd.randint(1, 6)):
        d = rnd.choice([0, 1, world - 1 or 1, world, world + 1, rnd.randint(1, 9 * world + 5)])
        shapes.append((d,) if rnd.random() < 0.2 else (d, rnd.choice([1, 2, 3, 8, 17, 64, 130])))
    w = workloads.custom(world, shapes, index=600 + seed)
    g = workloads.make_grads(w, device="cuda")
    dims = w.dim0_rownumel()
    R = [-(-d // world) for d, _ in dims]
    S = sum(r * k for r, (_, k) in zip(R, dims))
    stride = S + rnd.choice([0, 1, 7])
    alpha = rnd.choice([1.0, 0.5, -0.25, 1.0 / world])
    acc = rnd.random() < 0.4
    init = torch.randn(world, max(stride, 1), device="cuda") if acc else torch.zeros(world, max(stride, 1),
                                                                                      device="cuda")
    got = init.clone()
    _noalloc(world, g.views, got, stride, alpha, acc)
    torch.cuda.synchronize()
    assert tide.tide_last_device_status(0, _stream()) == tide.TIDE_OK
    want = oracle_rs_full(world, dims, g.views, alpha, acc, init)
    assert_same_f32(got[:, :S].cpu().numpy(), want[:, :S], f"seed {seed}: W={world} {shapes} acc={acc}")
    assert torch.equal(got[:, S:stride], init[:, S:stride])


def test_noalloc_allocates_nothing_after_set_up():
    torch.cuda.set_device(0)
    w = workloads.custom(8, [(1000, 64), (4096,), (129, 128)], index=126)
    g = workloads.make_grads(w, device="cuda")
    out = torch.zeros(w.world, 200_000, device="cuda")
    tide.tide_rs_fold_noalloc(w.world, [], 0, 0, 1.0, 0, _stream())  # empty call: the per-device set-up
    _noalloc(w.world, g.views, out, out.shape[1], 1.0, False)         # warm-up call
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for i in range(4):
        _noalloc(w.world, g.views, out, out.shape[1], 0.5 * (i + 1), i % 2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device free memory changed across allocation-free calls"
    assert torch.cuda.memory_allocated() == alloc0
    assert tide.tide_last_device_status(0, _stream()) == tide.TIDE_OK


def test_noalloc_rejects_tables_beyond_its_array():
    # 9,000 parameters x 64 ranks = 576,000 pieces: far more table bytes than
    # the fixed array holds; refused on the host before any GPU work.
    W, P = 64, 9000
    fake = [([0x7F0000000000 + 256 * (p * W + u) for u in range(W)], 64, 1, -1) for p in range(P)]
    with pytest.raises(tide.TideError) as e:
        tide.tide_rs_fold_noalloc(W, fake, 0x7E0000000000, 10**6, 1.0, 0, 0)
    assert e.value.status == tide.TIDE_ERR_INVALID_ARG
    assert "bytes of tables" in e.value.detail
