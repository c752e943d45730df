"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Reduce-scatter fold: bit-exact (rank-ascending fp32 order is the contract).
All-gather placement: bit-exact.  Small cases compare every element.  At full
size: every element of both epilogues of each workload, of the other orders
and of fp32 gradients, and of every placement mode; a parameter of
2^31 + 1,024 elements on sampled windows; launch-shape determinism bitwise
across launches.
"""
import random

import numpy as np
import pytest
import torch

import all_gather_gb300 as tide
import oracle
import workloads
from bits import assert_same_bf16, assert_same_f32, assert_same_u16, bf16_bits_to_f32
from gpu_helpers import ag_expected, bits16, full_rs_check, oracle_rs_full, sentinel_slots

U = 2.0 ** -24  # half an ulp of 1.0 in binary32

pytestmark = pytest.mark.gpu

CANARY = float.fromhex("0x1.deadbep+100")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from all_gather_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _fold(w_or_world, grads_uv, alpha, acc, out, **flag_kw):
    world = len(grads_uv)
    flags = tide.make_flags(**flag_kw) if flag_kw else None
    with tide.Plan(grads_uv, flags) as plan:
        plan.rs_fold(out, alpha=alpha, accumulate=acc)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    return out


def _random_grads(world, shapes, seed, scale=1e-3):
    w = workloads.custom(world, shapes, sigma=scale, index=50 + seed % 1000)
    return w, workloads.make_grads(w, device="cuda")


def _guarded_out(world, S, extra, init=None):
    """fp32 [W, S + extra] inside a larger buffer with canary bands around it."""
    stride = S + extra
    buf = torch.full((world * stride + 64,), CANARY, device="cuda", dtype=torch.float32)
    out = buf[32:32 + world * stride].view(world, stride)
    if init is not None:
        out[:, :S].copy_(init[:, :S])
    return buf, out


def _check_canaries(buf, out, S):
    host = buf.cpu().numpy()
    assert (host[:32] == np.float32(CANARY)).all(), "wrote before the output"
    assert (host[32 + out.numel():] == np.float32(CANARY)).all(), "wrote after the output"
    tail = out[:, S:].cpu().numpy()
    assert (tail == np.float32(CANARY)).all(), "wrote past S inside a slot"


KERNELS = {"direct": dict(kernel=tide.TIDE_KERNEL_DIRECT),  # the default schedule: dynamic
           "direct_static": dict(kernel=tide.TIDE_KERNEL_DIRECT, sched=tide.TIDE_SCHED_STATIC),
           "bulk": dict(kernel=tide.TIDE_KERNEL_BULK),
           "bulk_static": dict(kernel=tide.TIDE_KERNEL_BULK, sched=tide.TIDE_SCHED_STATIC),
           # tiny fills and odd rank groups: many stage fills per chunk, groups of 3, 3, ..., remainder
           "bulk_groups": dict(kernel=tide.TIDE_KERNEL_BULK, fill_bytes=64, fill_ranks=3),
           # one short-lived CTA per work item
           "bulk_per_item": dict(kernel=tide.TIDE_KERNEL_BULK, sched=tide.TIDE_SCHED_PER_ITEM),
           # persistent CTAs claiming items from the device counter, few CTAs and odd fills
           "bulk_dynamic_groups": dict(kernel=tide.TIDE_KERNEL_BULK, sched=tide.TIDE_SCHED_DYNAMIC, fill_bytes=64,
                                       fill_ranks=3, cta_budget=5),
           "bulk_static_groups": dict(kernel=tide.TIDE_KERNEL_BULK, sched=tide.TIDE_SCHED_STATIC, fill_bytes=64,
                                      fill_ranks=3, cta_budget=5)}


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("acc", [False, True])
@pytest.mark.parametrize("alpha", ["1/W", 1.0])
@pytest.mark.parametrize("kname", sorted(KERNELS))
def test_toy_full_parity(acc, alpha, kname):
    w = workloads.get(1)
    a = 1.0 / w.world if alpha == "1/W" else alpha
    dims = w.dim0_rownumel()
    gs = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, dims)
    init = workloads.make_out_init(w, S, device="cuda") if acc else None
    buf, out = _guarded_out(w.world, S, 5, init)
    before = out.clone()
    _fold(w, gs.views, a, acc, out, **KERNELS[kname])
    want = oracle_rs_full(w.world, dims, gs.views, a, acc, before)
    assert_same_f32(out[:, :S].cpu().numpy(), want[:, :S], f"toy alpha={a} acc={acc} {kname}")
    _check_canaries(buf, out, S)


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8, 16, 32])
@pytest.mark.parametrize("chunk", [256, 0])
@pytest.mark.parametrize("kname", ["direct", "bulk", "bulk_groups", "bulk_static"])
def test_ragged_shapes(world, chunk, kname):
    rnd = random.Random(world * 101 + chunk)
    shapes = [(rnd.randint(1, 3 * world + 7), rnd.choice([1, 3, 8, 17, 64, 129])) for _ in range(5)]
    shapes += [(world * 37 + 5, 100), (rnd.randint(1, world), 7), (4099,)]
    w, gs = _random_grads(world, shapes, seed=world + chunk)
    dims = w.dim0_rownumel()
    _, _, S = oracle.geometry(world, dims)
    for acc in (False, True):
        init = torch.randn(world, S, device="cuda") if acc else None
        buf, out = _guarded_out(world, S, 3, init)
        before = out.clone()
        _fold(w, gs.views, 1.0 / world, acc, out, chunk_bytes=chunk, **KERNELS[kname])
        want = oracle_rs_full(world, dims, gs.views, 1.0 / world, acc, before)
        assert_same_f32(out[:, :S].cpu().numpy(), want[:, :S], f"ragged W={world} chunk={chunk} acc={acc} {kname}")
        _check_canaries(buf, out, S)


@pytest.mark.parametrize("case", ["uniform_phase", "mixed_phase", "odd_out", "odd_stride"])
@pytest.mark.parametrize("kname", ["direct", "bulk", "bulk_groups"])
def test_misaligned(case, kname):
    world, shapes = 4, [(67, 33), (9, 8), (130, 64), (5,)]
    rnd = random.Random(7)
    numels = [int(np.prod(s)) for s in shapes]
    # each rank's tensors live at chosen element offsets inside one buffer
    views = []
    for u in range(world):
        shift = {"uniform_phase": 3, "mixed_phase": u, "odd_out": 0, "odd_stride": 0}[case]
        buf = torch.empty(sum(numels) + 64 * len(shapes) + 16, dtype=torch.bfloat16, device="cuda")
        vs, cur = [], shift
        for s, n in zip(shapes, numels):
            x = torch.randn(n, device="cuda") * 1e-3
            vs.append(buf[cur:cur + n].view(s))
            vs[-1].copy_(x.view(s).to(torch.bfloat16))
            cur += n + 8 * rnd.randint(0, 3) + (1 if case == "mixed_phase" else 0)
        views.append(vs)
    dims = [(s[0], int(np.prod(s[1:])) if len(s) > 1 else 1) for s in shapes]
    _, _, S = oracle.geometry(world, dims)
    stride = S + (3 if case == "odd_stride" else 0)
    base = torch.full((world * stride + 8,), CANARY, device="cuda", dtype=torch.float32)
    off = 1 if case == "odd_out" else 0
    out = base[off:off + world * stride].view(world, stride)
    before = out.clone()
    _fold(None, views, 0.25, False, out, **KERNELS[kname])
    want = oracle_rs_full(world, dims, views, 0.25, False, before)
    assert_same_f32(out[:, :S].cpu().numpy(), want[:, :S], f"{case} {kname}")


@pytest.mark.parametrize("kname", ["direct", "bulk", "bulk_groups"])
def test_special_values(kname):
    world, shapes = 5, [(41, 24), (13,), (7, 9)]
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 2.0 ** -133, -(2.0 ** -130), 3.3895e38, -3.3895e38,
                         1.0, 2.0 ** -24], dtype=np.float32)
    rng = np.random.default_rng(3)

    def fill(u, p, n, device):
        x = rng.standard_normal(n).astype(np.float32)
        m = rng.random(n) < 0.3
        x[m] = rng.choice(specials, size=int(m.sum()))
        return torch.from_numpy(x).to(device)

    w = workloads.custom(world, shapes, index=77)
    gs = workloads.make_grads(w, device="cuda", fill=fill)
    dims = w.dim0_rownumel()
    _, _, S = oracle.geometry(world, dims)
    for acc in (False, True):
        init = torch.from_numpy(rng.choice(specials, size=(world, S))).cuda() if acc else None
        buf, out = _guarded_out(world, S, 0, init)
        before = out.clone()
        _fold(w, gs.views, 1.0, acc, out, **KERNELS[kname])
        want = oracle_rs_full(world, dims, gs.views, 1.0, acc, before)
        assert_same_f32(out.cpu().numpy(), want, f"special values acc={acc} {kname}")


@pytest.mark.parametrize("world", [2, 3, 8, 32])
@pytest.mark.parametrize("kname", ["direct", "bulk", "bulk_groups"])
def test_order_probe(world, kname):
    """Closed form: 1.0 on rank 0 and 2^-24 elsewhere sums to exactly 1.0 in
    rank order; 1.0 on the last rank gives round(1 + (W-1) 2^-24)."""
    n = 4096 + 3
    for big_rank, expect in ((0, 1.0), (world - 1, float(np.float32(1.0 + (world - 1) * 2.0 ** -24)))):
        grads = [[torch.full((n,), 1.0 if u == big_rank else 2.0 ** -24, device="cuda").to(torch.bfloat16)]
                 for u in range(world)]
        out = torch.zeros(world, -(-n // world), device="cuda")
        _fold(None, grads, 1.0, False, out, **KERNELS[kname])
        flat = out.reshape(-1)[:n].cpu().numpy()
        assert_same_f32(flat, np.full(n, expect, np.float32), f"order probe W={world} big={big_rank}")


def test_determinism_across_launch_shapes():
    w = workloads.get(1)
    gs = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, w.dim0_rownumel())
    ref = None
    for kw in ({}, {"cta_budget": 1}, {"cta_budget": 3}, {"cta_budget": 152}, {"chunk_bytes": 256},
               {"chunk_bytes": 65536}, {"sched": tide.TIDE_SCHED_DYNAMIC, "cta_budget": 7},
               {"sched": tide.TIDE_SCHED_DYNAMIC, "chunk_bytes": 512},
               {"kernel": tide.TIDE_KERNEL_BULK}, {"kernel": tide.TIDE_KERNEL_BULK, "cta_budget": 5},
               {"kernel": tide.TIDE_KERNEL_BULK, "chunk_bytes": 512},
               {"kernel": tide.TIDE_KERNEL_BULK, "fill_bytes": 16, "fill_ranks": 1},
               {"kernel": tide.TIDE_KERNEL_BULK, "fill_bytes": 4096, "fill_ranks": 4},
               {"kernel": tide.TIDE_KERNEL_BULK, "cta_budget": 9},
               {"kernel": tide.TIDE_KERNEL_BULK, "sched": tide.TIDE_SCHED_STATIC},
               {"kernel": tide.TIDE_KERNEL_BULK, "sched": tide.TIDE_SCHED_STATIC, "cta_budget": 2},
               {"kernel": tide.TIDE_KERNEL_BULK, "sched": tide.TIDE_SCHED_STATIC, "cta_budget": 100},
               {"kernel": tide.TIDE_KERNEL_DIRECT, "sched": tide.TIDE_SCHED_STATIC}):
        out = torch.zeros(w.world, S, device="cuda")
        _fold(w, gs.views, 0.25, False, out, **kw)
        got = out.cpu().numpy()
        if ref is None:
            ref = got
        else:
            assert_same_f32(got, ref, f"launch shape {kw}")


ORDER_CASES = [("staged", tide.TIDE_ORDER_STAGED_OWN, 0), ("nodes2", tide.TIDE_ORDER_NODES, 2),
               ("nodes_w", tide.TIDE_ORDER_NODES, -1), ("nodes1", tide.TIDE_ORDER_NODES, 1),
               ("tree", tide.TIDE_ORDER_TREE, 0)]
ORDER_NAMES = {tide.TIDE_ORDER_STAGED_OWN: "staged", tide.TIDE_ORDER_NODES: "nodes", tide.TIDE_ORDER_TREE: "tree",
               tide.TIDE_ORDER_RANK_ASC: "rank"}


def _ordered_fold(grads_uv, alpha, acc, out, order, node_size, f32=False, **kw):
    flags = tide.make_flags(kernel=tide.TIDE_KERNEL_BULK, order=order, node_size=node_size,
                            grad_dtype=tide.TIDE_DTYPE_F32 if f32 else tide.TIDE_DTYPE_BF16, **kw)
    with tide.Plan(grads_uv, flags) as plan:
        plan.rs_fold(out, alpha=alpha, accumulate=acc)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    return out


def _host_grads(grads_uv, f32):
    W, P = len(grads_uv), len(grads_uv[0])
    if f32:
        return [[grads_uv[u][p].reshape(-1).cpu().numpy() for u in range(W)] for p in range(P)]
    return [[bits16(grads_uv[u][p]) for u in range(W)] for p in range(P)]


@pytest.mark.parametrize("case", ORDER_CASES, ids=[c[0] for c in ORDER_CASES])
@pytest.mark.parametrize("f32", [False, True], ids=["bf16", "fp32"])
@pytest.mark.parametrize("world", [1, 3, 4, 6, 8, 32])
def test_orders_and_fp32_grads(case, f32, world):
    """Every Section 4.3 order and the tree order, bf16 and fp32 gradients:
    bit-exact against the oracle in the same order, and within 1e-6 (max-norm,
    per parameter and rank) of the rank-order oracle.  The fill_ranks = 3
    launch runs the tree in fills of 2 ranks (the deep counter at W = 32)."""
    name, order, L = case
    L = world if L == -1 else L
    if order == tide.TIDE_ORDER_NODES and world % L:
        pytest.skip("node size must divide the world")
    rnd = random.Random(world * 7 + L)
    shapes = [(rnd.randint(1, 3 * world + 7), rnd.choice([1, 3, 8, 17, 64])) for _ in range(4)]
    shapes += [(world * 37 + 5, 100), (4099,)]
    w = workloads.custom(world, shapes, index=200 + world)
    gs = workloads.make_grads(w, device="cuda")
    views = [[v.float() for v in gs.views[u]] for u in range(world)] if f32 else gs.views
    if f32:  # fp32 gradients carry bits below bf16 precision
        views = [[v + torch.randn_like(v) * 1e-6 for v in vs] for vs in views]
    dims = w.dim0_rownumel()
    R, o, S = oracle.geometry(world, dims)
    oname = ORDER_NAMES[order]
    host = _host_grads(views, f32)
    for acc, kw in ((False, {}), (True, {"fill_bytes": 64, "fill_ranks": 3}), (False, {"chunk_bytes": 256})):
        init = torch.randn(world, S, device="cuda") if acc else None
        buf, out = _guarded_out(world, S, 2, init)
        before = out.clone()
        _ordered_fold(views, 0.5, acc, out, order, L if order == tide.TIDE_ORDER_NODES else 0, f32, **kw)
        want = before.cpu().numpy().copy()
        oracle.rs_ex(world, dims, host, 0.5, acc, want, oname, L if oname == "nodes" else 0)
        got = out.cpu().numpy()
        assert_same_f32(got[:, :S], want[:, :S], f"{name} f32={f32} W={world} acc={acc} {kw}")
        _check_canaries(buf, out, S)
        rank = before.cpu().numpy().copy()
        oracle.rs_ex(world, dims, host, 0.5, acc, rank, "rank", 0)
        old_h = before.cpu().numpy()
        gamma = (world + 1) * 2.0 ** -24 / (1 - (world + 1) * 2.0 ** -24)
        for p, (d, k) in enumerate(dims):
            a = np.concatenate([got[r, o[p]:o[p] + R[p] * k] for r in range(world)])[:d * k]
            b = np.concatenate([rank[r, o[p]:o[p] + R[p] * k] for r in range(world)])[:d * k]
            if d * k >= 1024:  # reordered-variant tolerance, max-norm over the parameter tensor
                assert np.abs(a - b).max() <= 1e-6 * np.abs(b).max(), f"{name} tolerance p={p}"
            # any order: textbook bound around the exact sum, for every element
            vals = np.stack([np.asarray(host[p][u], dtype=np.float32).astype(np.float64) if f32 else
                             bf16_bits_to_f32(host[p][u]).astype(np.float64) for u in range(world)])
            base = np.concatenate([old_h[r, o[p]:o[p] + R[p] * k] for r in range(world)])[:d * k].astype(np.float64)
            exact = 0.5 * vals.sum(0) + (base if acc else 0.0)
            mag = 0.5 * np.abs(vals).sum(0) + (np.abs(base) if acc else 0.0)
            assert (np.abs(a.astype(np.float64) - exact) <= gamma * mag + 1e-45).all(), f"{name} bound p={p}"


@pytest.mark.parametrize("f32", [False, True], ids=["bf16", "fp32"])
def test_orders_misaligned_pieces(f32):
    """Pieces the bulk producer cannot stage (rank phases differ) take the
    scalar path, in the same order."""
    world, shapes = 4, [(67, 33), (9, 8), (5,)]
    esz = 4 if f32 else 2
    dt = torch.float32 if f32 else torch.bfloat16
    views = []
    for u in range(world):
        buf = torch.empty(4096, dtype=dt, device="cuda")
        vs, cur = [], u + 1
        for s_ in shapes:
            n = int(np.prod(s_))
            vs.append(buf[cur:cur + n].view(s_))
            vs[-1].copy_(torch.randn(s_, device="cuda").to(dt))
            cur += n + 3
        views.append(vs)
    dims = [(s_[0], int(np.prod(s_[1:])) if len(s_) > 1 else 1) for s_ in shapes]
    _, _, S = oracle.geometry(world, dims)
    host = _host_grads(views, f32)
    for order, L, oname in ((tide.TIDE_ORDER_STAGED_OWN, 0, "staged"), (tide.TIDE_ORDER_NODES, 2, "nodes"),
                            (tide.TIDE_ORDER_RANK_ASC, 0, "rank"), (tide.TIDE_ORDER_TREE, 0, "tree")):
        out = torch.zeros(world, S, device="cuda")
        _ordered_fold(views, 1.0, False, out, order, L, f32)
        want = np.zeros((world, S), np.float32)
        oracle.rs_ex(world, dims, host, 1.0, False, want, oname, L)
        assert_same_f32(out.cpu().numpy(), want, f"misaligned {oname} f32={f32}")


TREE_PROBES = [([1.0, U, U], 1.0), ([U, U, 1.0], 1 + 2 ** -23), ([1.0, U, U, U], 1 + 2 ** -23),
               ([1.0] + [U] * 4, 1 + 2 ** -22), ([1.0, 0.0, U, U, 0.0, 0.0], 1 + 2 ** -23),
               ([1.0] + [U] * 6, 1 + 2 ** -22), ([1.0] + [U] * 7, 1 + 3 * 2 ** -23),
               ([1.0] + [U] * 15, 1 + 7 * 2 ** -23), ([1.0] + [U] * 11, None)]


@pytest.mark.parametrize("case", range(len(TREE_PROBES)))
@pytest.mark.parametrize("fill_ranks", [0, 2, 4])
def test_tree_order_probe(case, fill_ranks):
    """Hand-worked pairwise sums of 1.0 and 2^-24 terms (rank q holds vals[q]
    in every element): W = 3 .. 16, whole-vector, tail and padding elements,
    stage fills of 8, 2 and 4 ranks; the last case (W = 12) is checked against
    the oracle."""
    vals, want = TREE_PROBES[case]
    world = len(vals)
    shapes = [(world * 300 + 5, 8), (world + 1, 3)]
    w = workloads.custom(world, shapes, index=700 + world)
    gs = workloads.make_grads(w, device="cuda", fill=lambda u, p, n, dev: torch.full((n,), vals[u], device=dev))
    dims = w.dim0_rownumel()
    R, o, S = oracle.geometry(world, dims)
    out = torch.zeros(world, S, device="cuda")
    _ordered_fold(gs.views, 1.0, False, out, tide.TIDE_ORDER_TREE, 0, fill_ranks=fill_ranks)
    got = out.cpu().numpy()
    if want is None:
        ref = np.zeros((world, S), np.float32)
        oracle.rs_ex(world, dims, _host_grads(gs.views, False), 1.0, False, ref, "tree", 0)
        assert_same_f32(got, ref, "tree W=12 vs oracle")
        return
    for p, (d, k) in enumerate(dims):
        flat = np.concatenate([got[r, o[p]:o[p] + R[p] * k] for r in range(world)])[:d * k]
        assert_same_f32(flat, np.full(d * k, want, np.float32), f"tree probe W={world} p={p}")


def _random_flags(rnd, world):
    """A valid random flag set: orders other than rank order and fp32
    gradients take the bulk kernel (any schedule)."""
    order = rnd.choice([tide.TIDE_ORDER_RANK_ASC] * 3 + [tide.TIDE_ORDER_STAGED_OWN, tide.TIDE_ORDER_NODES,
                                                         tide.TIDE_ORDER_TREE])
    f32 = rnd.random() < 0.3
    restricted = order != tide.TIDE_ORDER_RANK_ASC or f32
    kernel = tide.TIDE_KERNEL_BULK if restricted else rnd.choice(
        [tide.TIDE_KERNEL_AUTO, tide.TIDE_KERNEL_DIRECT, tide.TIDE_KERNEL_BULK])
    sched = rnd.choice([tide.TIDE_SCHED_AUTO, tide.TIDE_SCHED_DYNAMIC, tide.TIDE_SCHED_STATIC,
                        tide.TIDE_SCHED_STATIC, tide.TIDE_SCHED_PER_ITEM])
    kw = dict(kernel=kernel, sched=sched, order=order,
              grad_dtype=tide.TIDE_DTYPE_F32 if f32 else tide.TIDE_DTYPE_BF16,
              cta_budget=0 if sched == tide.TIDE_SCHED_PER_ITEM else rnd.choice([0, 0, 1, 3, rnd.randint(1, 400)]),
              chunk_bytes=rnd.choice([0, 256, 256 * rnd.randint(1, 256)]),
              fill_bytes=rnd.choice([0, 16, 16 * rnd.randint(1, 1024)]),
              fill_ranks=rnd.choice([0, 1, 2, rnd.randint(1, world + 2)]))
    if order == tide.TIDE_ORDER_NODES:
        kw["node_size"] = rnd.choice([d for d in range(1, world + 1) if world % d == 0])
    oname = {tide.TIDE_ORDER_RANK_ASC: "rank", tide.TIDE_ORDER_STAGED_OWN: "staged",
             tide.TIDE_ORDER_NODES: "nodes", tide.TIDE_ORDER_TREE: "tree"}[order]
    return kw, oname, f32


@pytest.mark.parametrize("seed", range(1000))
def test_random_flag_combinations(seed):
    """Seeded random groups (1..40 ranks, ragged shapes, zero-size parameters)
    under random valid flag sets and epilogues: the fold bit-exact against
    the oracle in the same order, canary bands intact, and a random placement
    mode bit-exact."""
    rnd = random.Random(1000 + seed)
    world = rnd.choice([1, 2, 3, 5, 7, 8, 12, 16, 31, 40])
    shapes = []
    for _ in range(rnd.randint(1, 6)):
        d = rnd.choice([0, 1, world - 1 or 1, world, world + 1, rnd.randint(1, 9 * world + 5)])
        shapes.append((d,) if rnd.random() < 0.2 else (d, rnd.choice([1, 2, 3, 8, 17, 64, 130])))
    kw, oname, f32 = _random_flags(rnd, world)
    w = workloads.custom(world, shapes, index=400 + seed)
    gs = workloads.make_grads(w, device="cuda")
    views = gs.views
    if f32:
        views = [[v.float() + 1e-6 * torch.randn_like(v.float()) for v in vs] for vs in views]
    dims = w.dim0_rownumel()
    _, _, S = oracle.geometry(world, dims)
    alpha = rnd.choice([1.0, 0.5, -0.25, 1.0 / world, 3.0])
    acc = rnd.random() < 0.4
    init = torch.randn(world, S, device="cuda") if acc else None
    buf, out = _guarded_out(world, S, rnd.choice([0, 1, 5, 64]), init)
    before = out.clone()
    flags = tide.make_flags(**kw)
    with tide.Plan(views, flags) as plan:
        plan.rs_fold(out, alpha=alpha, accumulate=acc)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
        want = before.cpu().numpy().copy()
        oracle.rs_ex(world, dims, _host_grads(views, f32), alpha, acc, want, oname, kw.get("node_size", 0))
        assert_same_f32(out.cpu().numpy()[:, :S], want[:, :S], f"seed {seed}: W={world} {kw} acc={acc}")
        _check_canaries(buf, out, S)
        # a placement in a random mode, from sentinel slots
        mode = rnd.choice(["sm", "ce2d", "ce1d"])
        slots = sentinel_slots(world, dims, S + rnd.choice([0, 3, 8]), seed=seed)
        full = [torch.full(s_, float("nan"), dtype=torch.bfloat16, device="cuda") for s_ in w.shapes]
        plan.ag_place(slots, full, mode=mode)
        torch.cuda.synchronize()
        wf = ag_expected(world, dims, slots)
        for p, f in enumerate(full):
            assert_same_u16(bits16(f), wf[p], f"seed {seed}: ag {mode} p={p}")


@pytest.mark.parametrize("sched_kw", [{}, {"sched": tide.TIDE_SCHED_DYNAMIC},
                                      {"sched": tide.TIDE_SCHED_DYNAMIC, "cta_budget": 3}],
                         ids=["default", "dynamic", "dynamic_3ctas"])
def test_bulk_wait_timeout_reports_status(sched_kw):
    """A bounded device-side wait that expires is reported as TIMEOUT and the
    context stays usable: the CTA that takes work item 0 skips that item's
    first stage fill (debug flag), its consumers give up after 50 ms, the
    producer drains the copies it issued, and the kernel returns.  A second
    launch of the same plan times out the same way, which under the dynamic
    schedule shows that the aborted launch reset the claim counters (else
    item 0 would never be claimed again); a plan with the same schedule and no
    planted skip then matches the oracle."""
    w = workloads.get(1)
    gs = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, w.dim0_rownumel())
    flags = tide.make_flags(kernel=tide.TIDE_KERNEL_BULK,
                            debug=tide.TIDE_DEBUG_SHORT_WAIT | tide.TIDE_DEBUG_SKIP_FILL, **sched_kw)
    out = torch.zeros(w.world, S, device="cuda")
    with tide.Plan(gs.views, flags) as plan:
        for _ in range(2):
            plan.rs_fold(out, alpha=0.25)
            torch.cuda.synchronize()
            assert plan.device_status() == tide.TIDE_ERR_TIMEOUT
            assert plan.device_status() == tide.TIDE_OK  # reading clears the word
    if sched_kw:  # the same schedule without the planted skip, twice on one plan: counters reset
        with tide.Plan(gs.views, tide.make_flags(kernel=tide.TIDE_KERNEL_BULK, **sched_kw)) as plan:
            want = oracle_rs_full(w.world, w.dim0_rownumel(), gs.views, 0.25, False, torch.zeros(w.world, S))
            for _ in range(2):
                out = torch.zeros(w.world, S, device="cuda")
                plan.rs_fold(out, alpha=0.25)
                torch.cuda.synchronize()
                assert plan.device_status() == tide.TIDE_OK
                assert_same_f32(out.cpu().numpy(), want, "dynamic schedule after a timeout")
    # the context is healthy: a normal fold still matches the oracle
    out = torch.zeros(w.world, S, device="cuda")
    _fold(w, gs.views, 0.25, False, out, kernel=tide.TIDE_KERNEL_BULK)
    want = oracle_rs_full(w.world, w.dim0_rownumel(), gs.views, 0.25, False, torch.zeros(w.world, S))
    assert_same_f32(out.cpu().numpy(), want, "after timeout")


@pytest.mark.parametrize("world", [33, 257, 1024])
def test_maximum_and_odd_worlds(world):
    """The widest groups: up to 1024 virtual ranks (the library's maximum),
    every kernel, rank order and the one-node order, against the oracle."""
    shapes = [(world * 3 + 1, 24), (world // 2 + 1, 8), (7,)]
    w = workloads.custom(world, shapes, index=300 + world)
    gs = workloads.make_grads(w, device="cuda")
    dims = w.dim0_rownumel()
    _, _, S = oracle.geometry(world, dims)
    host = _host_grads(gs.views, False)
    for kw, oname in (({"kernel": tide.TIDE_KERNEL_DIRECT}, "rank"), ({"kernel": tide.TIDE_KERNEL_BULK}, "rank"),
                      ({"kernel": tide.TIDE_KERNEL_BULK, "order": tide.TIDE_ORDER_STAGED_OWN}, "staged"),
                      ({"kernel": tide.TIDE_KERNEL_BULK, "order": tide.TIDE_ORDER_TREE}, "tree")):
        out = torch.zeros(world, S, device="cuda")
        with tide.Plan(gs.views, tide.make_flags(**kw)) as plan:
            plan.rs_fold(out, alpha=1.0 / world)
            torch.cuda.synchronize()
            assert plan.device_status() == tide.TIDE_OK
        want = np.zeros((world, S), np.float32)
        oracle.rs_ex(world, dims, host, 1.0 / world, False, want, oname, 0)
        assert_same_f32(out.cpu().numpy(), want, f"W={world} {kw}")


def test_repeated_calls_and_rebind():
    w = workloads.get(1)
    dims = w.dim0_rownumel()
    g1 = workloads.make_grads(w, device="cuda")
    w2 = workloads.custom(w.world, w.shapes, index=91)
    g2 = workloads.make_grads(w2, device="cuda")
    _, _, S = oracle.geometry(w.world, dims)
    flags = tide.make_flags(sched=tide.TIDE_SCHED_DYNAMIC)
    with tide.Plan(g1.views, flags) as plan:
        for grads in (g1, g2, g1):
            plan.rebind(grads.views)
            for _ in range(3):  # the dynamic-schedule counters must reset between launches
                out = torch.zeros(w.world, S, device="cuda")
                plan.rs_fold(out, alpha=0.5)
                torch.cuda.synchronize()
                want = oracle_rs_full(w.world, dims, grads.views, 0.5, False, torch.zeros(w.world, S))
                assert_same_f32(out.cpu().numpy(), want, "rebind")


def test_empty_and_degenerate():
    # no parameters at all
    with tide.Plan([[] for _ in range(3)]) as plan:
        assert plan.slot_numel == 0
        plan.rs_fold(torch.zeros(3, 1, device="cuda"))
    # zero-size parameters mixed with real ones
    shapes = [(0, 5), (3, 2), (4, 0)]
    grads = [[torch.zeros(s, dtype=torch.bfloat16, device="cuda") + u for s in shapes] for u in range(2)]
    dims = [(0, 5), (3, 2), (4, 0)]
    _, _, S = oracle.geometry(2, dims)
    out = torch.full((2, S), 9.0, device="cuda")
    with tide.Plan(grads) as plan:
        assert plan.slot_numel == S
        plan.rs_fold(out)
        torch.cuda.synchronize()
    want = oracle_rs_full(2, dims, grads, 1.0, False, torch.full((2, S), 9.0))
    assert_same_f32(out.cpu().numpy(), want, "degenerate shapes")


def test_call_errors():
    w = workloads.get(1)
    gs = workloads.make_grads(w, device="cuda")
    with tide.Plan(gs.views) as plan:
        S = plan.slot_numel
        with pytest.raises(tide.TideError) as e:  # output aliasing a gradient
            tide.tide_rs_fold(plan.handle, gs.arenas[2].data_ptr(), S, 1.0, 0, 0)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        out = torch.zeros(w.world * S + 1, device="cuda")
        with pytest.raises(tide.TideError) as e:  # 2-byte misaligned fp32 output
            tide.tide_rs_fold(plan.handle, out.data_ptr() + 2, S, 1.0, 0, 0)
        assert e.value.status == tide.TIDE_ERR_ALIGNMENT
        with pytest.raises(tide.TideError) as e:  # stride below S
            tide.tide_rs_fold(plan.handle, out.data_ptr(), S - 1, 1.0, 0, 0)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        with pytest.raises(tide.TideError):
            tide.tide_rs_fold(plan.handle, out.data_ptr(), S, 1.0, 2, 0)
        slots = torch.zeros(w.world, S, dtype=torch.bfloat16, device="cuda")
        full = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in w.shapes]
        with pytest.raises(tide.TideError) as e:  # a full tensor inside the slots
            tide.tide_ag_place(plan.handle, slots.data_ptr(), S, [slots.data_ptr()] + [f.data_ptr() for f in full[1:]],
                               tide.TIDE_AG_SM, 0)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        with pytest.raises(tide.TideError):
            tide.tide_ag_place(plan.handle, slots.data_ptr(), S, [f.data_ptr() for f in full], 9, 0)


# ---------------------------------------------------------------------------
# all-gather placement
@pytest.mark.parametrize("mode", ["sm", "ce2d", "ce1d"])
def test_ag_toy_and_ragged(mode):
    cases = [workloads.get(1)]
    rnd = random.Random(5)
    for world in (1, 3, 8, 16):
        shapes = [(rnd.randint(1, 4 * world + 3), rnd.choice([1, 5, 8, 64])) for _ in range(4)] + [(world * 100 + 1,)]
        cases.append(workloads.custom(world, shapes, index=60 + world))
    for w in cases:
        dims = w.dim0_rownumel()
        _, _, S = oracle.geometry(w.world, dims)
        grads = workloads.make_grads(w, device="cuda")  # only used to build the plan's geometry
        slots = sentinel_slots(w.world, dims, S + 7, seed=w.index)
        total = sum(d * k for d, k in dims)
        guard = 64
        buf = torch.full((total + guard * (len(dims) + 1),), -7.0, device="cuda").to(torch.bfloat16)
        full, cur = [], guard
        for s, (d, k) in zip(w.shapes, dims):
            full.append(buf[cur:cur + d * k].view(s))
            cur += d * k + guard
        with tide.Plan(grads.views) as plan:
            # the full tensors as a list (checked per call) or bound once
            plan.ag_place(slots, plan.bind_full(full) if w.world % 2 else full, mode=mode)
            torch.cuda.synchronize()
        want = ag_expected(w.world, dims, slots)
        for p, f in enumerate(full):
            assert_same_u16(bits16(f), want[p], f"ag {mode} {w.name} p={p}")
        host = bits16(buf)
        guard_bits = bits16(torch.tensor([-7.0], dtype=torch.bfloat16))[0]
        cur = 0
        for d, k in dims:
            assert (host[cur:cur + guard] == guard_bits).all(), "placement wrote outside a full tensor"
            cur += guard + d * k
        assert (host[cur:] == guard_bits).all()


@pytest.mark.parametrize("case", ["aligned", "odd_slots", "odd_full"])
def test_ag_f32_mixed_precision(case):
    """fp32 master-shard slots -> bf16 full tensors, against the oracle's
    round-to-nearest-even placement; rounding-critical values and NaN padding."""
    rnd = random.Random(31)
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 3.4e38, -3.4e38, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8,
                         1.0 + 2.0 ** -8 + 2.0 ** -20, 2.0 ** -130, 1e-40], dtype=np.float32)
    for world in (1, 3, 4, 8):
        shapes = [(rnd.randint(1, 4 * world + 3), rnd.choice([1, 5, 8, 64])) for _ in range(4)] + [(world * 100 + 1,)]
        w = workloads.custom(world, shapes, index=80 + world)
        dims = w.dim0_rownumel()
        R, o, S = oracle.geometry(world, dims)
        rng = np.random.default_rng(world)
        host = rng.standard_normal((world, S + 5)).astype(np.float32)
        m = rng.random(host.shape) < 0.2
        host[m] = rng.choice(specials, size=int(m.sum()))
        mask = np.ones(host.shape, dtype=bool)
        for p, (d, k) in enumerate(dims):
            for r in range(world):
                mask[r, o[p]:o[p] + oracle.valid_rows(d, R[p], r) * k] = False
        host[mask] = np.nan
        off = 1 if case == "odd_slots" else 0
        buf = torch.from_numpy(np.concatenate([np.zeros(off, np.float32), host.reshape(-1)])).cuda()
        slots = buf[off:].view(world, S + 5)
        grads = workloads.make_grads(w, device="cuda")
        foff = 3 if case == "odd_full" else 0
        fbuf = torch.zeros(sum(d * k for d, k in dims) + foff + 8 * len(dims), dtype=torch.bfloat16, device="cuda")
        full, cur = [], foff
        for s_, (d, k) in zip(w.shapes, dims):
            full.append(fbuf[cur:cur + d * k].view(s_))
            cur += d * k + 8
        with tide.Plan(grads.views) as plan:
            plan.ag_place_f32(slots, full)
            torch.cuda.synchronize()
        want = oracle.ag_cast(world, dims, host)
        for p, f in enumerate(full):
            assert_same_bf16(bits16(f), want[p], f"ag_f32 {case} W={world} p={p}")


def test_ag_shard_roundtrip_identity():
    """AG(shard(x)) == x for full-size-like shapes with misaligned offsets."""
    world = 8
    shapes = [(1000, 33), (77,), (64, 64)]
    xs = [torch.randn(s, device="cuda").to(torch.bfloat16) for s in shapes]
    dims = [(s[0], int(np.prod(s[1:])) if len(s) > 1 else 1) for s in shapes]
    R, o, S = oracle.geometry(world, dims)
    slots = torch.full((world, S + 1), float("nan"), device="cuda").to(torch.bfloat16)
    for p, x in enumerate(xs):
        for r, ch in enumerate(torch.chunk(x, world)):
            slots[r, o[p]:o[p] + ch.numel()] = ch.reshape(-1)
    grads = [[torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in shapes] for _ in range(world)]
    for mode in ("sm", "ce2d", "ce1d"):
        full = [torch.empty_like(x) for x in xs]
        with tide.Plan(grads) as plan:
            plan.ag_place(slots, full, mode=mode)
            torch.cuda.synchronize()
        for p, (x, f) in enumerate(zip(xs, full)):
            assert_same_u16(bits16(f), bits16(x), f"AG(shard(x)) {mode} p={p}")


@pytest.mark.parametrize("kw", [{}, {"sched": tide.TIDE_SCHED_DYNAMIC},
                                {"sched": tide.TIDE_SCHED_DYNAMIC, "cta_budget": 3}],
                         ids=["default", "dynamic", "dynamic_3ctas"])
def test_graph_captured_step(kw):
    """The step (fold, placement, mixed-precision placement) captured once in a
    CUDA graph and replayed on new inputs copied into the same buffers; with
    the dynamic schedule every replay must find the claim counters reset."""
    w = workloads.get(1)
    dims = w.dim0_rownumel()
    g1 = workloads.make_grads(w, device="cuda")
    g2 = workloads.make_grads(workloads.custom(w.world, w.shapes, index=93), device="cuda")
    _, _, S = oracle.geometry(w.world, dims)
    out = torch.zeros(w.world, S, device="cuda")
    slots = workloads.make_slots(w, S, device="cuda")
    slots32 = torch.randn(w.world, S, device="cuda")
    full = [torch.empty(s_, dtype=torch.bfloat16, device="cuda") for s_ in w.shapes]
    full32 = [torch.empty_like(f) for f in full]
    with tide.Plan(g1.views, tide.make_flags(**kw) if kw else None) as plan:
        plan.rs_fold(out, alpha=0.25)  # warm-up outside the capture
        plan.ag_place(slots, full)
        plan.ag_place_f32(slots32, full32)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            plan.rs_fold(out, alpha=0.25)
            plan.ag_place(slots, full)
            plan.ag_place_f32(slots32, full32)
        for src in (g2, g1, g2):
            for a, b in zip(g1.arenas, src.arenas):
                if a.data_ptr() != b.data_ptr():
                    a.copy_(b)
            slots.copy_(slots.flip(0))
            slots32.mul_(-1.5)
            out.zero_()
            graph.replay()
            torch.cuda.synchronize()
            want = oracle_rs_full(w.world, dims, src.views, 0.25, False, torch.zeros(w.world, S))
            assert_same_f32(out.cpu().numpy(), want, "replayed fold")
            wf = ag_expected(w.world, dims, slots)
            wf32 = oracle.ag_cast(w.world, dims, slots32.cpu().numpy())
            for p in range(len(dims)):
                assert_same_u16(bits16(full[p]), wf[p], "replayed placement")
                assert_same_bf16(bits16(full32[p]), wf32[p], "replayed mixed-precision placement")
        del graph


@pytest.mark.parametrize("mode", ["ce2d", "ce1d"])
@pytest.mark.parametrize("index", [1, 5])
def test_graph_captured_copy_engine_placement(mode, index):
    """The copy-engine placement (copies spread over the plan's internal
    streams, forked from and joined back to the caller's stream) captured once
    in a CUDA graph and replayed on new slot contents: the replay places every
    shard as the oracle does.  The MoE layer (389 parameters) is its largest
    copy list."""
    w = workloads.get(index)
    dims = w.dim0_rownumel()
    g = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, dims)
    slots = workloads.make_slots(w, S, device="cuda")
    full = [torch.empty(s_, dtype=torch.bfloat16, device="cuda") for s_ in w.shapes]
    stream = torch.cuda.Stream()
    with tide.Plan(g.views) as plan:
        bound = plan.bind_full(full)
        with torch.cuda.stream(stream):
            plan.ag_place(slots, bound, mode=mode)  # warm-up outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            plan.ag_place(slots, bound, mode=mode)
        for step in range(3):
            slots.copy_(slots.roll(step + 1, dims=0))
            for f in full:
                f.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            host_slots = slots.cpu()
            if index == 1:
                want = ag_expected(w.world, dims, slots)
                for p in range(len(dims)):
                    assert_same_u16(bits16(full[p]), want[p], f"replayed {mode} placement p={p}")
            else:  # every parameter, sampled rows: full row i of rank r is slot r at o_p + i K
                R, o, _ = oracle.geometry(w.world, dims)
                rnd = random.Random(step)
                for p in rnd.sample(range(len(dims)), 40):
                    d, k = dims[p]
                    for row in rnd.sample(range(d), min(d, 8)):
                        r, i = divmod(row, R[p])
                        got = full[p].reshape(-1)[row * k:(row + 1) * k].cpu()
                        ref = host_slots[r, o[p] + i * k:o[p] + (i + 1) * k]
                        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (mode, p, row)
        del graph
    del g
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration
@pytest.mark.parametrize("index", [2, 3, 4, 5])
def test_full_size_epilogues_and_placements(index):
    """Full-size workloads: the fold with the benchmark's epilogue and with the
    other one (alpha = 1/W, accumulate flipped), every output element against
    the oracle; every placement mode and the mixed-precision placement, every
    element."""
    w = workloads.get(index)
    dims = w.dim0_rownumel()
    gs = workloads.make_grads(w, device="cuda")
    R, o, S = oracle.geometry(w.world, dims)
    with tide.Plan(gs.views) as plan:   # default flags: what the benchmark times
        assert plan.slot_numel == S
        for alpha, acc in ((w.alpha, w.accumulate), (1.0 / w.world, not w.accumulate)):
            out = workloads.make_out_init(w, S, device="cuda") if acc else torch.empty(w.world, S, device="cuda")
            before = out.clone() if acc else None
            plan.rs_fold(out, alpha=alpha, accumulate=acc)
            torch.cuda.synchronize()
            n = full_rs_check(w.world, dims, gs.views, before, out, alpha, acc,
                              what=f"{w.name} alpha={alpha} acc={acc}")
            assert n == w.world * S
            del out, before
        # all-gather placement of full-size slots, every element
        slots = workloads.make_slots(w, S, device="cuda")
        full = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in w.shapes]
        plan.ag_place(slots, full, mode="sm")
        torch.cuda.synchronize()
        want = ag_expected(w.world, dims, slots)
        for p, f in enumerate(full):
            assert_same_u16(bits16(f), want[p], f"{w.name} ag p={p}")
        # the copy-engine placements, every element
        bound = plan.bind_full(full)
        for mode in ("ce2d", "ce1d"):
            for f in full:
                f.fill_(float("nan"))
            plan.ag_place(slots, bound, mode=mode)
            torch.cuda.synchronize()
            for p, f in enumerate(full):
                assert_same_u16(bits16(f), want[p], f"{w.name} ag {mode} p={p}")
        # mixed-precision placement from fp32 master shards, every element
        del slots
        slots32 = torch.stack([workloads.normal_fp32(S, workloads.slot_seed(w, r), 0.02, "cuda")
                               for r in range(w.world)])
        plan.ag_place_f32(slots32, full)
        torch.cuda.synchronize()
        want = oracle.ag_cast(w.world, dims, slots32.cpu().numpy())
        for p, f in enumerate(full):
            assert_same_bf16(bits16(f), want[p], f"{w.name} ag_f32 p={p}")
    del gs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("index", [2, 3, 5])
def test_full_size_bitwise_across_launch_shapes(index):
    """Full-size groups: the rank-order fold is bitwise identical, over every
    output element, at full wave (two CTAs per SM), with 152, 64, 16 and 7 CTAs
    (one CTA per SM: eight consumer warps and 16 KB copies), with one CTA per
    work item, with the direct-load kernel, and with odd stage shapes."""
    w = workloads.get(index)
    gs = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, w.dim0_rownumel())
    init = workloads.make_out_init(w, S, device="cuda") if w.accumulate else None
    ref = None
    for kw in ({}, {"cta_budget": 152}, {"cta_budget": 64}, {"cta_budget": 16}, {"cta_budget": 7},
               {"sched": tide.TIDE_SCHED_PER_ITEM}, {"sched": tide.TIDE_SCHED_STATIC},
               {"sched": tide.TIDE_SCHED_STATIC, "cta_budget": 16}, {"kernel": tide.TIDE_KERNEL_DIRECT},
               {"kernel": tide.TIDE_KERNEL_DIRECT, "sched": tide.TIDE_SCHED_PER_ITEM},
               {"fill_bytes": 1008, "fill_ranks": 3},
               {"cta_budget": 32, "fill_bytes": 12288, "fill_ranks": 5}):
        out = init.clone() if init is not None else torch.zeros(w.world, S, device="cuda")
        with tide.Plan(gs.views, tide.make_flags(**kw)) as plan:
            plan.rs_fold(out, alpha=w.alpha, accumulate=w.accumulate)
            torch.cuda.synchronize()
            assert plan.device_status() == tide.TIDE_OK
        if ref is None:
            ref = out
        else:
            same = torch.equal(out.view(torch.int32), ref.view(torch.int32))
            assert same, f"{w.name}: {kw} differs from the full-wave fold"
            del out
    del gs, ref, init
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["bulk", "direct"])
def test_explicit_shard_offsets(kernel):
    """Caller-chosen shard offsets (parameters in reverse order inside the
    slot, odd gaps, so fp32 and bf16 windows start misaligned): every
    parameter's fold window equals the oracle's window for that parameter,
    the gaps keep their canaries, and every placement mode reads the shards
    from those offsets."""
    world = 5
    shapes = [(23, 16), (9, 3), (64,), (11, 8)]
    w = workloads.custom(world, shapes, index=510)
    dims = w.dim0_rownumel()
    R, o, S = oracle.geometry(world, dims)
    sizes = [R[p] * k for p, (_, k) in enumerate(dims)]
    offsets, cur = [0] * len(dims), 3
    for p in reversed(range(len(dims))):
        offsets[p] = cur
        cur += sizes[p] + 5
    stride = cur + 2
    gs = workloads.make_grads(w, device="cuda")
    kw = {"kernel": tide.TIDE_KERNEL_DIRECT} if kernel == "direct" else {}
    want = oracle_rs_full(world, dims, gs.views, 0.5, False, torch.zeros(world, S))
    with tide.Plan(gs.views, tide.make_flags(**kw), offsets=offsets) as plan:
        assert plan.slot_numel == cur - 5
        out = torch.full((world, stride), CANARY, device="cuda")
        plan.rs_fold(out, alpha=0.5)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        mask = np.ones((world, stride), bool)
        for p in range(len(dims)):
            assert_same_f32(got[:, offsets[p]:offsets[p] + sizes[p]], want[:, o[p]:o[p] + sizes[p]],
                            f"{kernel} p={p} at offset {offsets[p]}")
            mask[:, offsets[p]:offsets[p] + sizes[p]] = False
        assert (got[mask] == np.float32(CANARY)).all(), "the fold wrote into a gap between shards"
        # placement: slots hold each shard at its explicit offset
        prefix = sentinel_slots(world, dims, S, seed=11)
        slots = torch.full((world, stride), float("nan"), dtype=torch.bfloat16, device="cuda")
        for p in range(len(dims)):
            slots[:, offsets[p]:offsets[p] + sizes[p]] = prefix[:, o[p]:o[p] + sizes[p]]
        wf = ag_expected(world, dims, prefix)
        for mode in ("sm", "ce2d", "ce1d"):
            full = [torch.full(s_, float("nan"), dtype=torch.bfloat16, device="cuda") for s_ in w.shapes]
            plan.ag_place(slots, full, mode=mode)
            torch.cuda.synchronize()
            for p, f in enumerate(full):
                assert_same_u16(bits16(f), wf[p], f"{mode} p={p} from offset {offsets[p]}")


def test_parameter_beyond_2g_elements():
    """One parameter of 2,097,153 x 1,024 = 2^31 + 1,024 elements on 2 ranks
    (about 26 GB with outputs): rank 1's rows start at element 1,073,742,848 and
    end past 2^31, so every offset of the fold and the placements must be 64-bit.
    Every output element against the oracle, both kernels and the tree order;
    every element of the placements, every mode (compared on the device with
    Equation (2)'s two row ranges: rank r's shard is rows [r R, r R + v_r))."""
    world, shape = 2, (2_097_153, 1024)
    w = workloads.custom(world, [shape, (5, 3)], index=77)
    dims = w.dim0_rownumel()
    gs = workloads.make_grads(w, device="cuda")
    R, o, S = oracle.geometry(world, dims)
    out = torch.empty(world, S, device="cuda")
    for kw, oname in (({}, "rank"), ({"kernel": tide.TIDE_KERNEL_DIRECT}, "rank"),
                      ({"order": tide.TIDE_ORDER_TREE}, "tree")):
        out.fill_(float("nan"))
        with tide.Plan(gs.views, tide.make_flags(**kw)) as plan:
            plan.rs_fold(out, alpha=0.5)
            torch.cuda.synchronize()
            assert plan.device_status() == tide.TIDE_OK
        n = full_rs_check(world, dims, gs.views, None, out, 0.5, False, what=f"2G+ {kw}", order=oname)
        assert n == world * S
    del out
    torch.cuda.empty_cache()
    slots = workloads.make_slots(w, S, device="cuda")
    full = [torch.empty(s_, dtype=torch.bfloat16, device="cuda") for s_ in w.shapes]
    with tide.Plan(gs.views) as plan:
        bound = plan.bind_full(full)
        for mode in ("sm", "ce2d", "ce1d"):
            for f in full:
                f.fill_(float("nan"))
            plan.ag_place(slots, bound, mode=mode)
            torch.cuda.synchronize()
            for p, (d, k) in enumerate(dims):
                flat = full[p].reshape(-1).view(torch.int16)
                for r in range(world):
                    v = oracle.valid_rows(d, R[p], r) * k
                    got = flat[r * R[p] * k:r * R[p] * k + v]
                    ref = slots[r, o[p]:o[p] + v].view(torch.int16)
                    assert torch.equal(got, ref), (mode, p, r)
    del gs, full, slots
    torch.cuda.empty_cache()


@pytest.mark.parametrize("index", [2, 5])
def test_full_size_orders_and_fp32(index):
    """Full-size groups: the Section 4.3 orders, the tree order and fp32
    gradients, every output element recomputed by the oracle in the same order,
    and each order within 1e-6 of the rank-order fold in the max-norm over
    every parameter tensor (the reordered-variant tolerance)."""
    w = workloads.get(index)
    dims = w.dim0_rownumel()
    gs = workloads.make_grads(w, device="cuda")
    _, _, S = oracle.geometry(w.world, dims)
    L = w.world // 2
    R, o, _ = oracle.geometry(w.world, dims)
    rank_out = torch.empty(w.world, S, device="cuda")
    with tide.Plan(gs.views) as plan:
        plan.rs_fold(rank_out, alpha=w.alpha)
        torch.cuda.synchronize()
    for order, oname, ns in ((tide.TIDE_ORDER_STAGED_OWN, "staged", 0), (tide.TIDE_ORDER_NODES, "nodes", L),
                             (tide.TIDE_ORDER_TREE, "tree", 0)):
        out = torch.full((w.world, S), float("nan"), device="cuda")
        with tide.Plan(gs.views, tide.make_flags(order=order, node_size=ns)) as plan:
            plan.rs_fold(out, alpha=w.alpha)
            torch.cuda.synchronize()
            assert plan.device_status() == tide.TIDE_OK
        n = full_rs_check(w.world, dims, gs.views, None, out, w.alpha, False, what=f"{w.name} {oname}",
                          order=oname, node_size=ns)
        assert n == w.world * S
        # the reordered-variant tolerance against rank order, max-norm over each parameter tensor
        for p, (d, k) in enumerate(dims):
            a = out[:, o[p]:o[p] + R[p] * k].double()
            b = rank_out[:, o[p]:o[p] + R[p] * k].double()
            assert float((a - b).abs().max()) <= 1e-6 * float(b.abs().max()), f"{w.name} {oname} p={p}"
        del out
    del rank_out
    # fp32 gradients (the bf16 values plus a small fp32 perturbation), accumulate mode
    views32 = [[v.float() + 1e-6 * torch.randn(v.shape, device="cuda") for v in vs] for vs in gs.views]
    del gs
    out = workloads.make_out_init(w, S, device="cuda")
    before = out.clone()
    with tide.Plan(views32, tide.make_flags(grad_dtype=tide.TIDE_DTYPE_F32)) as plan:
        plan.rs_fold(out, alpha=1.0 / w.world, accumulate=True)
        torch.cuda.synchronize()
        assert plan.device_status() == tide.TIDE_OK
    n = full_rs_check(w.world, dims, views32, before, out, 1.0 / w.world, True, what=f"{w.name} fp32 grads")
    assert n == w.world * S
    del views32, out, before
    torch.cuda.empty_cache()
