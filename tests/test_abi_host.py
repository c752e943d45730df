"""Host logic of the C-ABI library, no GPU needed: the library loads and
exports every symbol include/tide.h declares; host-only plans reproduce the
oracle's shard geometry (Section 2.1) and tile each slot exactly; argument
validation returns the documented status codes without touching the device."""
import os
import random
import re

import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tide():
    from all_gather_gb300 import build
    build.build()
    import all_gather_gb300
    all_gather_gb300.load_library()
    return all_gather_gb300


def _fake_ptrs(W, P, numels, align=256, base=0x7F0000000000):
    """Distinct, non-overlapping fake device addresses [p][u]."""
    ptrs, cur = [], base
    for p in range(P):
        row = []
        for u in range(W):
            row.append(cur)
            cur += (max(numels[p], 1) * 2 + align - 1) // align * align + align
        ptrs.append(row)
    return ptrs, cur


def _host_plan(tide, W, dims, ptrs=None, offsets=None, **flag_kw):
    numels = [d * k for d, k in dims]
    if ptrs is None:
        ptrs, _ = _fake_ptrs(W, len(dims), numels)
    params = [(ptrs[p], d, k, -1 if offsets is None else offsets[p]) for p, (d, k) in enumerate(dims)]
    flags = tide.make_flags(debug=tide.TIDE_DEBUG_HOST_ONLY, **flag_kw)
    return tide.tide_plan_build(W, params, flags, 0)


def test_exports_match_header(tide):
    with open(os.path.join(ROOT, "include", "tide.h")) as f:
        declared = set(re.findall(r"TIDE_API[^;(]*?\b(tide_\w+)\s*\(", f.read()))
    assert declared == set(tide.EXPORTED), declared ^ set(tide.EXPORTED)
    lib = tide.load_library()
    for name in declared:
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(tide):
    for code, name in [(0, "TIDE_OK"), (1, "TIDE_ERR_INVALID_ARG"), (2, "TIDE_ERR_ALIGNMENT"),
                       (3, "TIDE_ERR_UNSUPPORTED"), (4, "TIDE_ERR_OOM"), (5, "TIDE_ERR_CUDA"),
                       (6, "TIDE_ERR_TIMEOUT")]:
        assert tide.tide_status_string(code) == name


def _check_geometry(tide, W, dims):
    plan = _host_plan(tide, W, dims)
    try:
        R, o, S = oracle.geometry(W, dims)
        assert tide.tide_plan_slot_numel(plan) == S
        segs = [tide.tide_plan_segment(plan, i) for i in range(tide.tide_plan_num_segments(plan))]
        assert len(segs) == W * len(dims)
        covered = [[0] * S for _ in range(W)] if S * W <= 200_000 else None
        pad_total = 0
        for s in segs:
            p, r = s["param"], s["rank"]
            d, k = dims[p]
            v = oracle.valid_rows(d, R[p], r)
            assert s["src_elem"] == r * R[p] * k
            assert s["dst_elem"] == o[p]
            assert (s["n_valid"], s["n_pad"]) == (v * k, (R[p] - v) * k)
            pad_total += s["n_pad"]
            if covered is not None:
                for j in range(s["n_valid"] + s["n_pad"]):
                    covered[r][o[p] + j] += 1
        assert pad_total == W * S - sum(d * k for d, k in dims)
        if covered is not None:
            assert all(c == 1 for row in covered for c in row), "pieces must tile every slot exactly once"
        cfg = tide.tide_plan_fold_config(plan)
        ch = cfg["chunk_elems"]
        want_items = sum(-(-s["n_valid"] // ch) + -(-s["n_pad"] // ch) for s in segs)
        assert cfg["items"] == want_items
    finally:
        tide.tide_plan_destroy(plan)


@pytest.mark.parametrize("w", workloads.WORKLOADS, ids=[w.name for w in workloads.WORKLOADS])
def test_geometry_matches_oracle_workloads(tide, w):
    _check_geometry(tide, w.world, w.dim0_rownumel())


def test_geometry_matches_oracle_random(tide):
    rnd = random.Random(1)
    for _ in range(60):
        W = rnd.choice([1, 2, 3, 4, 5, 7, 8, 16, 32, 33])
        dims = [(rnd.choice([0, 1, 2, W - 1 or 1, W, W + 1, 3 * W + 2, 100]), rnd.choice([0, 1, 3, 8, 17]))
                for _ in range(rnd.randint(0, 6))]
        _check_geometry(tide, W, dims)


def test_explicit_offsets(tide):
    dims = [(10, 4), (3, 3)]
    plan = _host_plan(tide, 2, dims, offsets=[64, 0])
    try:
        assert tide.tide_plan_slot_numel(plan) == 64 + 5 * 4
        seg = tide.tide_plan_segment(plan, 0)
        assert seg["dst_elem"] == 64
    finally:
        tide.tide_plan_destroy(plan)
    with pytest.raises(tide.TideError) as e:
        _host_plan(tide, 2, dims, offsets=[0, 10])  # [0, 20) and [10, 16) overlap
    assert e.value.status == tide.TIDE_ERR_INVALID_ARG


def test_empty_group(tide):
    plan = _host_plan(tide, 4, [])
    try:
        assert tide.tide_plan_slot_numel(plan) == 0
        assert tide.tide_plan_fold_config(plan)["items"] == 0
    finally:
        tide.tide_plan_destroy(plan)


@pytest.mark.parametrize("case, status", [
    ("world0", "TIDE_ERR_INVALID_ARG"), ("world_big", "TIDE_ERR_INVALID_ARG"),
    ("neg_dim", "TIDE_ERR_INVALID_ARG"), ("null_ptr", "TIDE_ERR_INVALID_ARG"),
    ("odd_ptr", "TIDE_ERR_ALIGNMENT"), ("reserved", "TIDE_ERR_INVALID_ARG"),
    ("chunk", "TIDE_ERR_INVALID_ARG"), ("order", "TIDE_ERR_UNSUPPORTED"),
    ("dtype", "TIDE_ERR_UNSUPPORTED"), ("overflow", "TIDE_ERR_INVALID_ARG"),
    ("neg_offset", "TIDE_ERR_INVALID_ARG"), ("sched", "TIDE_ERR_INVALID_ARG"),
    ("fill", "TIDE_ERR_INVALID_ARG"), ("nodes_direct", "TIDE_ERR_UNSUPPORTED"),
    ("skip_fill_direct", "TIDE_ERR_INVALID_ARG"), ("debug_bits", "TIDE_ERR_INVALID_ARG"),
    ("node_size_not_dividing", "TIDE_ERR_INVALID_ARG"), ("node_size_without_nodes", "TIDE_ERR_INVALID_ARG"),
    ("nodes_without_size", "TIDE_ERR_INVALID_ARG"), ("staged_direct", "TIDE_ERR_UNSUPPORTED"),
    ("f32_direct", "TIDE_ERR_UNSUPPORTED"), ("f32_misaligned", "TIDE_ERR_ALIGNMENT"),
    ("ce_streams", "TIDE_ERR_INVALID_ARG"), ("tree_direct", "TIDE_ERR_UNSUPPORTED"),
    ("tree_node_size", "TIDE_ERR_INVALID_ARG"), ("tree_direct_dynamic", "TIDE_ERR_UNSUPPORTED"),
    ("per_item_budget", "TIDE_ERR_INVALID_ARG"),
])
def test_build_validation(tide, case, status):
    W, dims = 4, [(8, 8), (5, 1)]
    ptrs, _ = _fake_ptrs(W, 2, [64, 5])
    kw = {}
    offsets = None
    world = W
    if case == "world0":
        world = 0
    elif case == "world_big":
        world = 1025
        ptrs = [[0x10000] * 1025, [0x20000] * 1025]
    elif case == "neg_dim":
        dims = [(-1, 8), (5, 1)]
    elif case == "null_ptr":
        ptrs[1][2] = 0
    elif case == "odd_ptr":
        ptrs[0][3] += 1
    elif case == "chunk":
        kw["chunk_bytes"] = 300
    elif case == "order":
        kw["order"] = 7
    elif case == "dtype":
        kw["grad_dtype"] = 7
    elif case == "overflow":
        dims = [(1 << 40, 1 << 30), (5, 1)]
    elif case == "neg_offset":
        offsets = [-2, -1]
    elif case == "sched":
        kw["sched"] = 9
    elif case == "fill":
        kw["fill_bytes"] = 24
    elif case == "nodes_direct":
        kw.update(order=tide.TIDE_ORDER_NODES, node_size=2, kernel=tide.TIDE_KERNEL_DIRECT)
    elif case == "skip_fill_direct":
        kw.update(kernel=tide.TIDE_KERNEL_DIRECT)
    elif case == "node_size_not_dividing":
        kw.update(order=tide.TIDE_ORDER_NODES, node_size=3)
    elif case == "node_size_without_nodes":
        kw.update(node_size=2)
    elif case == "nodes_without_size":
        kw.update(order=tide.TIDE_ORDER_NODES)
    elif case == "staged_direct":
        kw.update(order=tide.TIDE_ORDER_STAGED_OWN, kernel=tide.TIDE_KERNEL_DIRECT)
    elif case == "f32_direct":
        kw.update(grad_dtype=tide.TIDE_DTYPE_F32, kernel=tide.TIDE_KERNEL_DIRECT, sched=tide.TIDE_SCHED_DYNAMIC)
    elif case == "ce_streams":
        kw.update(ce_streams=9)
    elif case == "tree_direct":
        kw.update(order=tide.TIDE_ORDER_TREE, kernel=tide.TIDE_KERNEL_DIRECT)
    elif case == "tree_node_size":
        kw.update(order=tide.TIDE_ORDER_TREE, node_size=2)
    elif case == "tree_direct_dynamic":
        kw.update(order=tide.TIDE_ORDER_TREE, kernel=tide.TIDE_KERNEL_DIRECT, sched=tide.TIDE_SCHED_DYNAMIC)
    elif case == "per_item_budget":
        kw.update(sched=tide.TIDE_SCHED_PER_ITEM, cta_budget=16)
    elif case == "f32_misaligned":
        kw.update(grad_dtype=tide.TIDE_DTYPE_F32)
        ptrs[1][1] += 2
    flags_debug = tide.TIDE_DEBUG_HOST_ONLY
    if case == "skip_fill_direct":
        flags_debug |= tide.TIDE_DEBUG_SKIP_FILL
    if case == "debug_bits":
        flags_debug |= 0x100
    flags = tide.make_flags(debug=flags_debug, **kw)
    if case == "reserved":
        flags.reserved[0] = 1
    params = [(ptrs[p], d, k, -1 if offsets is None else offsets[p]) for p, (d, k) in enumerate(dims)]
    with pytest.raises(tide.TideError) as e:
        tide.tide_plan_build(world, params, flags, 0)
    assert tide.tide_status_string(e.value.status) == status, str(e.value)
    assert e.value.detail, "a failing call must leave a detail message"


def test_tree_order_fill_limit(tide):
    """The tree order keeps one partial per level of full stage fills in
    registers: at most 255 full fills per chunk (W / fill_ranks, the fill
    ranks rounded down to a power of two, at most 8)."""
    W = 1024
    dims = [(W, 1)]
    for fill_ranks, ok in ((0, True), (8, True), (16, True), (5, False), (4, False), (1, False)):
        if ok:
            tide.tide_plan_destroy(_host_plan(tide, W, dims, order=tide.TIDE_ORDER_TREE, fill_ranks=fill_ranks))
        else:
            with pytest.raises(tide.TideError) as e:
                _host_plan(tide, W, dims, order=tide.TIDE_ORDER_TREE, fill_ranks=fill_ranks)
            assert e.value.status == tide.TIDE_ERR_INVALID_ARG, fill_ranks
    tide.tide_plan_destroy(_host_plan(tide, 1020, [(1020, 1)], order=tide.TIDE_ORDER_TREE, fill_ranks=4))


def test_per_item_schedule_grid(tide):
    """TIDE_SCHED_PER_ITEM: the fold's grid is its work list, one CTA per item."""
    plan = _host_plan(tide, 8, [(4096, 4096), (1024, 4096), (4096, 1)], sched=tide.TIDE_SCHED_PER_ITEM)
    try:
        cfg = tide.tide_plan_fold_config(plan)
        assert cfg["grid"] == cfg["items"] > 1000
    finally:
        tide.tide_plan_destroy(plan)


def test_host_only_plan_cannot_launch(tide):
    plan = _host_plan(tide, 2, [(4, 4)])
    try:
        with pytest.raises(tide.TideError) as e:
            tide.tide_rs_fold(plan, 0x1000, 100, 1.0, 0, 0)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        with pytest.raises(tide.TideError) as e:
            tide.tide_ag_place(plan, 0x1000, 100, [0x2000], tide.TIDE_AG_SM, 0)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
    finally:
        tide.tide_plan_destroy(plan)


def test_rebind_checks_geometry(tide):
    W, dims = 2, [(4, 4), (3, 1)]
    plan = _host_plan(tide, W, dims)
    try:
        ptrs, _ = _fake_ptrs(W, 2, [16, 3], base=0x6F0000000000)
        tide.tide_plan_rebind(plan, [(ptrs[0], 4, 4, -1), (ptrs[1], 3, 1, -1)], 0)
        with pytest.raises(tide.TideError):
            tide.tide_plan_rebind(plan, [(ptrs[0], 5, 4, -1), (ptrs[1], 3, 1, -1)], 0)
        bad = [list(ptrs[0]), list(ptrs[1])]
        bad[0][1] += 1
        with pytest.raises(tide.TideError) as e:
            tide.tide_plan_rebind(plan, [(bad[0], 4, 4, -1), (bad[1], 3, 1, -1)], 0)
        assert e.value.status == tide.TIDE_ERR_ALIGNMENT
    finally:
        tide.tide_plan_destroy(plan)


def test_bound_full_tensors_are_checked_once(tide):
    """bind_full checks the full tensors' dtype, contiguity and shapes once and
    keeps their pointers; a mismatched list is refused before any call."""
    import torch
    shapes = [(8, 3), (5,)]
    plan = tide.Plan([[torch.zeros(s_, dtype=torch.bfloat16) for s_ in shapes] for _ in range(2)], host_only=True)
    try:
        full = [torch.empty(s_, dtype=torch.bfloat16) for s_ in shapes]
        bound = plan.bind_full(full)
        assert [bound.ptrs[i] for i in range(2)] == [f.data_ptr() for f in full]
        for bad in ([full[0]], [full[0], torch.empty(6, dtype=torch.bfloat16)],
                    [full[0].float(), full[1]], [torch.empty(3, 8, dtype=torch.bfloat16).t(), full[1]]):
            with pytest.raises(ValueError):
                plan.bind_full(bad)
    finally:
        plan.close()


def test_launch_count_starts_at_zero_without_gpu(tide):
    import torch
    if torch.cuda.is_available():
        pytest.skip("only meaningful before any GPU work")
    assert tide.tide_launch_count() == 0


def test_corun_cta_budget(tide):
    """Section 2.2, Equation (4): (n_slot - n_gemm) * cluster CTAs keep the
    GEMM in one wave; worked values, and the documented edge cases."""
    f = tide.tide_corun_cta_budget
    assert f(36, 128, 4) == 16      # GB300: 36 slots, 32 four-CTA clusters
    assert f(33, 128, 4) == 4       # the paper's GPU: one spare slot
    assert f(32, 128, 4) == 0       # no spare slot
    assert f(20, 128, 4) == 0
    assert f(36, 129, 4) == 12      # a partial 33rd cluster takes a slot too
    assert f(10, 3, 1) == 7
    assert f(1, 16, 16) == 0 and f(2, 16, 16) == 16 and f(8, 8, 16) == 7 * 16
    for bad in ((0, 128, 4), (36, 0, 4), (36, 128, 0), (36, 128, 17), (-1, 1, 1)):
        assert f(*bad) == -1, bad


@pytest.mark.parametrize("order", [0, 1, 2, 3])
@pytest.mark.parametrize("dtype", [0, 1])
def test_bulk_kernel_schedules_dynamically(tide, order, dtype):
    """The bulk kernel claims work items dynamically in every order and for
    both gradient types; the default kernel is the bulk kernel."""
    W, dims = 4, [(8, 8), (5, 1)]
    plan = _host_plan(tide, W, dims, sched=tide.TIDE_SCHED_DYNAMIC, order=order, grad_dtype=dtype,
                      node_size=2 if order == tide.TIDE_ORDER_NODES else 0)
    tide.tide_plan_destroy(plan)
