"""The full-size comparator of the GPU parity tests, exercised on the CPU.

gpu_helpers.full_rs_check must compare every output element: run on CPU
tensors it accepts the oracle's own result and rejects it after one element
(of a padding row, then of a real row) is changed by one ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import bits16, full_rs_check


@pytest.mark.parametrize("acc", [False, True])
def test_full_rs_check_compares_every_element(acc):
    w = workloads.custom(3, [(10, 7), (5,), (33, 8)], index=401)
    dims = w.dim0_rownumel()
    R, o, S = oracle.geometry(w.world, dims)
    gs = workloads.make_grads(w, device="cpu")
    before = torch.randn(w.world, S) if acc else None
    want = before.numpy().copy() if acc else np.zeros((w.world, S), np.float32)
    host = [[bits16(gs.views[u][p]) for u in range(w.world)] for p in range(len(dims))]
    oracle.rs(w.world, dims, host, 0.5, acc, want)
    out = torch.from_numpy(want.copy())
    assert full_rs_check(w.world, dims, gs.views, before, out, 0.5, acc, window=4) == w.world * S
    for r, j in ((w.world - 1, o[0] + R[0] * 7 - 1), (1, o[2] + 3)):  # a padding element, a real one
        bad = out.clone()
        bad[r, j] = float(np.nextafter(np.float32(bad[r, j]), np.float32(np.inf)))
        with pytest.raises(AssertionError):
            full_rs_check(w.world, dims, gs.views, before, bad, 0.5, acc, window=4)


@pytest.mark.parametrize("order,node_size,f32", [("tree", 0, False), ("nodes", 2, False), ("rank", 0, True)])
def test_full_rs_check_other_orders_and_fp32(order, node_size, f32):
    w = workloads.custom(4, [(10, 7), (5,), (33, 8)], index=402)
    dims = w.dim0_rownumel()
    R, o, S = oracle.geometry(w.world, dims)
    gs = workloads.make_grads(w, device="cpu")
    views = [[v.float() + 1e-6 * torch.randn(v.shape) for v in vs] for vs in gs.views] if f32 else gs.views
    host = [[(views[u][p].reshape(-1).numpy() if f32 else bits16(views[u][p])) for u in range(w.world)]
            for p in range(len(dims))]
    want = np.zeros((w.world, S), np.float32)
    oracle.rs_ex(w.world, dims, host, 0.5, False, want, order, node_size)
    out = torch.from_numpy(want.copy())
    assert full_rs_check(w.world, dims, views, None, out, 0.5, False, window=5, order=order,
                         node_size=node_size) == w.world * S
    bad = out.clone()
    bad[2, o[2] + 1] = float(np.nextafter(np.float32(bad[2, o[2] + 1]), np.float32(np.inf)))
    with pytest.raises(AssertionError):
        full_rs_check(w.world, dims, views, None, bad, 0.5, False, window=5, order=order, node_size=node_size)
