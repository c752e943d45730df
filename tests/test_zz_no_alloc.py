"""The allocation-free fold (tide_rs_fold_noalloc) against the plan-based one.

Some callers cannot allocate GPU memory (code running inside an allocator or
an out-of-memory handler, under a pool or cap that forbids new device
allocations), so they cannot build a plan, whose device tables come from
cudaMalloc.  tide_rs_fold_noalloc serves them from a fixed device array owned
by the library.  This test calls it through the C ABI twice in a row, with
different groups, and checks that each result equals the plan-based
tide_rs_fold's bit for bit (the same tolerance as every fold parity test:
none).  It also checks that an oversized request is refused.  The file sorts
last so that a run stopping at the first failure has run everything else.
"""
import pytest
import torch

import all_gather_gb300 as tide
import workloads
from bits import assert_same_f32

pytestmark = pytest.mark.gpu


def _descs(grads_uv):
    W, P = len(grads_uv), len(grads_uv[0])
    out = []
    for p in range(P):
        t = grads_uv[0][p]
        d0 = t.shape[0]
        out.append(([grads_uv[u][p].data_ptr() for u in range(W)], d0, t.numel() // d0 if d0 else 0, -1))
    return out


def _both(w, gs, alpha, accumulate, stride_extra=0):
    """(plan-based result, allocation-free result) on identical inputs."""
    init = None
    with tide.Plan(gs.views) as plan:
        S = plan.slot_numel
        stride = S + stride_extra
        if accumulate:
            init = torch.randn(w.world, stride, device="cuda")
        ref = init.clone() if accumulate else torch.zeros(w.world, stride, device="cuda")
        plan.rs_fold(ref, alpha=alpha, accumulate=accumulate)
    got = init.clone() if accumulate else torch.full((w.world, stride), 7.0, device="cuda")
    if not accumulate:
        got[:, :S] = -1.0  # every element up to S must be overwritten
        ref[:, S:] = 7.0
    tide.tide_rs_fold_noalloc(w.world, _descs(gs.views), got.data_ptr(), stride, alpha, int(accumulate),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_matches_plan_fold_two_calls_in_a_row():
    torch.cuda.set_device(0)
    # call 1: the toy group (W = 4, ragged shapes, padding, scale 1/W)
    w1 = workloads.get(1)
    g1 = workloads.make_grads(w1, device="cuda")
    ref1, got1 = _both(w1, g1, w1.alpha, False, stride_extra=3)
    assert_same_f32(got1.cpu().numpy(), ref1.cpu().numpy(), "allocation-free fold, call 1")
    # call 2, straight after: a different group (W = 8) in accumulate mode
    w2 = workloads.custom(8, [(1000, 33), (17,), (4096, 64), (5, 3)], index=123)
    g2 = workloads.make_grads(w2, device="cuda")
    ref2, got2 = _both(w2, g2, 0.5, True)
    assert_same_f32(got2.cpu().numpy(), ref2.cpu().numpy(), "allocation-free fold, call 2")


def test_noalloc_rejects_tables_beyond_its_array():
    # 9,000 parameters x 64 ranks = 576,000 pieces: far more table bytes than
    # the fixed array holds; refused on the host before any GPU work.
    W, P = 64, 9000
    fake = [([0x7F0000000000 + 256 * (p * W + u) for u in range(W)], 64, 1, -1) for p in range(P)]
    with pytest.raises(tide.TideError) as e:
        tide.tide_rs_fold_noalloc(W, fake, 0x7E0000000000, 10**6, 1.0, 0, 0)
    assert e.value.status == tide.TIDE_ERR_INVALID_ARG
    assert "bytes of tables" in e.value.detail
