"""Helpers for the GPU parity tests: host copies, oracle runs and the
every-element full-size check."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Sequence

import numpy as np
import torch

import oracle
from bits import assert_same_f32


def bits16(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor (any device) as a flat host uint16 array."""
    return t.detach().reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_rs_full(world: int, dims, grads_uv: Sequence[Sequence[torch.Tensor]], alpha: float, accumulate: bool,
                   out_before: torch.Tensor) -> np.ndarray:
    """Run the oracle over everything (small cases).  grads_uv[u][p]."""
    host = [[bits16(grads_uv[u][p]) for u in range(world)] for p in range(len(dims))]
    want = out_before.detach().cpu().numpy().astype(np.float32, copy=True)
    oracle.rs(world, dims, host, alpha, accumulate, want)
    return want


def full_rs_check(world: int, dims, grads_uv, out_before, out_after: torch.Tensor, alpha: float,
                  accumulate: bool, what: str = "", window: int = 1 << 20, order: str = "rank",
                  node_size: int = 0) -> int:
    """Compare EVERY output element of a fold with the oracle, one parameter at
    a time (host memory stays at one parameter's W gradients): the W gradient
    tensors and the W output windows come to the host, the unchanged oracle
    (oracle.rs_window, Eq. (3) + (5); rs_window_ex for another order or fp32
    gradients) recomputes each (rank, window of at most `window` elements) on
    all host cores, and the two are compared bit for bit.  Returns the number
    of elements compared (W * S for prefix offsets)."""
    orc = oracle.load()
    R, o, S = orc.geometry(world, dims)
    threads = max(1, len(os.sched_getaffinity(0)))
    checked = 0
    with ThreadPoolExecutor(max_workers=threads) as pool:
        for p, (d, k) in enumerate(dims):
            n = R[p] * k
            if n == 0:
                continue
            f32 = grads_uv[0][p].dtype == torch.float32
            host = [grads_uv[u][p].detach().reshape(-1).cpu().numpy() if f32 else bits16(grads_uv[u][p])
                    for u in range(world)]
            got = out_after[:, o[p]:o[p] + n].cpu().numpy()
            old = out_before[:, o[p]:o[p] + n].cpu().numpy() if accumulate else None
            want = np.empty((world, n), dtype=np.float32)
            jobs = []
            for r in range(world):
                v = orc.valid_rows(d, R[p], r) * k
                for a in range(0, n, window):
                    b = min(a + window, n)
                    jobs.append((r, a, b, max(0, min(b, v) - a)))

            def run(job):
                r, a, b, nv = job
                srcs = [h[r * n + a:r * n + a + nv] for h in host]
                o_win = old[r, a:b] if accumulate else None
                if order == "rank" and not f32:
                    want[r, a:b] = orc.rs_window(srcs, nv, (b - a) - nv, alpha, accumulate, o_win)
                else:
                    want[r, a:b] = orc.rs_window_ex(srcs, nv, (b - a) - nv, alpha, accumulate, r, order,
                                                    node_size, o_win)

            list(pool.map(run, jobs))
            if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
                assert_same_f32(got, want, f"{what} p={p} (every element)")  # NaN classes match
            checked += world * n
    return checked


def ag_expected(world: int, dims, slots: torch.Tensor) -> List[np.ndarray]:
    return oracle.ag(world, dims, bits16(slots).reshape(world, -1))


def sentinel_slots(world: int, dims, stride: int, seed: int, device="cuda") -> torch.Tensor:
    """bf16 [W, stride] slots: random real rows, NaN sentinel (0x7FC1) in padding
    and past S, so that any padding read shows up in the output."""
    R, o, S = oracle.geometry(world, dims)
    g = torch.Generator(device="cpu").manual_seed(seed)
    vals = torch.randint(0, 0x7F00, (world, stride), generator=g, dtype=torch.int32).to(torch.int16)
    mask = np.ones((world, stride), dtype=bool)
    for p, (d, k) in enumerate(dims):
        for r in range(world):
            v = oracle.valid_rows(d, R[p], r)
            mask[r, o[p]:o[p] + v * k] = False
    vals[torch.from_numpy(mask)] = 0x7FC1
    return vals.view(torch.bfloat16).to(device)
