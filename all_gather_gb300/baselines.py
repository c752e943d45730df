"""Stock-FSDP2-style two-pass baselines, for comparison only (never on the
product path).

Reduce-scatter: the TIDE paper (Section 2.1, Equation (3)) describes stock
FSDP2 packing every rank's gradients with torch._chunk_cat (slice, zero-pad,
upcast, pack) into a transient fp32 rank-major buffer, then reducing that
buffer with a reduce-scatter.  With the W ranks virtual, the pack is W
_chunk_cat calls into a [W, W*S] fp32 buffer and the reduction a sum over the
source axis, then the scale (and the += of gradient accumulation).

All-gather: stock FSDP2 copies the rank-major all-gather output into padded
per-parameter storage with split_with_sizes_copy (Section 2.1).
"""
from __future__ import annotations

from typing import List, Sequence

import torch


def two_pass_rs(grads_uv: Sequence[Sequence[torch.Tensor]], pack: torch.Tensor, out: torch.Tensor, alpha: float,
                accumulate: bool) -> torch.Tensor:
    W, S = out.shape[0], out.shape[1]
    for u in range(W):
        torch._chunk_cat(list(grads_uv[u]), dim=0, num_chunks=W, out=pack[u].view(W, S))
    red = pack.sum(dim=0).view(W, S)
    if accumulate:
        out.add_(red, alpha=alpha)
    else:
        torch.mul(red, alpha, out=out)
    return out


def copy_out_ag(slots: torch.Tensor, padded: List[torch.Tensor], sizes: List[int]) -> List[torch.Tensor]:
    W = slots.shape[0]
    torch.split_with_sizes_copy(slots, sizes, dim=1, out=[p.view(W, -1) for p in padded])
    return padded


def time_two_pass(w, grads_uv, S: int, out: torch.Tensor, slots: torch.Tensor, full, steps: int = 10) -> dict:
    dev = out.device
    W = w.world
    dims = w.dim0_rownumel()
    sizes = [-(-d // W) * k for d, k in dims]
    pack = torch.empty(W, W * S, dtype=torch.float32, device=dev)
    out_b = out.clone()
    padded = [torch.empty(W * n, dtype=torch.bfloat16, device=dev) for n in sizes]
    stream = torch.cuda.current_stream()
    for _ in range(3):
        two_pass_rs(grads_uv, pack, out_b, w.alpha, w.accumulate)
        copy_out_ag(slots[:, :S], padded, sizes)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        torch.cuda.nvtx.range_push("two_pass_rs")  # lets a profiler select exactly these kernels
        two_pass_rs(grads_uv, pack, out_b, w.alpha, w.accumulate)
        torch.cuda.nvtx.range_pop()
        ev[i][1].record(stream)
        copy_out_ag(slots[:, :S], padded, sizes)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    rs_ms = sorted(e[0].elapsed_time(e[1]) for e in ev)[steps // 2]
    ag_ms = sorted(e[1].elapsed_time(e[2]) for e in ev)[steps // 2]
    numel = w.total_numel()
    rs_b = W * numel * 2 + numel * 4 + (numel * 4 if w.accumulate else 0)
    ag_b = 4 * numel
    res = {"rs_ms": round(rs_ms, 4), "rs_gbs": round(rs_b / (rs_ms * 1e-3) / 1e9, 1), "ag_ms": round(ag_ms, 4),
           "ag_gbs": round(ag_b / (ag_ms * 1e-3) / 1e9, 1), "pack_buffer_bytes": pack.numel() * 4,
           "fused_extra_buffer_bytes": 0, "steps": steps, "stat": "median",
           "what": "torch._chunk_cat fp32 pack per virtual rank + sum over ranks + scale; split_with_sizes_copy"}
    del pack, out_b, padded
    torch.cuda.empty_cache()
    return res
