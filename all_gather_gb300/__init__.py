"""GB300-native layout-folded reduce-scatter and all-gather placement for FSDP2.

Implements the data-parallel hot path of TIDE ("The Endgame of FSDP
Communication"): per-parameter bf16 gradients of W (virtual) ranks are read
in place and summed in fp32, in rank order, into each rank's padded dim-0
shard (Section 4, Equation (5)); rank-major bf16 shard slots are placed
straight into per-parameter full tensors (Section 2.1, Equation (2)).

Everything runs in libtide.so (hand-written sm_103a kernels behind a C ABI,
``include/tide.h``).  This package only marshals arguments: the ``tide_*``
functions mirror the C entry points one to one, and :class:`Plan` is a thin
convenience wrapper that takes torch tensors and passes their pointers.
torch is used for device memory and streams only.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

from ._binding import (  # noqa: F401  (re-exported C-ABI names)
    EXPORTED, LIB_PATH, TIDE_AG_CE_1D, TIDE_AG_CE_2D, TIDE_AG_SM, TIDE_DEBUG_HOST_ONLY, TIDE_DEBUG_SHORT_WAIT,
    TIDE_DEBUG_SKIP_FILL, TIDE_DTYPE_BF16,
    TIDE_ERR_ALIGNMENT, TIDE_ERR_CUDA, TIDE_ERR_INVALID_ARG, TIDE_ERR_OOM, TIDE_ERR_TIMEOUT, TIDE_ERR_UNSUPPORTED,
    TIDE_KERNEL_AUTO, TIDE_KERNEL_BULK, TIDE_KERNEL_DIRECT, TIDE_OK, TIDE_ORDER_NODES, TIDE_ORDER_RANK_ASC,
    TIDE_ORDER_STAGED_OWN, TIDE_ORDER_TREE, TIDE_DTYPE_F32, TIDE_SCHED_DYNAMIC,
    TIDE_SCHED_AUTO, TIDE_SCHED_STATIC, TIDE_SCHED_PER_ITEM, PlanFlags, TideError, load_library, make_flags, tide_ag_place, tide_ag_place_f32,
    tide_last_device_status,
    tide_last_error, tide_launch_count, tide_plan_build, tide_plan_destroy, tide_plan_fold_config,
    tide_plan_num_segments, tide_plan_rebind, tide_plan_segment, tide_plan_slot_numel, tide_rs_fold,
    tide_rs_fold_noalloc, tide_status_string, tide_latin_square_gpu, tide_rs_wave_plan, tide_rs_wave_zero_mask,
    tide_bruck_schedule, tide_sm_probe, tide_sm_probe_max_clusters, tide_corun_cta_budget, pointer_array)

AG_MODES = {"sm": TIDE_AG_SM, "ce2d": TIDE_AG_CE_2D, "ce1d": TIDE_AG_CE_1D}


def _stream_handle(stream) -> int:
    """cudaStream_t of `stream` (a torch stream or a raw handle); None = the
    current stream of the current device (read through torch's raw accessor
    when it has one: a fraction of the cost of building a Stream object, which
    matters for groups small enough to be bound by the host's enqueue)."""
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch._C._cuda_getDevice())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _param_descs(grads, offsets=None, require_cuda=True, dtype=None):
    """grads[u][p] tensors -> descriptor tuples (pointers [W], dim0, row_numel, offset)."""
    import torch
    dtype = dtype or torch.bfloat16
    W = len(grads)
    if W < 1:
        raise ValueError("need at least one rank")
    P = len(grads[0])
    descs = []
    for p in range(P):
        t0 = grads[0][p]
        if t0.dim() == 0:
            raise ValueError(f"parameter {p} is 0-d; FSDP2 shards along dim 0")
        ptrs = []
        for u in range(W):
            t = grads[u][p]
            if t.dtype != dtype:
                raise TypeError(f"gradient [{u}][{p}] is {t.dtype}, expected {dtype}")
            if t.shape != t0.shape:
                raise ValueError(f"gradient [{u}][{p}] shape {tuple(t.shape)} != rank 0's {tuple(t0.shape)}")
            if not t.is_contiguous():
                raise ValueError(f"gradient [{u}][{p}] is not contiguous")
            if require_cuda and t.numel() and not (t.is_cuda or t.is_pinned()):
                raise ValueError(f"gradient [{u}][{p}] is neither on a CUDA device nor in page-locked host memory")
            ptrs.append(t.data_ptr())
        d0 = t0.shape[0]
        k = t0.numel() // d0 if d0 else int(torch.Size(t0.shape[1:]).numel())
        descs.append((ptrs, d0, k, -1 if offsets is None else offsets[p]))
    return descs


class FullParams:
    """The P full parameter tensors of a group, checked once and kept as the
    pointer array the placements take (the paper registers the group's
    tables once instead of building them per call, Section 6).  Holds
    references to the tensors, so the pointers stay valid while it lives."""

    def __init__(self, full: Sequence, shapes: Sequence[tuple]):
        import torch
        if len(full) != len(shapes):
            raise ValueError(f"{len(full)} full tensors for {len(shapes)} parameters")
        for p, f in enumerate(full):
            if f.dtype != torch.bfloat16 or not f.is_contiguous() or tuple(f.shape) != shapes[p]:
                raise ValueError(f"full[{p}] must be a contiguous bfloat16 tensor of shape {shapes[p]}")
        self.tensors = list(full)
        self.ptrs = pointer_array([f.data_ptr() for f in full])


class Plan:
    """A built plan for one parameter group (owns the plan's device tables).

    ``grads[u][p]``: bf16 gradient of parameter p on virtual rank u (CUDA or
    page-locked host memory, contiguous, same shape on every rank; gradients in
    host memory are read in place over the host link).
    """

    def __init__(self, grads: Sequence[Sequence], flags: Optional[PlanFlags] = None, stream=None,
                 offsets: Optional[Sequence[int]] = None, host_only: bool = False):
        import torch
        self.world = len(grads)
        self.shapes = [tuple(t.shape) for t in grads[0]]
        self.grad_dtype = torch.float32 if (flags is not None and flags.grad_dtype == TIDE_DTYPE_F32) else torch.bfloat16
        descs = _param_descs(grads, offsets, require_cuda=not host_only, dtype=self.grad_dtype)
        if host_only:
            flags = flags or make_flags()
            flags.debug |= TIDE_DEBUG_HOST_ONLY
            stream = 0
        self.handle = tide_plan_build(self.world, descs, flags, 0 if host_only else _stream_handle(stream))
        self.slot_numel = tide_plan_slot_numel(self.handle)

    def rebind(self, grads, stream=None):
        tide_plan_rebind(self.handle, _param_descs(grads, dtype=self.grad_dtype), _stream_handle(stream))

    def rs_fold(self, out, alpha: float = 1.0, accumulate: bool = False, stream=None):
        """out: fp32 CUDA tensor [W, stride] with unit inner stride (stride >= slot_numel)."""
        import torch
        if out.dtype != torch.float32 or out.dim() != 2 or out.shape[0] != self.world or out.stride(1) != 1:
            raise ValueError("out must be float32 [W, stride] with unit inner stride")
        tide_rs_fold(self.handle, out.data_ptr(), out.stride(0) if self.world > 1 else out.shape[1], alpha,
                     int(bool(accumulate)), _stream_handle(stream))
        return out

    def bind_full(self, full: Sequence) -> FullParams:
        """Check the full parameter tensors once; pass the result to the
        placements instead of the list to skip the per-call checks."""
        return FullParams(full, self.shapes)

    def _full_ptrs(self, full):
        if isinstance(full, FullParams):
            if len(full.tensors) != len(self.shapes):
                raise ValueError("bound full tensors belong to another group")
            return full.ptrs
        return FullParams(full, self.shapes).ptrs

    def ag_place(self, slots, full, mode: str = "sm", stream=None):
        """slots: bf16 CUDA tensor [W, stride]; full: a list whose entry p is a
        contiguous bf16 tensor of parameter p's shape, or bind_full(list)."""
        import torch
        if slots.dtype != torch.bfloat16 or slots.dim() != 2 or slots.shape[0] != self.world or slots.stride(1) != 1:
            raise ValueError("slots must be bfloat16 [W, stride] with unit inner stride")
        tide_ag_place(self.handle, slots.data_ptr(), slots.stride(0) if self.world > 1 else slots.shape[1],
                      self._full_ptrs(full), AG_MODES[mode], _stream_handle(stream))
        return full

    def ag_place_f32(self, slots, full, stream=None):
        """Mixed-precision placement: slots fp32 CUDA tensor [W, stride]; full as for ag_place."""
        import torch
        if slots.dtype != torch.float32 or slots.dim() != 2 or slots.shape[0] != self.world or slots.stride(1) != 1:
            raise ValueError("slots must be float32 [W, stride] with unit inner stride")
        tide_ag_place_f32(self.handle, slots.data_ptr(), slots.stride(0) if self.world > 1 else slots.shape[1],
                          self._full_ptrs(full), _stream_handle(stream))
        return full

    def fold_config(self) -> dict:
        return tide_plan_fold_config(self.handle)

    def segments(self) -> list:
        return [tide_plan_segment(self.handle, i) for i in range(tide_plan_num_segments(self.handle))]

    def device_status(self, stream=None) -> int:
        return tide_last_device_status(self.handle, _stream_handle(stream))

    def close(self):
        if getattr(self, "handle", None):
            tide_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
