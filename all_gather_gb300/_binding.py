"""ctypes binding of libtide (include/tide.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own; a non-OK status raises :class:`TideError`.  The
library must have been built (``python -m all_gather_gb300.build``); there is
no fallback of any kind when it is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libtide.so")

# status codes
TIDE_OK = 0
TIDE_ERR_INVALID_ARG = 1
TIDE_ERR_ALIGNMENT = 2
TIDE_ERR_UNSUPPORTED = 3
TIDE_ERR_OOM = 4
TIDE_ERR_CUDA = 5
TIDE_ERR_TIMEOUT = 6
# enums
TIDE_ORDER_RANK_ASC, TIDE_ORDER_STAGED_OWN, TIDE_ORDER_NODES, TIDE_ORDER_TREE = 0, 1, 2, 3
TIDE_SCHED_AUTO, TIDE_SCHED_DYNAMIC, TIDE_SCHED_PER_ITEM, TIDE_SCHED_STATIC = 0, 1, 2, 3
TIDE_KERNEL_AUTO, TIDE_KERNEL_DIRECT, TIDE_KERNEL_BULK = 0, 1, 2
TIDE_AG_SM, TIDE_AG_CE_2D, TIDE_AG_CE_1D = 0, 1, 2
TIDE_DTYPE_BF16, TIDE_DTYPE_F32 = 0, 1
TIDE_DEBUG_HOST_ONLY = 0x1
TIDE_DEBUG_SHORT_WAIT = 0x2
TIDE_DEBUG_SKIP_FILL = 0x4

EXPORTED = ("tide_plan_build", "tide_plan_rebind", "tide_rs_fold", "tide_ag_place", "tide_plan_destroy",
            "tide_plan_slot_numel", "tide_plan_num_segments", "tide_plan_segment", "tide_plan_fold_config",
            "tide_last_device_status", "tide_launch_count", "tide_status_string", "tide_last_error",
            "tide_rs_fold_noalloc", "tide_ag_place_f32", "tide_latin_square_gpu", "tide_rs_wave_plan",
            "tide_rs_wave_zero_mask", "tide_bruck_schedule", "tide_sm_probe", "tide_sm_probe_max_clusters",
            "tide_corun_cta_budget")


class WavePlan(ctypes.Structure):
    _fields_ = [("waves", ctypes.c_int32), ("generations", ctypes.c_int32), ("network_rounds", ctypes.c_int32),
                ("zero_blocks", ctypes.c_int32)]


class TideError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{where}: {_status_name(status)}: {detail}")


class ParamDesc(ctypes.Structure):
    _fields_ = [("rank_base", ctypes.POINTER(ctypes.c_void_p)), ("dim0", ctypes.c_int64),
                ("row_numel", ctypes.c_int64), ("shard_offset", ctypes.c_int64)]


class PlanFlags(ctypes.Structure):
    _fields_ = [("cta_budget", ctypes.c_int32), ("chunk_bytes", ctypes.c_int32), ("order", ctypes.c_int32),
                ("sched", ctypes.c_int32), ("kernel", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("debug", ctypes.c_uint32), ("fill_bytes", ctypes.c_int32), ("fill_ranks", ctypes.c_int32),
                ("node_size", ctypes.c_int32), ("ce_streams", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1)]


class Segment(ctypes.Structure):
    _fields_ = [("param", ctypes.c_int32), ("rank", ctypes.c_int32), ("src_elem", ctypes.c_int64),
                ("dst_elem", ctypes.c_int64), ("n_valid", ctypes.c_int64), ("n_pad", ctypes.c_int64)]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtide.so; raises ImportError (never falls back) if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libtide.so is not built ({path}); run `python -m all_gather_gb300.build` "
                          "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(path)
    vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    lib.tide_plan_build.argtypes = [i32, i32, ctypes.POINTER(ParamDesc), ctypes.POINTER(PlanFlags), vp,
                                    ctypes.POINTER(vp)]
    lib.tide_plan_build.restype = st
    lib.tide_plan_rebind.argtypes = [vp, ctypes.POINTER(ParamDesc), vp]
    lib.tide_plan_rebind.restype = st
    lib.tide_rs_fold.argtypes = [vp, vp, i64, ctypes.c_float, i32, vp]
    lib.tide_rs_fold.restype = st
    lib.tide_ag_place.argtypes = [vp, vp, i64, ctypes.POINTER(vp), i32, vp]
    lib.tide_ag_place.restype = st
    lib.tide_plan_destroy.argtypes = [vp]
    lib.tide_plan_destroy.restype = st
    lib.tide_plan_slot_numel.argtypes = [vp]
    lib.tide_plan_slot_numel.restype = i64
    lib.tide_plan_num_segments.argtypes = [vp]
    lib.tide_plan_num_segments.restype = i64
    lib.tide_plan_segment.argtypes = [vp, i64, ctypes.POINTER(Segment)]
    lib.tide_plan_segment.restype = st
    lib.tide_plan_fold_config.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i64),
                                          ctypes.POINTER(i64)]
    lib.tide_plan_fold_config.restype = st
    lib.tide_last_device_status.argtypes = [vp, vp]
    lib.tide_last_device_status.restype = st
    lib.tide_launch_count.argtypes = []
    lib.tide_launch_count.restype = ctypes.c_uint64
    lib.tide_status_string.argtypes = [st]
    lib.tide_status_string.restype = ctypes.c_char_p
    lib.tide_last_error.argtypes = []
    lib.tide_last_error.restype = ctypes.c_char_p
    lib.tide_rs_fold_noalloc.argtypes = [i32, i32, ctypes.POINTER(ParamDesc), vp, i64, ctypes.c_float, i32, vp]
    lib.tide_rs_fold_noalloc.restype = st
    lib.tide_ag_place_f32.argtypes = [vp, vp, i64, ctypes.POINTER(vp), vp]
    lib.tide_ag_place_f32.restype = st
    lib.tide_latin_square_gpu.argtypes = [i32, i32, i32, i32, i32]
    lib.tide_latin_square_gpu.restype = i32
    lib.tide_rs_wave_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(WavePlan)]
    lib.tide_rs_wave_plan.restype = st
    lib.tide_rs_wave_zero_mask.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_uint64)]
    lib.tide_rs_wave_zero_mask.restype = st
    lib.tide_bruck_schedule.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(i32), i32]
    lib.tide_bruck_schedule.restype = i32
    lib.tide_sm_probe.argtypes = [i32, i32, i32, ctypes.c_uint64, vp, vp, vp, vp, vp]
    lib.tide_sm_probe.restype = st
    lib.tide_sm_probe_max_clusters.argtypes = [i32, i32]
    lib.tide_sm_probe_max_clusters.restype = i32
    lib.tide_corun_cta_budget.argtypes = [i32, i32, i32]
    lib.tide_corun_cta_budget.restype = i32
    _lib = lib
    return lib


def _status_name(status: int) -> str:
    try:
        return load_library().tide_status_string(status).decode()
    except ImportError:
        return str(status)


def _check(status: int, where: str):
    if status != TIDE_OK:
        raise TideError(status, where, load_library().tide_last_error().decode())


def _descs(params: Sequence[Tuple[Sequence[int], int, int, int]]):
    """params[p] = (rank_base pointers [W], dim0, row_numel, shard_offset)."""
    arr = (ParamDesc * max(len(params), 1))()
    keep = []
    for i, (ptrs, d0, k, off) in enumerate(params):
        base = (ctypes.c_void_p * max(len(ptrs), 1))(*[ctypes.c_void_p(int(x) or None) for x in ptrs])
        keep.append(base)
        arr[i].rank_base = ctypes.cast(base, ctypes.POINTER(ctypes.c_void_p))
        arr[i].dim0, arr[i].row_numel, arr[i].shard_offset = int(d0), int(k), int(off)
    return arr, keep


def make_flags(cta_budget=0, chunk_bytes=0, order=TIDE_ORDER_RANK_ASC, sched=TIDE_SCHED_AUTO,
               kernel=TIDE_KERNEL_AUTO, grad_dtype=TIDE_DTYPE_BF16, debug=0, fill_bytes=0,
               fill_ranks=0, node_size=0, ce_streams=0) -> PlanFlags:
    f = PlanFlags()
    f.cta_budget, f.chunk_bytes, f.order, f.sched = cta_budget, chunk_bytes, order, sched
    f.kernel, f.grad_dtype, f.debug, f.fill_bytes, f.fill_ranks = kernel, grad_dtype, debug, fill_bytes, fill_ranks
    f.node_size, f.ce_streams = node_size, ce_streams
    return f


def tide_plan_build(world: int, params, flags: Optional[PlanFlags] = None, stream: int = 0) -> int:
    lib = load_library()
    arr, _keep = _descs(params)
    out = ctypes.c_void_p()
    fl = ctypes.byref(flags) if flags is not None else None
    _check(lib.tide_plan_build(world, len(params), arr, fl, ctypes.c_void_p(stream or None), ctypes.byref(out)),
           "tide_plan_build")
    return out.value


def tide_plan_rebind(plan: int, params, stream: int = 0) -> None:
    arr, _keep = _descs(params)
    _check(load_library().tide_plan_rebind(ctypes.c_void_p(plan), arr, ctypes.c_void_p(stream or None)),
           "tide_plan_rebind")


def tide_rs_fold(plan: int, out_base: int, out_slot_stride: int, alpha: float, accumulate: int,
                 stream: int = 0) -> None:
    _check(load_library().tide_rs_fold(ctypes.c_void_p(plan), ctypes.c_void_p(out_base or None), out_slot_stride,
                                       ctypes.c_float(alpha), int(accumulate), ctypes.c_void_p(stream or None)),
           "tide_rs_fold")


def pointer_array(ptrs: Sequence[int]):
    """A C array of device pointers (void *const *) for the placements; build
    it once and pass it again to skip the per-call conversion."""
    return (ctypes.c_void_p * max(len(ptrs), 1))(*[int(x) or None for x in ptrs])


def _as_pointer_array(full):
    return full if isinstance(full, ctypes.Array) else pointer_array(full)


def tide_ag_place(plan: int, slots_base: int, slot_stride: int, full, mode: int, stream: int = 0) -> None:
    """full: device pointers of the P full tensors (a sequence, or pointer_array(...))."""
    _check(load_library().tide_ag_place(ctypes.c_void_p(plan), ctypes.c_void_p(slots_base or None), slot_stride,
                                        _as_pointer_array(full), mode, ctypes.c_void_p(stream or None)),
           "tide_ag_place")


def tide_ag_place_f32(plan: int, slots_base: int, slot_stride: int, full, stream: int = 0) -> None:
    _check(load_library().tide_ag_place_f32(ctypes.c_void_p(plan), ctypes.c_void_p(slots_base or None), slot_stride,
                                            _as_pointer_array(full), ctypes.c_void_p(stream or None)),
           "tide_ag_place_f32")


def tide_plan_destroy(plan: int) -> None:
    _check(load_library().tide_plan_destroy(ctypes.c_void_p(plan)), "tide_plan_destroy")


def tide_plan_slot_numel(plan: int) -> int:
    return int(load_library().tide_plan_slot_numel(ctypes.c_void_p(plan)))


def tide_plan_num_segments(plan: int) -> int:
    return int(load_library().tide_plan_num_segments(ctypes.c_void_p(plan)))


def tide_plan_segment(plan: int, index: int) -> dict:
    s = Segment()
    _check(load_library().tide_plan_segment(ctypes.c_void_p(plan), index, ctypes.byref(s)), "tide_plan_segment")
    return {k: getattr(s, k) for k, _ in Segment._fields_}


def tide_plan_fold_config(plan: int) -> dict:
    g, b = ctypes.c_int32(), ctypes.c_int32()
    n, c = ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().tide_plan_fold_config(ctypes.c_void_p(plan), ctypes.byref(g), ctypes.byref(b),
                                                ctypes.byref(n), ctypes.byref(c)), "tide_plan_fold_config")
    return {"grid": g.value, "block": b.value, "items": n.value, "chunk_elems": c.value}


def tide_last_device_status(plan: int, stream: int = 0) -> int:
    """Returns the status code (TIDE_OK or TIDE_ERR_TIMEOUT) instead of raising on a timeout."""
    st = load_library().tide_last_device_status(ctypes.c_void_p(plan), ctypes.c_void_p(stream or None))
    if st not in (TIDE_OK, TIDE_ERR_TIMEOUT):
        _check(st, "tide_last_device_status")
    return st


def tide_launch_count() -> int:
    return int(load_library().tide_launch_count())


def tide_status_string(status: int) -> str:
    return load_library().tide_status_string(status).decode()


def tide_last_error() -> str:
    return load_library().tide_last_error().decode()


def tide_rs_fold_noalloc(world: int, params, out_base: int, out_slot_stride: int, alpha: float, accumulate: int,
                         stream: int = 0) -> None:
    """The allocation-free fold: same arguments as tide_plan_build + tide_rs_fold, no plan."""
    arr, _keep = _descs(params)
    _check(load_library().tide_rs_fold_noalloc(world, len(params), arr, ctypes.c_void_p(out_base or None),
                                               out_slot_stride, ctypes.c_float(alpha), int(accumulate),
                                               ctypes.c_void_p(stream or None)), "tide_rs_fold_noalloc")


def tide_latin_square_gpu(s: int, m: int, n: int, M: int, L: int) -> int:
    return int(load_library().tide_latin_square_gpu(s, m, n, M, L))


def tide_rs_wave_plan(M: int, L: int, w_wave: int, k: int, me: int):
    """(status, dict) -- status TIDE_OK (accepted) or TIDE_ERR_UNSUPPORTED (collision); other errors raise."""
    plan = WavePlan()
    st = load_library().tide_rs_wave_plan(M, L, w_wave, k, me, ctypes.byref(plan))
    if st not in (TIDE_OK, TIDE_ERR_UNSUPPORTED):
        _check(st, "tide_rs_wave_plan")
    return st, {k_: getattr(plan, k_) for k_, _ in WavePlan._fields_}


def tide_rs_wave_zero_mask(M: int, L: int, w_wave: int, me: int, wave: int):
    arr = (ctypes.c_uint64 * L)()
    _check(load_library().tide_rs_wave_zero_mask(M, L, w_wave, me, wave, arr), "tide_rs_wave_zero_mask")
    return list(arr)


def tide_bruck_schedule(M: int, max_rounds: int = 64):
    cnt, stp = (ctypes.c_int32 * max_rounds)(), (ctypes.c_int32 * max_rounds)()
    R = load_library().tide_bruck_schedule(M, cnt, stp, max_rounds)
    if R < 0:
        raise ValueError(f"tide_bruck_schedule rejected M={M}")
    return [(d, cnt[d], stp[d]) for d in range(R)]


def tide_sm_probe(ctas: int, cluster: int, smem_bytes: int, hold_ns: int, smid: int, t_in: int, t_out: int,
                  t_ready: int = 0, stream: int = 0) -> None:
    _check(load_library().tide_sm_probe(ctas, cluster, smem_bytes, hold_ns, ctypes.c_void_p(smid),
                                        ctypes.c_void_p(t_in), ctypes.c_void_p(t_out),
                                        ctypes.c_void_p(t_ready or None), ctypes.c_void_p(stream or None)),
           "tide_sm_probe")


def tide_sm_probe_max_clusters(cluster: int, smem_bytes: int) -> int:
    return int(load_library().tide_sm_probe_max_clusters(cluster, smem_bytes))


def tide_corun_cta_budget(cluster_slots: int, gemm_ctas: int, cluster: int) -> int:
    return int(load_library().tide_corun_cta_budget(cluster_slots, gemm_ctas, cluster))
