"""CPU oracle for the TIDE layout-folded reduce-scatter and all-gather placement.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product package
(``all_gather_gb300``) never does, and this package never imports it.

The arithmetic lives in ``tide_oracle.c`` (plain C, single-threaded, built
with ``-ffp-contract=off -fno-fast-math``); this module compiles it on first
use with the host C compiler and marshals numpy arrays through ctypes.
``oracle.brute`` is a second, independent pure-Python formulation used only
to pin the C oracle on tiny shapes.

What each function follows (TIDE paper, "The Endgame of FSDP Communication"):

* :func:`geometry` -- Section 2.1: R_p = ceil(D_p / W), prefix offsets o_p,
  slot size S; Table 2 notation.
* :func:`valid_rows` -- Section 2.1: rank r owns rows [r R_p, (r+1) R_p),
  rows past D_p are zero.
* :func:`rs_window`, :func:`rs` -- Equation (3) (FSDP2's zero-padded fp32
  pack) followed by Equation (5) (rank-ordered fp32 sum, scale alpha,
  optional accumulate), Section 4.
* :func:`ag` -- Section 2.1, Equation (2): rank-major slots placed into
  per-parameter full tensors, padding dropped.
* :func:`rs_ex`, ``Oracle.rs_window_ex`` -- Section 4.3's orders: rank
  order, the one-node Level 1 order (other ranks in local-rank order, then
  the destination's own contribution) and the two-level order (per-node
  Level 1 partials, then the node partials), for bf16 or fp32 gradients.
* :func:`f32_to_bf16`, :func:`ag_cast` -- Section 3.1 (mixed-precision
  groups cast fp32 master shards to bf16 for the all-gather): the same
  placement from fp32 slots, each element rounded to nearest even.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "tide_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtide_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_lock = threading.Lock()


def compile_library(source: str = SOURCE, out: str = LIB_PATH, extra: Sequence[str] = ()) -> str:
    """Compile the oracle C source into a shared library; returns its path."""
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if not cc:
        raise RuntimeError("no C compiler found to build the oracle")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, *extra, "-o", tmp, source], check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one build of the oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_geometry.argtypes = [ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _i64p, _i64p, _i64p]
        lib.oracle_geometry.restype = ctypes.c_int
        lib.oracle_valid_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
        lib.oracle_valid_rows.restype = ctypes.c_int64
        lib.oracle_rs_window.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.POINTER(_u16p), ctypes.c_float, ctypes.c_int32, _f32p, _f32p]
        lib.oracle_rs_window.restype = ctypes.c_int
        lib.oracle_rs.argtypes = [ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, ctypes.POINTER(_u16p),
                                  ctypes.c_float, ctypes.c_int32, _f32p, ctypes.c_int64]
        lib.oracle_rs.restype = ctypes.c_int
        lib.oracle_ag.argtypes = [ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _u16p, ctypes.c_int64,
                                  ctypes.POINTER(_u16p)]
        lib.oracle_ag.restype = ctypes.c_int
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_ag_cast.argtypes = [ctypes.c_int32, ctypes.c_int32, _i64p, _i64p, _f32p, ctypes.c_int64,
                                       ctypes.POINTER(_u16p)]
        lib.oracle_ag_cast.restype = ctypes.c_int
        lib.oracle_rs_window_ex.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.POINTER(ctypes.c_void_p), ctypes.c_float, ctypes.c_int32,
                                            _f32p, _f32p]
        lib.oracle_rs_window_ex.restype = ctypes.c_int
        lib.oracle_rs_ex.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     _i64p, _i64p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_float, ctypes.c_int32,
                                     _f32p, ctypes.c_int64]
        lib.oracle_rs_ex.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    # -- geometry -----------------------------------------------------------
    def geometry(self, world: int, dims: Sequence[Tuple[int, int]]) -> Tuple[List[int], List[int], int]:
        """(R_p list, o_p list, S) for parameters given as (dim0, row_numel)."""
        P = len(dims)
        d0 = np.array([d for d, _ in dims] or [0], dtype=np.int64)
        kk = np.array([k for _, k in dims] or [0], dtype=np.int64)
        R = np.zeros(max(P, 1), dtype=np.int64)
        o = np.zeros(max(P, 1), dtype=np.int64)
        S = ctypes.c_int64(0)
        rc = self.lib.oracle_geometry(world, P, d0.ctypes.data_as(_i64p), kk.ctypes.data_as(_i64p),
                                      R.ctypes.data_as(_i64p), o.ctypes.data_as(_i64p), ctypes.byref(S))
        if rc != 0:
            raise ValueError(f"oracle_geometry rejected world={world}, dims={dims}")
        return [int(x) for x in R[:P]], [int(x) for x in o[:P]], int(S.value)

    def valid_rows(self, dim0: int, rows_per_rank: int, r: int) -> int:
        return int(self.lib.oracle_valid_rows(dim0, rows_per_rank, r))

    # -- reduce-scatter -----------------------------------------------------
    def rs_window(self, srcs: Sequence[np.ndarray], n_valid: int, n_pad: int, alpha: float,
                  accumulate: bool, old: Optional[np.ndarray] = None) -> np.ndarray:
        """Eq. (3)+(5) on one window: srcs[u] holds >= n_valid bf16 bit patterns."""
        W = len(srcs)
        srcs = [np.ascontiguousarray(s, dtype=np.uint16) for s in srcs]
        for s in srcs:
            if s.size < n_valid:
                raise ValueError("source window shorter than n_valid")
        n = n_valid + n_pad
        out = np.empty(n, dtype=np.float32)
        if accumulate:
            if old is None or old.size < n:
                raise ValueError("accumulate needs the old shard window")
            old = np.ascontiguousarray(old, dtype=np.float32)
        else:
            old = out
        arr = (_u16p * W)(*[s.ctypes.data_as(_u16p) for s in srcs])
        rc = self.lib.oracle_rs_window(W, n_valid, n_pad, arr, ctypes.c_float(alpha), int(bool(accumulate)),
                                       old.ctypes.data_as(_f32p), out.ctypes.data_as(_f32p))
        if rc != 0:
            raise MemoryError(f"oracle_rs_window failed ({rc})")
        return out

    def rs(self, world: int, dims: Sequence[Tuple[int, int]], grads: Sequence[Sequence[np.ndarray]],
           alpha: float, accumulate: bool, out: np.ndarray) -> np.ndarray:
        """Full reduce-scatter.  grads[p][u]: parameter p on rank u as uint16 bf16 bits
        (any shape, contiguous, D_p*K_p elements).  out: float32 [W, stride], updated in place."""
        P = len(dims)
        assert out.dtype == np.float32 and out.ndim == 2 and out.shape[0] == world and out.flags.c_contiguous
        keep = []
        ptrs = (_u16p * max(P * world, 1))()
        for p in range(P):
            for u in range(world):
                g = np.ascontiguousarray(grads[p][u], dtype=np.uint16).reshape(-1)
                assert g.size == dims[p][0] * dims[p][1], "gradient size does not match (dim0, row_numel)"
                keep.append(g)
                ptrs[p * world + u] = g.ctypes.data_as(_u16p)
        d0 = np.array([d for d, _ in dims] or [0], dtype=np.int64)
        kk = np.array([k for _, k in dims] or [0], dtype=np.int64)
        rc = self.lib.oracle_rs(world, P, d0.ctypes.data_as(_i64p), kk.ctypes.data_as(_i64p), ptrs,
                                ctypes.c_float(alpha), int(bool(accumulate)), out.ctypes.data_as(_f32p),
                                out.shape[1])
        if rc != 0:
            raise ValueError(f"oracle_rs failed ({rc})")
        return out

    # -- all-gather placement ----------------------------------------------
    def ag(self, world: int, dims: Sequence[Tuple[int, int]], slots: np.ndarray,
           full: Optional[Sequence[np.ndarray]] = None) -> List[np.ndarray]:
        """slots: uint16 [W, stride].  Returns (or fills) the P full tensors as flat uint16 arrays."""
        P = len(dims)
        slots = np.ascontiguousarray(slots, dtype=np.uint16)
        assert slots.ndim == 2 and slots.shape[0] == world
        if full is None:
            full = [np.zeros(d * k, dtype=np.uint16) for d, k in dims]
        ptrs = (_u16p * max(P, 1))(*[f.ctypes.data_as(_u16p) for f in full])
        d0 = np.array([d for d, _ in dims] or [0], dtype=np.int64)
        kk = np.array([k for _, k in dims] or [0], dtype=np.int64)
        rc = self.lib.oracle_ag(world, P, d0.ctypes.data_as(_i64p), kk.ctypes.data_as(_i64p),
                                slots.ctypes.data_as(_u16p), slots.shape[1], ptrs)
        if rc != 0:
            raise ValueError(f"oracle_ag failed ({rc})")
        return list(full)


    def f32_to_bf16(self, x: float) -> int:
        """Round-to-nearest-even binary32 -> bf16 bit pattern (one value)."""
        return int(self.lib.oracle_f32_to_bf16(ctypes.c_float(x)))

    def ag_cast(self, world: int, dims: Sequence[Tuple[int, int]], slots: np.ndarray,
                full: Optional[Sequence[np.ndarray]] = None) -> List[np.ndarray]:
        """Mixed-precision placement: slots float32 [W, stride] -> P flat uint16 bf16 tensors."""
        P = len(dims)
        slots = np.ascontiguousarray(slots, dtype=np.float32)
        assert slots.ndim == 2 and slots.shape[0] == world
        if full is None:
            full = [np.zeros(d * k, dtype=np.uint16) for d, k in dims]
        ptrs = (_u16p * max(P, 1))(*[f.ctypes.data_as(_u16p) for f in full])
        d0 = np.array([d for d, _ in dims] or [0], dtype=np.int64)
        kk = np.array([k for _, k in dims] or [0], dtype=np.int64)
        rc = self.lib.oracle_ag_cast(world, P, d0.ctypes.data_as(_i64p), kk.ctypes.data_as(_i64p),
                                     slots.ctypes.data_as(_f32p), slots.shape[1], ptrs)
        if rc != 0:
            raise ValueError(f"oracle_ag_cast failed ({rc})")
        return list(full)


    # -- other summation orders, fp32 gradients ----------------------------
    ORDERS = {"rank": 0, "staged": 1, "nodes": 2, "tree": 3}

    def rs_ex(self, world: int, dims, grads, alpha: float, accumulate: bool, out: np.ndarray,
              order: str = "rank", node_size: int = 0) -> np.ndarray:
        """Reduce-scatter in a given order.  grads[p][u]: uint16 (bf16 bits) or float32 arrays."""
        P = len(dims)
        assert out.dtype == np.float32 and out.ndim == 2 and out.shape[0] == world and out.flags.c_contiguous
        dtype = 1 if (P and np.asarray(grads[0][0]).dtype == np.float32) else 0
        keep = []
        ptrs = (ctypes.c_void_p * max(P * world, 1))()
        for p in range(P):
            for u in range(world):
                g = np.ascontiguousarray(grads[p][u], dtype=np.float32 if dtype else np.uint16).reshape(-1)
                assert g.size == dims[p][0] * dims[p][1]
                keep.append(g)
                ptrs[p * world + u] = g.ctypes.data
        d0 = np.array([d for d, _ in dims] or [0], dtype=np.int64)
        kk = np.array([k for _, k in dims] or [0], dtype=np.int64)
        rc = self.lib.oracle_rs_ex(world, dtype, self.ORDERS[order], node_size, P, d0.ctypes.data_as(_i64p),
                                   kk.ctypes.data_as(_i64p), ptrs, ctypes.c_float(alpha), int(bool(accumulate)),
                                   out.ctypes.data_as(_f32p), out.shape[1])
        if rc != 0:
            raise ValueError(f"oracle_rs_ex failed ({rc})")
        return out

    def rs_window_ex(self, srcs, n_valid: int, n_pad: int, alpha: float, accumulate: bool, dest: int,
                     order: str = "rank", node_size: int = 0, old=None) -> np.ndarray:
        W = len(srcs)
        dtype = 1 if np.asarray(srcs[0]).dtype == np.float32 else 0
        srcs = [np.ascontiguousarray(x, dtype=np.float32 if dtype else np.uint16) for x in srcs]
        n = n_valid + n_pad
        out = np.empty(n, dtype=np.float32)
        old = np.ascontiguousarray(old, dtype=np.float32) if accumulate else out
        arr = (ctypes.c_void_p * W)(*[x.ctypes.data for x in srcs])
        rc = self.lib.oracle_rs_window_ex(W, dtype, self.ORDERS[order], node_size, dest, n_valid, n_pad, arr,
                                          ctypes.c_float(alpha), int(bool(accumulate)), old.ctypes.data_as(_f32p),
                                          out.ctypes.data_as(_f32p))
        if rc != 0:
            raise ValueError(f"oracle_rs_window_ex failed ({rc})")
        return out


_default: Optional[Oracle] = None


def load(rebuild: bool = False) -> Oracle:
    """The oracle built from ``tide_oracle.c`` (compiled if missing or stale)."""
    global _default
    with _lock:
        if _default is not None and not rebuild:
            return _default
        stale = (not os.path.exists(LIB_PATH)
                 or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE))
        if rebuild or stale:
            compile_library()
        _default = Oracle(LIB_PATH)
        return _default


def geometry(world, dims):
    return load().geometry(world, dims)


def valid_rows(dim0, rows_per_rank, r):
    return load().valid_rows(dim0, rows_per_rank, r)


def rs_window(srcs, n_valid, n_pad, alpha, accumulate, old=None):
    return load().rs_window(srcs, n_valid, n_pad, alpha, accumulate, old)


def rs(world, dims, grads, alpha, accumulate, out):
    return load().rs(world, dims, grads, alpha, accumulate, out)


def ag(world, dims, slots, full=None):
    return load().ag(world, dims, slots, full)


def rs_ex(world, dims, grads, alpha, accumulate, out, order="rank", node_size=0):
    return load().rs_ex(world, dims, grads, alpha, accumulate, out, order, node_size)


def f32_to_bf16(x):
    return load().f32_to_bf16(x)


def ag_cast(world, dims, slots, full=None):
    return load().ag_cast(world, dims, slots, full)
