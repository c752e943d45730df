"""Brute-force restatement of the reduce-scatter and all-gather placement.

TEST INFRASTRUCTURE ONLY (pins the C oracle on tiny shapes; pure-Python loops,
so keep inputs to a few thousand elements).

It is written from the opposite direction to the C oracle so that an index
mistake in one does not hide in the other: the C oracle gathers, for each
destination shard, the rows it owns; this module walks every *source* row
d of every parameter, works out its owner r = d // R_p and local row
i = d - r R_p from the dim-0 sharding rule of the TIDE paper (Section 2.1),
and scatters the reduced row to slot r at offset o_p + i K_p.  Positions a
source row never reaches are padding; Eq. (5) reduces zeros there.

bf16 decoding is done arithmetically (sign, exponent, mantissa, ldexp),
independently of the C oracle's bit shift.  fp32 rounding after every
operation comes from numpy float32 scalar arithmetic.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def bf16_value(bits: int) -> np.float32:
    """Value of a bf16 bit pattern: 1 sign, 8 exponent, 7 mantissa bits."""
    sign = -1.0 if (bits >> 15) & 1 else 1.0
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0xFF:
        return np.float32(sign * math.inf) if m == 0 else np.float32(math.nan)
    if e == 0:
        return np.float32(sign * math.ldexp(m, -133))      # subnormal: m * 2^(1-127-7)
    return np.float32(sign * math.ldexp(128 + m, e - 134))  # (1 + m/128) * 2^(e-127)


def reduce_scatter(world: int, shapes: Sequence[Tuple[int, int]], grads: Sequence[Sequence[np.ndarray]],
                   alpha: float, accumulate: bool, old: np.ndarray) -> np.ndarray:
    """grads[p][u]: flat uint16 bf16 bits of parameter p on rank u.
    old: float32 [W, stride] (read only in accumulate mode).  Returns a new array."""
    a = np.float32(alpha)
    rows = [-(-d // world) for d, _ in shapes]           # ceil(D / W)
    starts, s = [], 0
    for (d, k), R in zip(shapes, rows):
        starts.append(s)
        s += R * k
    out = old.copy()
    written = np.zeros(out.shape, dtype=bool)
    for p, ((d, k), R) in enumerate(zip(shapes, rows)):
        for row in range(d):
            r, i = divmod(row, R)
            for c in range(k):
                acc = bf16_value(int(grads[p][0][row * k + c]))
                for u in range(1, world):
                    acc = np.float32(acc + bf16_value(int(grads[p][u][row * k + c])))
                y = np.float32(a * acc)
                pos = starts[p] + i * k + c
                out[r, pos] = np.float32(old[r, pos] + y) if accumulate else y
                written[r, pos] = True
        # padding: every position of every rank's shard no source row reached
        zero = np.float32(0.0)
        for r in range(world):
            for j in range(R * k):
                pos = starts[p] + j
                if not written[r, pos]:
                    acc = zero
                    for u in range(1, world):
                        acc = np.float32(acc + zero)
                    y = np.float32(a * acc)
                    out[r, pos] = np.float32(old[r, pos] + y) if accumulate else y
    return out


def all_gather(world: int, shapes: Sequence[Tuple[int, int]], slots: np.ndarray) -> List[np.ndarray]:
    """slots: uint16 [W, stride].  Returns flat uint16 full tensors."""
    rows = [-(-d // world) for d, _ in shapes]
    starts, s = [], 0
    for (d, k), R in zip(shapes, rows):
        starts.append(s)
        s += R * k
    full = []
    for p, ((d, k), R) in enumerate(zip(shapes, rows)):
        t = np.zeros(d * k, dtype=np.uint16)
        for row in range(d):
            r, i = divmod(row, R)
            for c in range(k):
                t[row * k + c] = slots[r, starts[p] + i * k + c]
        full.append(t)
    return full


def order_of(world: int, order: str, node_size: int, dest: int):
    """List of rank groups whose partials are added in list order; inside a
    group the ranks are added in list order (Section 4.3 readings)."""
    if order in ("rank", "tree"):
        return [list(range(world))]
    if order == "staged":
        return [[u for u in range(world) if u != dest] + [dest]]
    groups = []
    for n in range(world // node_size):
        members = list(range(n * node_size, (n + 1) * node_size))
        owner = n * node_size + dest % node_size
        groups.append([u for u in members if u != owner] + [owner])
    return groups


def tree_sum(xs):
    """Pairwise summation of xs (fp32) written recursively: the values before
    the largest power of two below len(xs) form one balanced subtree, the rest
    the other.  This is the same tree as adding neighbours level by level and
    carrying an odd last value up (a different construction of it)."""
    n = len(xs)
    if n == 1:
        return xs[0]
    h = 1
    while 2 * h < n:
        h *= 2
    return np.float32(tree_sum(xs[:h]) + tree_sum(xs[h:]))


def reduce_scatter_ordered(world, shapes, grads, alpha, accumulate, old, order="rank", node_size=0):
    """Like reduce_scatter, in a given order; grads are uint16 (bf16) or float32 arrays."""
    a = np.float32(alpha)
    is_f32 = np.asarray(grads[0][0]).dtype == np.float32

    def val(p, u, idx):
        return np.float32(grads[p][u][idx]) if is_f32 else bf16_value(int(grads[p][u][idx]))

    rows = [-(-d // world) for d, _ in shapes]
    starts, s = [], 0
    for (d, k), R in zip(shapes, rows):
        starts.append(s)
        s += R * k
    out = old.copy()
    for p, ((d, k), R) in enumerate(zip(shapes, rows)):
        for r in range(world):
            groups = order_of(world, order, node_size, r)
            for i in range(R):
                row = r * R + i
                for c in range(k):
                    total = None
                    if order == "tree":
                        total = tree_sum([val(p, u, row * k + c) if row < d else np.float32(0.0)
                                          for u in range(world)])
                    for grp in ([] if order == "tree" else groups):
                        part = None
                        for u in grp:
                            x = val(p, u, row * k + c) if row < d else np.float32(0.0)
                            part = x if part is None else np.float32(part + x)
                        total = part if total is None else np.float32(total + part)
                    y = np.float32(a * total)
                    pos = starts[p] + i * k + c
                    out[r, pos] = np.float32(old[r, pos] + y) if accumulate else y
    return out
