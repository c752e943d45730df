"""Checks that pin the CPU oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them against the
oracle as built; ``test_oracle_mutants.py`` runs them against copies of the
oracle with a planted mistake and requires that some pin fails.

What pins what:
* hand-worked fixtures (tests/golden/) -- geometry, padding, scale, accumulate;
* torch.chunk (FSDP2's dim-0 sharding routine) -- padded row counts and the
  valid rows per rank;
* torch._chunk_cat (FSDP2's pack, Eq. (3) of the TIDE paper) followed by a
  rank-ordered fp32 sum -- the whole reduce-scatter on ragged shapes;
* a brute-force scatter formulation (oracle/brute.py) on tiny shapes;
* integer-valued inputs -- exact in any order (paper Section 4.3);
* a closed-form summation-order probe (1 + 2^-24 ties to even);
* the textbook recursive-summation error bound against an fp64 sum, and the
  paper's own 1e-5 max(1, |y_ref|_inf) criterion (Section 4.3);
* special values: NaN, +-inf, -0, subnormals, overflow (Section 4.3: NaN and
  inf inputs give the expected output classes);
* slot sizes S of the five workloads, computed by hand.
"""
from __future__ import annotations

import random

import numpy as np
import torch

from bits import (assert_same_f32, assert_same_u16, bf16_bits_to_f32, f32_to_bf16_bits, parse_golden)

U = 2.0 ** -24  # unit roundoff of binary32


# ---------------------------------------------------------------------------
# helpers
def _rand_bits(rng: np.random.Generator, n: int, scale: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32) * np.float32(scale))


def _grads(world, dims, rng, scale=1.0):
    return [[_rand_bits(rng, d * k, scale) for _ in range(world)] for d, k in dims]


def _run_rs(orc, world, dims, grads, alpha, accumulate, old=None, extra=0):
    _, _, S = orc.geometry(world, dims)
    stride = S + extra
    out = np.zeros((world, stride), dtype=np.float32) if old is None else old.copy()
    orc.rs(world, dims, grads, alpha, accumulate, out)
    return out, S


# ---------------------------------------------------------------------------
def pin_golden(orc):
    """Hand-worked fixtures, bitwise."""
    for name in ("rs_w2_hand.txt", "rs_w3_hand.txt"):
        g = parse_golden(name)
        W = g["world"]
        dims = [(d, k) for _, d, k in g["params"]]
        grads = [[f32_to_bf16_bits(g["grad"][(pname, u)]) for u in range(W)] for pname, _, _ in g["params"]]
        _, _, S = orc.geometry(W, dims)
        assert S == len(g["expect"][0]), f"{name}: slot size {S}"
        out = np.full((W, g["stride"]), 12345.0, dtype=np.float32)
        orc.rs(W, dims, grads, g["alpha"], False, out)
        for r in range(W):
            assert_same_f32(out[r, :S], np.array(g["expect"][r], np.float32), f"{name} rank {r}")
        if g["old"]:
            out = np.stack([np.array(g["old"][r], np.float32) for r in range(W)])
            orc.rs(W, dims, grads, g["alpha"], True, out)
            for r in range(W):
                assert_same_f32(out[r], np.array(g["expect_acc"][r], np.float32), f"{name} acc rank {r}")
    g = parse_golden("ag_w2_hand.txt")
    W = g["world"]
    dims = [(d, k) for _, d, k in g["params"]]
    slots = np.stack([f32_to_bf16_bits(g["slot"][r]) for r in range(W)])
    full = orc.ag(W, dims, slots)
    for (pname, _, _), f in zip(g["params"], full):
        assert_same_u16(f, f32_to_bf16_bits(g["full"][pname]), f"ag {pname}")


def pin_slot_sizes(orc):
    """S per rank slot and total padding of the five workloads (computed by hand:
    e.g. the toy group has R = 250, 16, 84, 2, 1024, 33 rows, so
    S = 16000 + 16 + 1428 + 10 + 1024 + 4224 = 22702 and W S - N = 440)."""
    import workloads
    expect = {1: (22_702, 440), 2: (27_264_000, 0), 3: (106_956_800, 0), 4: (21_957_760, 0), 5: (19_472_384, 0)}
    for w in workloads.WORKLOADS:
        _, _, S = orc.geometry(w.world, w.dim0_rownumel())
        assert (S, w.world * S - w.total_numel()) == expect[w.index], f"{w.name}: S={S}"


def pin_torch_chunk(orc):
    """Row counts against torch.chunk, the routine FSDP2 shards dim 0 with:
    R_p is the first chunk's length and rank r holds chunk r (or nothing)."""
    for W in (1, 2, 3, 4, 7, 8, 16, 32):
        for D in (1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 100, 333):
            chunks = torch.chunk(torch.arange(D), W)
            R, _, _ = orc.geometry(W, [(D, 3)])
            assert R[0] == chunks[0].numel(), f"W={W} D={D}: R={R[0]}"
            for r in range(W):
                want = chunks[r].numel() if r < len(chunks) else 0
                got = orc.valid_rows(D, R[0], r)
                assert got == want, f"W={W} D={D} r={r}: {got} rows, torch.chunk gives {want}"


def _chunk_cat_reduce(world, shapes, grads_bits, alpha, accumulate, old):
    """Stock FSDP2's two passes with library routines: torch._chunk_cat packs
    each source rank's gradients into fp32 [W, S] (slice, zero-pad, upcast),
    then the W packs are added in rank order in fp32."""
    packs = []
    for u in range(world):
        ts = [torch.from_numpy(grads_bits[p][u].view(np.int16).copy()).view(torch.bfloat16).reshape(shapes[p])
              for p in range(len(shapes))]
        S = sum(-(-t.shape[0] // world) * (t.numel() // t.shape[0]) for t in ts)
        out = torch.empty(world, S, dtype=torch.float32)
        torch._chunk_cat(ts, dim=0, num_chunks=world, out=out)
        packs.append(out)
    acc = packs[0].clone()
    for u in range(1, world):
        acc = acc + packs[u]
    y = acc * torch.tensor(alpha, dtype=torch.float32)
    if accumulate:
        y = torch.from_numpy(old) + y
    return y.numpy()


def pin_chunk_cat(orc, seed=7):
    rng = np.random.default_rng(seed)
    cases = [
        (4, [(1000, 64), (64, 1), (333, 17), (7, 5), (4096, 1), (129, 128)]),
        (3, [(5, 2), (1, 1), (2, 9), (10, 3)]),
        (8, [(3, 4), (17, 5), (8, 8), (64, 1)]),
        (5, [(23, 7), (4, 4)]),
    ]
    for W, dims in cases:
        shapes = [(d, k) for d, k in dims]
        grads = _grads(W, dims, rng, 1e-3)
        for alpha, acc in ((1.0, False), (1.0 / W, False), (0.3, True)):
            _, _, S = orc.geometry(W, dims)
            old = rng.standard_normal((W, S)).astype(np.float32) * np.float32(1e-3)
            want = _chunk_cat_reduce(W, shapes, grads, alpha, acc, old)
            out = old.copy()
            orc.rs(W, dims, grads, alpha, acc, out)
            assert_same_f32(out, want, f"chunk_cat W={W} dims={dims} alpha={alpha} acc={acc}")


def pin_brute_force(orc, seed=11, cases=40):
    from oracle import brute
    rnd = random.Random(seed)
    rng = np.random.default_rng(seed)
    for c in range(cases):
        W = rnd.choice([1, 2, 3, 4, 5, 8])
        P = rnd.randint(1, 4)
        dims = [(rnd.choice([1, 2, 3, W - 1 or 1, W, W + 1, 2 * W + 1, 7, 13]), rnd.choice([1, 2, 3, 5, 8]))
                for _ in range(P)]
        grads = _grads(W, dims, rng)
        alpha = rnd.choice([1.0, 1.0 / W, 0.3, -2.0])
        acc = rnd.random() < 0.5
        _, _, S = orc.geometry(W, dims)
        stride = S + rnd.choice([0, 1, 3])
        old = rng.standard_normal((W, stride)).astype(np.float32)
        out = old.copy()
        orc.rs(W, dims, grads, alpha, acc, out)
        want = brute.reduce_scatter(W, dims, grads, alpha, acc, old)
        assert_same_f32(out, want, f"brute case {c}: W={W} dims={dims} alpha={alpha} acc={acc}")
        slots = rng.integers(0, 0x7F00, size=(W, stride), dtype=np.uint16)
        assert_same_u16(np.concatenate(orc.ag(W, dims, slots)), np.concatenate(brute.all_gather(W, dims, slots)),
                        f"brute ag case {c}")


def pin_integer_exact(orc, seed=3):
    """Integer-valued inputs with exactly representable sums: every summation
    order gives the exact sum, times a power-of-two alpha (Section 4.3)."""
    rng = np.random.default_rng(seed)
    for W in (2, 4, 8, 16, 32):
        dims = [(3 * W + 1, 5), (W, 8), (1, 3)]
        ints = [[rng.integers(-128, 129, size=d * k) for _ in range(W)] for d, k in dims]
        grads = [[f32_to_bf16_bits(x.astype(np.float32)) for x in per] for per in ints]
        for alpha in (1.0, 1.0 / W, 0.5):
            out, S = _run_rs(orc, W, dims, grads, alpha, False)
            R, o, _ = orc.geometry(W, dims)
            for p, (d, k) in enumerate(dims):
                exact = np.zeros(d * k, dtype=np.int64)
                for u in range(W):
                    exact += ints[p][u]
                flat = np.concatenate([out[r, o[p]:o[p] + R[p] * k] for r in range(W)])[:d * k]
                assert_same_f32(flat, (exact.astype(np.float64) * alpha).astype(np.float32),
                                f"integer W={W} p={p} alpha={alpha}")


def pin_order_probe(orc):
    """Closed form of the rank-ascending fp32 order.  With 1.0 on rank 0 and
    2^-24 on every other rank, each step 1 + 2^-24 is a tie that rounds to
    even, so the result is exactly 1.0 for every W.  With 1.0 on the last rank
    instead, the small terms add exactly to (W-1) 2^-24 first and the result is
    that sum plus 1 rounded once."""
    for W in (2, 3, 4, 8, 16, 32):
        big, small = f32_to_bf16_bits([1.0])[0], f32_to_bf16_bits([U])[0]
        first = [[np.array([big if u == 0 else small], np.uint16) for u in range(W)]]
        out, _ = _run_rs(orc, W, [(1, 1)], first, 1.0, False)
        assert_same_f32(out[0, :1], np.array([1.0], np.float32), f"order probe (big first) W={W}")
        last = [[np.array([big if u == W - 1 else small], np.uint16) for u in range(W)]]
        out, _ = _run_rs(orc, W, [(1, 1)], last, 1.0, False)
        assert_same_f32(out[0, :1], np.array([1.0 + (W - 1) * U], np.float32), f"order probe (big last) W={W}")


def pin_fp64_bound(orc, seed=5):
    """Recursive-summation error bound against an fp64 reference:
    |y - y64| <= gamma_{W+1} (|alpha| sum_u |G^(u)| + |old|), gamma_n = n u / (1 - n u),
    and the paper's criterion |y - y64| <= 1e-5 max(1, |y64|_inf) (Section 4.3)."""
    rng = np.random.default_rng(seed)
    for W in (2, 8, 32):
        dims = [(4 * W + 3, 33), (W + 1, 1)]
        grads = [[f32_to_bf16_bits(rng.standard_normal(d * k).astype(np.float32)
                                   * np.float32(10.0 ** rng.integers(-3, 3))) for _ in range(W)] for d, k in dims]
        for alpha, acc in ((1.0, False), (0.1, True)):
            _, _, S = orc.geometry(W, dims)
            old = rng.standard_normal((W, S)).astype(np.float32)
            out = old.copy()
            orc.rs(W, dims, grads, alpha, acc, out)
            R, o, _ = orc.geometry(W, dims)
            n = W + 1
            gamma = n * U / (1 - n * U)
            for p, (d, k) in enumerate(dims):
                vals = np.stack([bf16_bits_to_f32(grads[p][u]).astype(np.float64) for u in range(W)])
                s64 = vals.sum(axis=0) * float(np.float32(alpha))
                mag = np.abs(vals).sum(axis=0) * abs(float(np.float32(alpha)))
                got = np.concatenate([out[r, o[p]:o[p] + R[p] * k] for r in range(W)])[:d * k].astype(np.float64)
                base = np.concatenate([old[r, o[p]:o[p] + R[p] * k] for r in range(W)])[:d * k].astype(np.float64)
                if acc:
                    s64 = s64 + base
                    mag = mag + np.abs(base)
                err = np.abs(got - s64)
                assert (err <= gamma * mag + 1e-45).all(), f"fp64 bound W={W} p={p}: max excess {(err - gamma * mag).max()}"
                assert err.max() <= 1e-5 * max(1.0, np.abs(s64).max()), f"paper criterion W={W} p={p}"


def pin_special_values(orc):
    nan, inf = float("nan"), float("inf")

    def one(vals, alpha=1.0, acc=False, old=0.0):
        W = len(vals)
        grads = [[f32_to_bf16_bits([v]) for v in vals]]
        o = np.full((W, 1), old, dtype=np.float32)
        out, _ = _run_rs(orc, W, [(1, 1)], grads, alpha, acc, old=o)
        return out[0, :1]

    assert np.isnan(one([1.0, nan, 2.0]))[0], "NaN must propagate"
    assert_same_f32(one([1.0, inf, -3.0]), np.array([inf], np.float32), "+inf")
    assert np.isnan(one([inf, 1.0, -inf]))[0], "inf - inf is NaN"
    assert_same_f32(one([-0.0, -0.0, -0.0]), np.array([-0.0], np.float32), "all -0 stays -0")
    assert_same_f32(one([-0.0, -0.0], alpha=0.25), np.array([-0.0], np.float32), "-0 times alpha")
    assert_same_f32(one([-0.0, 0.0]), np.array([0.0], np.float32), "-0 + +0 is +0")
    assert_same_f32(one([-0.0, -0.0], acc=True, old=-0.0), np.array([-0.0], np.float32), "-0 accumulate")
    # subnormal bf16 (0x0001 = 2^-133) summed W times is exact in binary32
    for W in (2, 5, 32):
        grads = [[np.array([1], np.uint16) for _ in range(W)]]
        out, _ = _run_rs(orc, W, [(1, 1)], grads, 1.0, False)
        assert_same_f32(out[0, :1], np.array([W * 2.0 ** -133], np.float32), f"subnormal sum W={W}")
    # bf16 max (0x7F7F) twice overflows binary32
    grads = [[np.array([0x7F7F], np.uint16), np.array([0x7F7F], np.uint16)]]
    out, _ = _run_rs(orc, 2, [(1, 1)], grads, 1.0, False)
    assert_same_f32(out[0, :1], np.array([inf], np.float32), "overflow to +inf")
    # padding: rows past D_p reduce zeros -> +0 (alpha > 0), -0 (alpha < 0),
    # old + (+0) in accumulate mode (which turns an old -0 into +0)
    W, dims = 4, [(1, 2)]
    grads = [[f32_to_bf16_bits([3.0, -1.0]) for _ in range(W)]]
    out, _ = _run_rs(orc, W, dims, grads, 0.5, False, old=np.full((W, 2), 7.0, np.float32))
    assert_same_f32(out[1:], np.zeros((W - 1, 2), np.float32), "padding is +0")
    out, _ = _run_rs(orc, W, dims, grads, -1.0, False, old=np.full((W, 2), 7.0, np.float32))
    assert_same_f32(out[1:], np.full((W - 1, 2), -0.0, np.float32), "padding times negative alpha is -0")
    out, _ = _run_rs(orc, W, dims, grads, 0.5, True, old=np.full((W, 2), -0.0, np.float32))
    assert_same_f32(out[1:], np.zeros((W - 1, 2), np.float32), "accumulate onto padding: -0 + +0")
    assert_same_f32(out[0], np.array([6.0, -2.0], np.float32), "accumulate real row")


def pin_ag_identity(orc, seed=13):
    """AG(shard(x)) == x bitwise, with shard(x) built by torch.chunk and every
    padding position holding a NaN sentinel that must never reach an output."""
    rng = np.random.default_rng(seed)
    sentinel = np.uint16(0x7FC1)
    for W, dims in ((4, [(1000, 64), (64, 1), (333, 17), (7, 5), (4096, 1), (129, 128)]),
                    (3, [(1, 1), (2, 7), (5, 3)]), (8, [(3, 2), (9, 9)])):
        R, o, S = orc.geometry(W, dims)
        stride = S + 5
        xs = [rng.integers(0, 0x7F00, size=(d, k), dtype=np.uint16) for d, k in dims]
        slots = np.full((W, stride), sentinel, dtype=np.uint16)
        for p, x in enumerate(xs):
            for r, ch in enumerate(torch.chunk(torch.from_numpy(x.astype(np.int32)), W)):
                flat = ch.numpy().astype(np.uint16).reshape(-1)
                slots[r, o[p]:o[p] + flat.size] = flat
        full = orc.ag(W, dims, slots)
        for p, x in enumerate(xs):
            assert_same_u16(full[p], x.reshape(-1), f"AG(shard(x)) W={W} p={p}")
            assert not (full[p] == sentinel).any()


def pin_window_matches_full(orc, seed=17):
    """The windowed entry point used for sampled checks agrees with the full one."""
    rng = np.random.default_rng(seed)
    W, dims = 4, [(333, 17), (7, 5)]
    grads = _grads(W, dims, rng)
    R, o, S = orc.geometry(W, dims)
    old = rng.standard_normal((W, S)).astype(np.float32)
    for acc in (False, True):
        full = old.copy()
        orc.rs(W, dims, grads, 0.25, acc, full)
        for p, (d, k) in enumerate(dims):
            for r in range(W):
                v = orc.valid_rows(d, R[p], r)
                for (i0, i1) in ((0, R[p]), (1, max(1, v)), (max(0, v - 1), R[p])):
                    lo, hi = i0 * k, i1 * k
                    nv = max(0, min(hi, v * k) - lo)
                    srcs = [grads[p][u][r * R[p] * k + lo: r * R[p] * k + lo + nv] for u in range(W)]
                    win = orc.rs_window(srcs, nv, (hi - lo) - nv, 0.25, acc, old[r, o[p] + lo:o[p] + hi])
                    assert_same_f32(win, full[r, o[p] + lo:o[p] + hi], f"window p={p} r={r} [{i0},{i1})")


def _cast_patterns(rng) -> np.ndarray:
    """binary32 bit patterns: every sign and exponent with the mantissas that
    decide a rounding (0, ties with even and odd kept part, one below and one
    above a tie, all ones), plus random patterns."""
    mants = np.array([0x000000, 0x000001, 0x007FFF, 0x008000, 0x008001, 0x00FFFF, 0x010000, 0x017FFF, 0x018000,
                      0x018001, 0x3F8000, 0x7F8000, 0x7FFFFF, 0x7F7FFF, 0x400000, 0x408000, 0x7E8000, 0x7F0000],
                     dtype=np.uint32)
    se = np.arange(512, dtype=np.uint32) << np.uint32(23)
    structured = (se[:, None] | mants[None, :]).reshape(-1)
    randoms = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([structured, randoms])


def pin_cast_vs_torch(orc, seed=19):
    """The fp32 -> bf16 rounding against torch's round-to-nearest-even cast,
    bit for bit (NaN by class)."""
    bits = _cast_patterns(np.random.default_rng(seed))
    x = bits.view(np.float32)
    got = np.concatenate(orc.ag_cast(1, [(x.size, 1)], x.reshape(1, -1)))
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    gnan = (got & 0x7F80) == 0x7F80
    gnan &= (got & 0x7F) != 0
    wnan = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    assert (gnan == wnan).all(), "NaN class differs"
    bad = (got != want) & ~wnan
    assert not bad.any(), f"{int(bad.sum())} casts differ; first input 0x{bits[bad][0]:08x}"
    for v, w in ((1.0, 0x3F80), (-2.0, 0xC000), (float("inf"), 0x7F80), (0.0, 0x0000), (-0.0, 0x8000)):
        assert orc.f32_to_bf16(v) == w, v


def pin_ag_cast_identity(orc, seed=23):
    """Mixed-precision placement: AG_cast(shard(x)) == bf16(x) for x in fp32,
    shards built by torch.chunk, NaN in every padding position."""
    rng = np.random.default_rng(seed)
    for W, dims in ((4, [(1000, 64), (64, 1), (333, 17), (7, 5), (129, 128)]), (3, [(1, 1), (5, 3)]),
                    (8, [(9, 9), (3, 2)])):
        R, o, S = orc.geometry(W, dims)
        xs = [rng.standard_normal((d, k)).astype(np.float32) * np.float32(10.0 ** rng.integers(-3, 3))
              for d, k in dims]
        slots = np.full((W, S + 3), np.nan, dtype=np.float32)
        for p, x in enumerate(xs):
            for r, ch in enumerate(torch.chunk(torch.from_numpy(x), W)):
                flat = ch.numpy().reshape(-1)
                slots[r, o[p]:o[p] + flat.size] = flat
        full = orc.ag_cast(W, dims, slots)
        for p, x in enumerate(xs):
            want = torch.from_numpy(x.reshape(-1).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert_same_u16(full[p], want, f"AG_cast(shard(x)) W={W} p={p}")


def pin_orders_closed_form(orc):
    """Hand-worked values of the Section 4.3 orders (1.0 and 2^-24 terms):
    * W=4, one node, destination 0 holding 1.0: the three staged 2^-24 add
      exactly to 3*2^-24, then 1 + 3*2^-24 is 1.5 ulp: ties to even, 1 + 2^-22;
      destinations 1..3 start from 1.0 and every +2^-24 ties back to 1.0.
    * W=4 in nodes of 2, rank 0 holding 1.0: node 0 gives 1.0 (whichever rank
      is last), node 1 gives 2^-23, the sum 1 + 2^-23 is exact.
    * W=8 in nodes of 4: destination 0 (node 0's own rank is 0, added last):
      node 0 = 1 + 3*2^-24 -> 1 + 2^-22, node 1 = 4*2^-24 = 2^-22, total
      1 + 2^-21; destination 1 (rank 0 comes first): node 0 = 1.0, total 1 + 2^-22.
    * W=8, one node, destination 3 holding 1.0: 7*2^-24 + 1 is 3.5 ulp: 1 + 2^-21."""
    big, small = f32_to_bf16_bits([1.0])[0], f32_to_bf16_bits([U])[0]

    def run(W, holder, order, L=0):
        g = [[np.array([big if u == holder else small] * W, np.uint16) for u in range(W)]]
        out = np.zeros((W, 1), np.float32)
        orc.rs_ex(W, [(W, 1)], g, 1.0, False, out, order, L)
        return out.reshape(-1)

    e = np.float32
    assert_same_f32(run(4, 0, "staged"), np.array([1 + 2 ** -22, 1, 1, 1], e), "staged W=4")
    assert_same_f32(run(4, 0, "nodes", 2), np.full(4, 1 + 2 ** -23, e), "nodes W=4 L=2")
    got = run(8, 0, "nodes", 4)
    assert_same_f32(got[:2], np.array([1 + 2 ** -21, 1 + 2 ** -22], e), "nodes W=8 L=4")
    assert_same_f32(run(8, 3, "staged")[3:4], np.array([1 + 2 ** -21], e), "staged W=8 dest 3")
    assert_same_f32(run(8, 0, "nodes", 8), run(8, 0, "staged"), "nodes with L = W is the one-node order")
    assert_same_f32(run(8, 0, "nodes", 1), run(8, 0, "rank"), "nodes of one rank is rank order")


def pin_tree_closed_form(orc):
    """Hand-worked values of the pairwise (tree) order, 1.0 and U = 2^-24 terms
    listed in rank order (near 1.0 one ulp is 2^-23, so U is half an ulp):
    * W=3 [1,U,U]: (1+U)+U, each a tie back to 1: 1.0 (the odd value is
      added last, as in rank order); [U,U,1]: 2U+1 = 1 + 2^-23.
    * W=4 [1,U,U,U]: (1+U) = 1, (U+U) = 2U, 1 + 2U = 1 + 2^-23 exact
      (rank order gives 1.0).
    * W=5 [1,U,U,U,U]: 1, 2U, U -> 1 + 2^-23, U -> 1 + 1.5 ulp, tie to even:
      1 + 2^-22.
    * W=6 [1,0,U,U,0,0]: 1, 2U, 0 -> 1 + 2^-23, 0 -> 1 + 2^-23 (halving the
      ranks 3 | 3 would give ((1+0)+U) + ((U+0)+0) = 1.0).
    * W=7 [1,U,U,U,U,U,U]: 1, 2U, 2U, U -> 1 + 2^-23, 3U -> 1 + 2.5 ulp,
      tie to even: 1 + 2^-22.
    * W=8 [1,U x 7]: 1, 2U, 2U, 2U -> 1 + 2^-23, 4U -> 1 + 3 * 2^-23 exact.
    * W=16 [1,U x 15]: 1, 2U x 7 -> 1 + 2^-23, 4U x 3 -> 1 + 3 * 2^-23, 8U
      -> 1 + 7 * 2^-23 exact."""
    one, u = 1.0, U

    def run(vals):
        W = len(vals)
        bits = f32_to_bf16_bits(np.array(vals, np.float32))
        g = [[np.array([bits[q]] * W, np.uint16) for q in range(W)]]
        out = np.zeros((W, 1), np.float32)
        orc.rs_ex(W, [(W, 1)], g, 1.0, False, out, "tree", 0)
        return out.reshape(-1)

    cases = [([one, u, u], 1.0), ([u, u, one], 1 + 2 ** -23), ([one, u, u, u], 1 + 2 ** -23),
             ([one] + [u] * 4, 1 + 2 ** -22), ([one, 0.0, u, u, 0.0, 0.0], 1 + 2 ** -23),
             ([one] + [u] * 6, 1 + 2 ** -22), ([one] + [u] * 7, 1 + 3 * 2 ** -23),
             ([one] + [u] * 15, 1 + 7 * 2 ** -23)]
    for vals, want in cases:
        W = len(vals)
        assert_same_f32(run(vals), np.full(W, want, np.float32), f"tree W={W} {vals[:3]}...")
    assert_same_f32(run([one, u]), np.full(2, 1.0, np.float32), "tree of two is one add")


def pin_orders_brute_force(orc, seed=29):
    from oracle import brute
    rnd = random.Random(seed)
    rng = np.random.default_rng(seed)
    for c in range(32):
        W = rnd.choice([1, 2, 3, 4, 5, 6, 7, 8, 11, 13])
        order = rnd.choice(["rank", "staged", "nodes", "tree"])
        L = rnd.choice([d for d in range(1, W + 1) if W % d == 0]) if order == "nodes" else 0
        dims = [(rnd.choice([1, 2, W, W + 1, 2 * W + 1]), rnd.choice([1, 3, 4])) for _ in range(rnd.randint(1, 3))]
        f32 = rnd.random() < 0.4
        grads = [[(rng.standard_normal(d * k).astype(np.float32) if f32 else _rand_bits(rng, d * k))
                  for _ in range(W)] for d, k in dims]
        alpha, acc = rnd.choice([1.0, 0.25, -3.0]), rnd.random() < 0.5
        _, _, S = orc.geometry(W, dims)
        old = rng.standard_normal((W, S)).astype(np.float32)
        out = old.copy()
        orc.rs_ex(W, dims, grads, alpha, acc, out, order, L)
        want = brute.reduce_scatter_ordered(W, dims, grads, alpha, acc, old, order, L)
        assert_same_f32(out, want, f"ordered brute case {c}: W={W} {order} L={L} f32={f32}")


def pin_orders_exact_and_bounded(orc, seed=37):
    """Every order: integer inputs give the exact sum; normal inputs stay
    within gamma_{W+1} (|alpha| sum |G| + |old|) of the fp64 sum (the tree
    order within gamma_{ceil(log2 W)}, its depth) and within 1e-6 of the
    rank-order result in the max-norm (the reordered-variant tolerance); the
    rank order reproduces the original oracle bit for bit."""
    rng = np.random.default_rng(seed)
    for W, L in ((8, 4), (16, 4), (32, 8), (6, 3)):
        dims = [(4 * W + 3, 9), (W, 1)]
        ints = [[rng.integers(-128, 129, size=d * k) for _ in range(W)] for d, k in dims]
        gi = [[f32_to_bf16_bits(x.astype(np.float32)) for x in per] for per in ints]
        R, o, S = orc.geometry(W, dims)
        for order in ("staged", "nodes", "tree"):
            out = np.zeros((W, S), np.float32)
            orc.rs_ex(W, dims, gi, 0.5, False, out, order, L if order == "nodes" else 0)
            for p, (d, k) in enumerate(dims):
                exact = sum(ints[p][u] for u in range(W)).astype(np.float64) * 0.5
                flat = np.concatenate([out[r, o[p]:o[p] + R[p] * k] for r in range(W)])[:d * k]
                assert_same_f32(flat, exact.astype(np.float32), f"integer {order} W={W}")
        g = [[_rand_bits(rng, d * k) for _ in range(W)] for d, k in dims]
        ref = np.zeros((W, S), np.float32)
        orc.rs(W, dims, g, 1.0, False, ref)
        rank_ex = np.zeros((W, S), np.float32)
        orc.rs_ex(W, dims, g, 1.0, False, rank_ex, "rank", 0)
        assert_same_f32(rank_ex, ref, "rank order of the ordered oracle == original oracle")
        gamma = (W + 1) * U / (1 - (W + 1) * U)
        depth = (W - 1).bit_length()
        for order in ("staged", "nodes", "tree"):
            out = np.zeros((W, S), np.float32)
            orc.rs_ex(W, dims, g, 1.0, False, out, order, L if order == "nodes" else 0)
            bound = gamma if order != "tree" else depth * U / (1 - depth * U)
            for p, (d, k) in enumerate(dims):
                vals = np.stack([bf16_bits_to_f32(g[p][u]).astype(np.float64) for u in range(W)])
                got = np.concatenate([out[r, o[p]:o[p] + R[p] * k] for r in range(W)])[:d * k]
                assert (np.abs(got - vals.sum(0)) <= bound * np.abs(vals).sum(0) + 1e-45).all(), order
                rk = np.concatenate([ref[r, o[p]:o[p] + R[p] * k] for r in range(W)])[:d * k]
                assert np.abs(got - rk).max() <= 1e-6 * np.abs(rk).max(), f"{order} vs rank order"


def pin_f32_grads_chunk_cat(orc, seed=41):
    """fp32 gradients (b_grad = 4): torch._chunk_cat's pack of fp32 tensors
    then a rank-ordered fp32 sum, against the oracle."""
    rng = np.random.default_rng(seed)
    for W, dims in ((4, [(333, 17), (7, 5), (64, 1)]), (3, [(5, 2), (1, 1)])):
        grads = [[rng.standard_normal(d * k).astype(np.float32) for _ in range(W)] for d, k in dims]
        _, _, S = orc.geometry(W, dims)
        packs = []
        for u in range(W):
            ts = [torch.from_numpy(grads[p][u].reshape(d, k)) for p, (d, k) in enumerate(dims)]
            t = torch.empty(W, S, dtype=torch.float32)
            torch._chunk_cat(ts, dim=0, num_chunks=W, out=t)
            packs.append(t)
        acc = packs[0].clone()
        for u in range(1, W):
            acc = acc + packs[u]
        want = (acc * torch.tensor(0.5, dtype=torch.float32)).numpy()
        out = np.zeros((W, S), np.float32)
        orc.rs_ex(W, dims, grads, 0.5, False, out, "rank", 0)
        assert_same_f32(out, want, f"fp32 grads W={W}")


ALL_PINS = [pin_golden, pin_slot_sizes, pin_torch_chunk, pin_chunk_cat, pin_brute_force, pin_integer_exact,
            pin_order_probe, pin_fp64_bound, pin_special_values, pin_ag_identity, pin_window_matches_full,
            pin_cast_vs_torch, pin_ag_cast_identity, pin_orders_closed_form, pin_tree_closed_form,
            pin_orders_brute_force,
            pin_orders_exact_and_bounded, pin_f32_grads_chunk_cat]
