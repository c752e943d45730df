"""Bit-level helpers shared by the tests: bf16 conversions, bitwise comparison
with NaN-class matching, and the golden-fixture parser."""
from __future__ import annotations

import os
from typing import Dict

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def tensor_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 torch tensor (any device) as a flat uint16 numpy array."""
    return t.detach().reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)


def assert_same_f32(actual, expected, what=""):
    """Bitwise equality of fp32 arrays; any NaN matches any NaN (payloads may differ)."""
    a = np.ascontiguousarray(actual, dtype=np.float32).reshape(-1)
    e = np.ascontiguousarray(expected, dtype=np.float32).reshape(-1)
    assert a.shape == e.shape, f"{what}: shape {a.shape} != {e.shape}"
    an, en = np.isnan(a), np.isnan(e)
    bad = (a.view(np.uint32) != e.view(np.uint32)) & ~(an & en)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {a.size} differ; first at {i}: "
                             f"{a[i]!r} (0x{a.view(np.uint32)[i]:08x}) vs {e[i]!r} (0x{e.view(np.uint32)[i]:08x})")


def assert_same_u16(actual, expected, what=""):
    a = np.asarray(actual, dtype=np.uint16).reshape(-1)
    e = np.asarray(expected, dtype=np.uint16).reshape(-1)
    assert a.shape == e.shape, f"{what}: shape {a.shape} != {e.shape}"
    bad = a != e
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {a.size} differ; first at {i}: 0x{a[i]:04x} vs 0x{e[i]:04x}")


def assert_same_bf16(actual, expected, what=""):
    """Bitwise equality of bf16 bit patterns; any NaN matches any NaN."""
    a = np.asarray(actual, dtype=np.uint16).reshape(-1)
    e = np.asarray(expected, dtype=np.uint16).reshape(-1)
    assert a.shape == e.shape, f"{what}: shape {a.shape} != {e.shape}"
    an = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    en = ((e & 0x7F80) == 0x7F80) & ((e & 0x7F) != 0)
    bad = (a != e) & ~(an & en)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {a.size} differ; first at {i}: 0x{a[i]:04x} vs 0x{e[i]:04x}")


def parse_golden(name: str) -> Dict:
    """Parse a hand-written fixture under tests/golden/."""
    out: Dict = {"params": [], "grad": {}, "expect": {}, "old": {}, "expect_acc": {}, "slot": {}, "full": {}}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                head, vals = line.split(":", 1)
                key = head.split()
                nums = [float("nan") if v == "nan" else float(v) for v in vals.split()]
                kind = key[0]
                if kind == "grad":
                    out["grad"][(key[1], int(key[2]))] = nums
                elif kind in ("expect", "old", "expect_acc", "slot"):
                    out[kind][int(key[1])] = nums
                elif kind == "full":
                    out["full"][key[1]] = nums
                continue
            key = line.split()
            if key[0] == "world":
                out["world"] = int(key[1])
            elif key[0] == "param":
                out["params"].append((key[1], int(key[2]), int(key[3])))
            elif key[0] == "alpha":
                out["alpha"] = float(key[1])
            elif key[0] == "stride":
                out["stride"] = int(key[1])
    return out
