"""Seeded synthetic inputs for the FSDP2 reduce-scatter / all-gather path.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It holds workload shapes and random-number recipes only: no
sharding geometry, no summation, no placement.  Anything that depends on the
dim-0 shard layout (row counts, offsets, slot sizes) is computed by the
caller, each side with its own code.

Shapes follow the five workloads the TIDE paper ("The Endgame of FSDP
Communication") trains or replays: a toy group, one Llama-3.1 8B / 70B
decoder block, one Wan2.2-style DiT block and one Qwen3-30B-A3B-style MoE
layer (Section 7.1).  The paper trains real models on public C4; here only
the layer shapes stand in, with i.i.d. normal gradients (no weights, no
dataset).

Recipe (all configurable pieces are stated, nothing is hidden):

* gradient of parameter ``p`` on virtual rank ``u`` of workload ``c``: a
  ``torch.Generator`` on the target device seeded with
  ``1_000_003 * c + 4099 * u + p``; ``x = randn(numel) * sigma`` in fp32; if
  the workload has outliers, ``mask = rand(numel) < rate`` from the same
  generator and ``x[mask] *= scale`` in fp32; finally a round-to-nearest-even
  cast to bf16.
* initial fp32 shard of destination rank ``r`` (accumulate mode):
  seed ``1_000_003 * c + 500_009 + r``, ``randn * 1e-3`` in fp32.
* bf16 parameter shard slot of rank ``r`` (all-gather input):
  seed ``1_000_003 * c + 700_001 + r``, ``randn * 0.02`` cast to bf16.

Each virtual rank's gradients live in one contiguous bf16 arena with every
parameter starting on a 256-byte boundary (the caching-allocator alignment a
real FSDP2 gradient would have).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from math import prod
from typing import List, Sequence, Tuple

import torch

ARENA_ALIGN_BYTES = 256


@dataclass(frozen=True)
class Workload:
    """One synthetic gradient group.

    ``alpha`` is the scale the benchmark uses; parity tests run both 1 and
    1/world on every workload.
    """

    index: int                      # 1-based workload number, part of every seed
    name: str
    world: int                      # W virtual ranks
    names: Tuple[str, ...]
    shapes: Tuple[Tuple[int, ...], ...]
    sigma: float
    outlier_rate: float = 0.0
    outlier_scale: float = 1.0
    alpha: float = 1.0
    accumulate: bool = False
    notes: str = ""

    @property
    def num_params(self) -> int:
        return len(self.shapes)

    def numels(self) -> List[int]:
        return [prod(s) for s in self.shapes]

    def total_numel(self) -> int:
        """N: unpadded elements of one gradient set."""
        return sum(self.numels())

    def dim0_rownumel(self) -> List[Tuple[int, int]]:
        """(dim0, product of trailing dims) per parameter; 1-d tensors have row_numel 1."""
        out = []
        for s in self.shapes:
            if len(s) == 0:
                raise ValueError("0-d parameters are not dim-0 shardable")
            out.append((s[0], prod(s[1:]) if len(s) > 1 else 1))
        return out


def _llama_block(idx, name, hidden, kv, ffn, world, accumulate, sigma, outlier_rate=0.0, outlier_scale=1.0):
    names = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj",
             "input_layernorm", "post_attention_layernorm")
    shapes = ((hidden, hidden), (kv, hidden), (kv, hidden), (hidden, hidden),
              (ffn, hidden), (ffn, hidden), (hidden, ffn), (hidden,), (hidden,))
    return Workload(idx, name, world, names, shapes, sigma, outlier_rate, outlier_scale,
                    alpha=1.0, accumulate=accumulate)


def _wan_block():
    d, f = 5120, 13824
    names, shapes = [], []
    for attn in ("self_attn", "cross_attn"):
        for m in ("q", "k", "v", "o"):
            names.append(f"{attn}.{m}")
            shapes.append((d, d))
    names += ["ffn.0", "ffn.2"]
    shapes += [(f, d), (d, f)]
    # The workload lists "norm/mod vectors [5120]" without a count; ten are
    # used here: q/k norms of both attentions (4) and six modulation slices.
    for attn in ("self_attn", "cross_attn"):
        for m in ("norm_q", "norm_k"):
            names.append(f"{attn}.{m}")
            shapes.append((d,))
    for i in range(6):
        names.append(f"modulation.{i}")
        shapes.append((d,))
    return Workload(4, "wan2.2_dit_block", 16, tuple(names), tuple(shapes), sigma=5e-4,
                    notes="10 norm/modulation vectors of [5120] assumed")


def _qwen3_moe_layer(experts=128, index=5, name="qwen3_30b_a3b_moe_layer"):
    names, shapes = [], []
    for e in range(experts):
        names += [f"experts.{e}.gate_proj", f"experts.{e}.up_proj", f"experts.{e}.down_proj"]
        shapes += [(768, 2048), (768, 2048), (2048, 768)]
    names += ["router", "q_proj", "k_proj", "v_proj", "o_proj"]
    shapes += [(128, 2048), (4096, 2048), (512, 2048), (512, 2048), (2048, 4096)]
    return Workload(index, name, 32, tuple(names), tuple(shapes), sigma=1e-3)


WORKLOADS: Tuple[Workload, ...] = (
    Workload(1, "toy", 4,
             ("w0", "b0", "w1", "w2", "b1", "w3"),
             ((1000, 64), (64,), (333, 17), (7, 5), (4096,), (129, 128)),
             sigma=1e-3, alpha=0.25),
    _llama_block(2, "llama3.1_8b_block", 4096, 1024, 14336, 8, False, 1e-3,
                 outlier_rate=1e-3, outlier_scale=100.0),
    _llama_block(3, "llama3.1_70b_block", 8192, 1024, 28672, 8, True, 1e-3),
    _wan_block(),
    _qwen3_moe_layer(),
)

# Reduced cases for profiler captures, which replay a kernel dozens of times
# and so want a few GB on the device at most: the Llama-3.1-8B block's
# attention projections and norms (~0.7 GB of gradients), and the MoE layer
# with 8 of its 128 experts (same W = 32 and shapes, 56.9 M elements per
# gradient set, 3.6 GB of gradients; its per-element traffic scales to the
# full layer).
PROFILE_CASES: Tuple[Workload, ...] = (
    Workload(6, "llama3.1_8b_attn", 8,
             ("q_proj", "k_proj", "v_proj", "o_proj", "input_layernorm", "post_attention_layernorm"),
             ((4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (4096,), (4096,)),
             sigma=1e-3, outlier_rate=1e-3, outlier_scale=100.0),
    _qwen3_moe_layer(experts=8, index=7, name="qwen3_moe_8experts"),
)

BY_NAME = {w.name: w for w in WORKLOADS + PROFILE_CASES}


def get(key) -> Workload:
    """Workload by 1-based index or by name."""
    if isinstance(key, int):
        return (WORKLOADS + PROFILE_CASES)[key - 1]
    return BY_NAME[key]


def grad_seed(w: Workload, u: int, p: int) -> int:
    return 1_000_003 * w.index + 4099 * u + p


def out_seed(w: Workload, r: int) -> int:
    return 1_000_003 * w.index + 500_009 + r


def slot_seed(w: Workload, r: int) -> int:
    return 1_000_003 * w.index + 700_001 + r


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_fp32(numel: int, seed: int, sigma: float, device="cpu",
                outlier_rate: float = 0.0, outlier_scale: float = 1.0) -> torch.Tensor:
    """randn * sigma in fp32, with optional Bernoulli outliers scaled in fp32."""
    g = _generator(seed, device)
    x = torch.randn(numel, generator=g, device=device, dtype=torch.float32)
    x.mul_(sigma)
    if outlier_rate > 0.0:
        mask = torch.rand(numel, generator=g, device=device, dtype=torch.float32) < outlier_rate
        x = torch.where(mask, x * outlier_scale, x)
    return x


def arena_offsets(numels: Sequence[int], elem_bytes: int = 2) -> Tuple[List[int], int]:
    """Element offsets of each tensor in an arena that starts every tensor on a
    256-byte boundary, and the arena's total element count."""
    step = ARENA_ALIGN_BYTES // elem_bytes
    offs, cur = [], 0
    for n in numels:
        offs.append(cur)
        cur += (n + step - 1) // step * step
    return offs, max(cur, step)


@dataclass
class GradSets:
    """W gradient sets: ``arenas[u]`` is rank u's bf16 arena, ``views[u][p]`` the
    parameter's tensor (original shape) inside it."""

    workload: Workload
    arenas: List[torch.Tensor]
    views: List[List[torch.Tensor]]
    offsets: List[int] = field(default_factory=list)

    def base_ptrs(self) -> List[List[int]]:
        """[p][u] data pointers."""
        W, P = self.workload.world, self.workload.num_params
        return [[self.views[u][p].data_ptr() for u in range(W)] for p in range(P)]


def make_grads(w: Workload, device="cpu", fill=None) -> GradSets:
    """Generate the W bf16 gradient sets of workload ``w`` on ``device``.

    ``fill`` (optional) replaces the normal recipe: a callable
    ``fill(u, p, numel, device) -> fp32 tensor`` used by special-value tests.
    """
    numels = w.numels()
    offs, total = arena_offsets(numels)
    arenas, views = [], []
    for u in range(w.world):
        arena = torch.zeros(total, dtype=torch.bfloat16, device=device)
        vs = []
        for p, (shape, n, o) in enumerate(zip(w.shapes, numels, offs)):
            if fill is None:
                x = normal_fp32(n, grad_seed(w, u, p), w.sigma, device, w.outlier_rate, w.outlier_scale)
            else:
                x = fill(u, p, n, device)
            arena[o:o + n].copy_(x.to(torch.bfloat16))
            vs.append(arena[o:o + n].view(shape))
        arenas.append(arena)
        views.append(vs)
    return GradSets(w, arenas, views, offs)


def make_out_init(w: Workload, stride: int, device="cpu") -> torch.Tensor:
    """fp32 [W, stride] initial shards for accumulate mode."""
    rows = [normal_fp32(stride, out_seed(w, r), 1e-3, device) for r in range(w.world)]
    return torch.stack(rows)


def make_slots(w: Workload, stride: int, device="cpu") -> torch.Tensor:
    """bf16 [W, stride] rank-major parameter shard slots (all-gather input)."""
    rows = [normal_fp32(stride, slot_seed(w, r), 0.02, device).to(torch.bfloat16) for r in range(w.world)]
    return torch.stack(rows)


def custom(world: int, shapes: Sequence[Tuple[int, ...]], sigma: float = 1e-3, index: int = 9,
           name: str = "custom", alpha: float = 1.0, accumulate: bool = False) -> Workload:
    """An ad-hoc workload (tests: ragged tails, tiny shapes, edge cases)."""
    shapes = tuple(tuple(s) for s in shapes)
    return Workload(index, name, world, tuple(f"t{i}" for i in range(len(shapes))), shapes,
                    sigma, alpha=alpha, accumulate=accumulate)
