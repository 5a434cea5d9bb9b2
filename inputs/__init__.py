"""Seeded synthetic workloads for the reshard, shared by the tests and the benchmark.

This module only DEFINES workloads (global shapes, meshes, placements, dtypes,
value distributions, seeds) and draws the global tensors' values.  It holds
none of the reshard's arithmetic: it never splits a tensor into shards, never
intersects boxes and never copies shard data.  Consumers scatter the global
tensor into source shards with their own layout rule (the tests use the CPU
oracle's, the benchmark uses the library's).

Placements are strings: "R" = Replicate, "S<d>" = Shard(d).  Meshes are tuples
of sizes, ranks are row-major coordinates.

The five workloads follow the shapes named for this reshard:
  1 worked_example  the 8x8 example of the Reshard collective write-ups
                    (Shard(0) on 2 ranks -> Shard(1) on 4 ranks);
  2 ffn_up          a dense FFN up-projection 14336x4096, (DP2,TP4) -> (DP4,TP2);
  3 hybridflow      a Llama-70B-shaped stack (8 layers of gate/up/down), training
                    TP8 -> generation TP2 x micro-DP4 with strided generation ranks
                    (HybridFlow's 3D-HybridEngine layout);
  4 uneven_stress   60 random tensors with non-divisible dims and random meshes;
  5 moe_refit       a DeepSeek-v3-shaped MoE layer (256 experts) plus the
                    attention/norm weights that go through gather-and-broadcast.
Each full-size workload has a reduced twin with the same meshes and placements
and ragged, much smaller shapes, sized for the CPU oracle.
"""
from __future__ import annotations

import dataclasses
import math
import random
from typing import Sequence

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32,
          "u8": torch.uint8, "fp64": torch.float64}
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4, "u8": 1, "fp64": 8}


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    """One global tensor and its source/destination DTensor layouts."""
    name: str
    global_shape: tuple
    dtype: str
    src_mesh: tuple
    src_placements: tuple
    dst_mesh: tuple
    dst_placements: tuple
    init: tuple = ("normal", 0.0, 0.02)   # ("normal", mean, std) | ("uniform", lo, hi) | ("bits",)
    seed: int = 0
    path: str = "reshard"                 # "reshard" | "gather_broadcast"

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def numel(self) -> int:
        return math.prod(self.global_shape)

    @property
    def global_bytes(self) -> int:
        return self.numel * self.elem_bytes

    @property
    def n_src(self) -> int:
        return math.prod(self.src_mesh)

    @property
    def n_dst(self) -> int:
        return math.prod(self.dst_mesh)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tensors: tuple
    note: str = ""

    @property
    def global_bytes(self) -> int:
        return sum(t.global_bytes for t in self.tensors)


# ----------------------------------------------------------------------------- values
def global_tensor(spec: TensorSpec, device: str | torch.device = "cpu") -> torch.Tensor:
    """The seeded global tensor of one spec, drawn on ``device``.

    Values are drawn in fp32 from the spec's distribution and cast once to the
    dtype ("bits" draws raw bit patterns, NaN payloads and -0 included).  The
    same seed gives the same bytes on the CPU every time; a CUDA device uses
    its own generator (deterministic, but different numbers from the CPU's).
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(spec.seed))
    shape = tuple(int(s) for s in spec.global_shape)
    dt = DTYPES[spec.dtype]
    kind = spec.init[0]
    if kind == "bits":
        nbits = 8 * ELEM_BYTES[spec.dtype]
        if nbits == 8:
            return torch.randint(0, 256, shape, generator=g, device=dev, dtype=torch.uint8)
        itype = {16: torch.int16, 32: torch.int32, 64: torch.int64}[nbits]
        info = torch.iinfo(itype)
        raw = torch.randint(info.min, info.max, shape, generator=g, device=dev, dtype=itype)
        return raw.view(dt)
    if kind == "normal":
        x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        x.mul_(float(spec.init[2])).add_(float(spec.init[1]))
    elif kind == "uniform":
        x = torch.rand(shape, generator=g, device=dev, dtype=torch.float32)
        lo, hi = float(spec.init[1]), float(spec.init[2])
        x.mul_(hi - lo).add_(lo)
    else:
        raise ValueError(f"unknown init {spec.init!r}")
    if dt == torch.uint8:
        return (x * 255).to(torch.uint8)
    return x.to(dt)


# ----------------------------------------------------------------------------- workloads
def worked_example() -> Workload:
    t = TensorSpec("w8x8", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",),
                   init=("uniform", -1.0, 1.0), seed=1)
    return Workload("worked_example_8x8", (t,),
                    "8x8 bf16, Shard(0) on 2 ranks -> Shard(1) on 4 ranks")


def ffn_up(scale: int = 1) -> Workload:
    rows, cols = (14336, 4096) if scale == 1 else (1433, 409)
    t = TensorSpec("ffn_up", (rows, cols), "bf16", (2, 4), ("R", "S0"), (4, 2), ("R", "S1"),
                   seed=2)
    return Workload("ffn_up_14336x4096" if scale == 1 else "ffn_up_reduced", (t,),
                    "(DP2,TP4)(R,S0) -> (DP4,TP2)(R,S1)")


def hybridflow(layers: int = 8, hidden: int = 8192, ffn: int = 28672,
               down_dim: int = 0, name: str | None = None) -> Workload:
    """Training TP8 Shard(out) -> generation (TP2 outer, micro-DP4) (S0, R).

    Weights are [out, in]; gate/up are [ffn, hidden] and down is [hidden, ffn].
    ``down_dim=1`` gives the row-parallel alternative (down sharded on its
    input dim) instead of the literal "output dim" reading.
    """
    ts = []
    for l in range(layers):
        for k, shape in (("gate", (ffn, hidden)), ("up", (ffn, hidden)), ("down", (hidden, ffn))):
            d = down_dim if k == "down" else 0
            ts.append(TensorSpec(f"layer{l}.{k}", shape, "bf16", (8,), (f"S{d}",), (2, 4),
                                 (f"S{d}", "R"), seed=3000 + len(ts)))
    if name is None:
        name = "hybridflow_llama70b_8layers" if (layers, hidden, ffn) == (8, 8192, 28672) \
            else f"hybridflow_{layers}x{ffn}x{hidden}"
    return Workload(name, tuple(ts), "TP8 (S0) -> (TP2,DP4) (S0,R), strided generation ranks")


def hybridflow_reduced() -> Workload:
    return hybridflow(layers=2, hidden=819, ffn=2867, name="hybridflow_reduced")


def moe_refit(experts: int = 256, ffn: int = 2048, hidden: int = 7168, qkv_rows: int = 21504,
              n_qkv: int = 3, n_norm: int = 6, name: str | None = None) -> Workload:
    """DeepSeek-v3-shaped MoE refit slice plus its gather-and-broadcast weights.

    Experts: gate/up [E, ffn, hidden], down [E, hidden, ffn]; source mesh
    (PP1, EP16, TP2) with (R, Shard(experts), Shard(ffn dim)); destination
    mesh (DP2, TP8) with (R, Shard(ffn dim)).  Attention and norm weights:
    source (R, R, Shard(0)) -> destination (R, Shard(0)), executed on the
    gather-and-broadcast path.
    """
    src_mesh, dst_mesh = (1, 16, 2), (2, 8)
    ts = [
        TensorSpec("experts.gate", (experts, ffn, hidden), "bf16", src_mesh, ("R", "S0", "S1"),
                   dst_mesh, ("R", "S1"), seed=5001),
        TensorSpec("experts.up", (experts, ffn, hidden), "bf16", src_mesh, ("R", "S0", "S1"),
                   dst_mesh, ("R", "S1"), seed=5002),
        TensorSpec("experts.down", (experts, hidden, ffn), "bf16", src_mesh, ("R", "S0", "S2"),
                   dst_mesh, ("R", "S2"), seed=5003),
    ]
    for i in range(n_qkv):
        ts.append(TensorSpec(f"attn.qkv{i}", (qkv_rows, hidden), "bf16", src_mesh,
                             ("R", "R", "S0"), dst_mesh, ("R", "S0"), seed=5100 + i,
                             path="gather_broadcast"))
    for i in range(n_norm):
        ts.append(TensorSpec(f"norm{i}", (hidden,), "bf16", src_mesh, ("R", "R", "S0"),
                             dst_mesh, ("R", "S0"), seed=5200 + i, path="gather_broadcast"))
    if name is None:
        name = "moe_refit_deepseekv3_256x2048x7168" if experts == 256 else f"moe_refit_{experts}"
    return Workload(name, tuple(ts),
                    "(PP1,EP16,TP2)(R,S0,Sffn) -> (DP2,TP8)(R,Sffn); attn/norm via gather-broadcast")


def moe_refit_reduced() -> Workload:
    return moe_refit(experts=19, ffn=203, hidden=71, qkv_rows=213, n_qkv=1, n_norm=2,
                     name="moe_refit_reduced")


def _random_mesh(rng: random.Random, ndim_tensor: int):
    while True:
        mnd = rng.randint(1, 3)
        mesh = tuple(rng.randint(1, 64) for _ in range(mnd))
        if math.prod(mesh) <= 64:
            break
    pl = tuple("R" if rng.random() < 1.0 / 3.0 else f"S{rng.randrange(ndim_tensor)}"
               for _ in mesh)
    return mesh, pl


def _replication(mesh, pl) -> int:
    return math.prod(m for m, p in zip(mesh, pl) if p == "R")


def uneven_stress(n: int = 60, seed: int = 20261202, max_dim: int = 9001,
                  max_numel: int = 1 << 27, max_bytes: int = 4 << 30,
                  name: str | None = None) -> Workload:
    """Random non-divisible tensors and meshes (rejection-sampled, seeded).

    ndim uniform in {2, 3}; each dim uniform in [1, max_dim]; redrawn until
    numel <= max_numel.  Each mesh has 1-3 dims of size 1-64 (redrawn until at
    most 64 ranks); each mesh dim is Replicate with probability 1/3, else
    Shard(d) with d uniform.  A draw whose source + destination + full-tensor
    scratch would exceed max_bytes is redrawn.  dtype uniform over
    {fp32, bf16, fp16}; values uniform(-1, 1).
    """
    rng = random.Random(seed)
    ts = []
    while len(ts) < n:
        nd = rng.choice((2, 3))
        while True:
            shape = tuple(rng.randint(1, max_dim) for _ in range(nd))
            if math.prod(shape) <= max_numel:
                break
        dtype = rng.choice(("fp32", "bf16", "fp16"))
        sm, sp = _random_mesh(rng, nd)
        dm, dp = _random_mesh(rng, nd)
        gb = math.prod(shape) * ELEM_BYTES[dtype]
        if gb * (_replication(sm, sp) + _replication(dm, dp) + 1) > max_bytes:
            continue
        ts.append(TensorSpec(f"stress{len(ts)}", shape, dtype, sm, sp, dm, dp,
                             init=("uniform", -1.0, 1.0), seed=seed + len(ts)))
    return Workload(name or f"uneven_stress_{n}", tuple(ts), "random meshes, torch.chunk splits")


def uneven_stress_reduced() -> Workload:
    return uneven_stress(n=60, seed=20261202, max_dim=61, max_numel=1 << 14,
                         name="uneven_stress_reduced")


FULL = {
    1: worked_example,
    2: ffn_up,
    3: hybridflow,
    4: uneven_stress,
    5: moe_refit,
}

REDUCED = {
    1: worked_example,
    2: lambda: ffn_up(scale=0),
    3: hybridflow_reduced,
    4: uneven_stress_reduced,
    5: moe_refit_reduced,
}


def workload(config: int, reduced: bool = False) -> Workload:
    return (REDUCED if reduced else FULL)[int(config)]()


def replication_factor(mesh: Sequence[int], placements: Sequence[str]) -> int:
    """How many ranks hold each element (product of the Replicate mesh dims)."""
    return _replication(mesh, placements)
