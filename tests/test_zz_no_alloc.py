"""The allocation-free gather-and-broadcast entry point (needs a GB300).

gather_broadcast_execute_static serves callers that cannot call cudaMalloc (an
engine whose pool already owns the device memory, a path that must not trigger
the synchronisation an allocation can cause, a plugin given only its buffers):
its scratch and tables live in the library's static device arrays.  Here it is
called through the C ABI on several plans in a row, and every result must equal,
byte for byte, both the oracle's destination shards and what
gather_broadcast_execute produces with a caller-owned scratch.  The plans cover
an attention-like weight, a ragged 3-D tensor with empty shards, rows at 2-byte
alignment (the TMA-staged realigning kernel, which takes its work from the
library's static work queue) and a plan that leaves a source replica and a
destination rank out (NULL pointers for both).  This file is collected last so
that a failure here cannot hide failures elsewhere; it also passes when run alone.
"""
import math

import numpy as np
import pytest
import torch

import dtensor_reshard_gb300 as rs
from inputs import TensorSpec, global_tensor

pytestmark = pytest.mark.gpu

SPECS = [
    # attention-like weight: (PP1, EP16, TP2) (R, R, S0) -> (DP2, TP8) (R, S0), 12.6 MB
    TensorSpec("qkv_small", (879, 7168), "bf16", (1, 16, 2), ("R", "R", "S0"), (2, 8),
               ("R", "S0"), init=("bits",), seed=91),
    # ragged 3-D fp32 with empty shards and nested sharding, 2 MB
    TensorSpec("ragged3d", (37, 61, 229), "fp32", (2, 3), ("S2", "S0"), (5, 2), ("S1", "S2"),
               init=("bits",), seed=92),
    # bf16 rows of 4098 / 4096 bytes at 2-byte offsets in the full tensor: the gather and
    # the slice go through the TMA-staged realigning kernel (one replica, long rows,
    # 2-byte accesses), 16.8 MB
    TensorSpec("odd_cols", (2048, 4097), "bf16", (2,), ("S1",), (3,), ("S0",),
               init=("bits",), seed=93),
]


def _plan(spec, src_gone=(), dst_gone=()):
    plan = rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                  spec.src_placements, spec.dst_mesh, spec.dst_placements)
    if src_gone or dst_gone:
        plan = rs.reshard_plan_exclude(plan, src_gone=src_gone, dst_gone=dst_gone)
    return plan


def _case(spec, dev, oracle, src_gone=(), dst_gone=()):
    plan = _plan(spec, src_gone, dst_gone)
    glob = global_tensor(spec)
    srcs, src_bytes = [], []
    # sources cut with the oracle's boxes, never with the library's
    for r, (off, shp) in enumerate(oracle.boxes(spec.global_shape, spec.src_mesh,
                                                spec.src_placements)):
        sl = tuple(slice(o, o + s) for o, s in zip(off, shp))
        shard = glob[sl].contiguous()
        src_bytes.append(shard.view(torch.uint8).reshape(-1).numpy() if shard.numel()
                         else np.zeros(0, np.uint8))
        srcs.append(None if r in src_gone else shard.to(dev))
    want = oracle.reshard(spec.global_shape, spec.elem_bytes, spec.src_mesh,
                          spec.src_placements, spec.dst_mesh, spec.dst_placements, src_bytes)

    def fresh_dsts():
        out = []
        for r in range(plan.n_dst):
            if r in dst_gone:
                out.append(None)
                continue
            d = torch.full((want[r].size,), 0xA5, dtype=torch.uint8, device=dev)
            out.append(d)
        return out
    return plan, srcs, fresh_dsts, want


def _check(dsts, want, dst_gone, what):
    for r, (d, w) in enumerate(zip(dsts, want)):
        if r in dst_gone:
            continue
        assert np.array_equal(d.cpu().numpy(), w), f"{what}: destination rank {r} differs"


def _caller_scratch_result(plan, srcs, fresh, dev):
    dsts = fresh()
    G = rs.reshard_plan_stats(plan)["global_bytes"]
    scratch = torch.empty(max(G, 1), dtype=torch.uint8, device=dev)
    rs.gather_broadcast_execute(plan, srcs, dsts, scratch, G)
    torch.cuda.synchronize()
    return dsts


def test_static_scratch_matches_oracle_and_caller_scratch_on_calls_in_a_row(oracle):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    dev = torch.device("cuda:0")
    cases = [_case(spec, dev, oracle) for spec in SPECS]
    expected = [_caller_scratch_result(plan, srcs, fresh, dev)
                for (plan, srcs, fresh, _) in cases]
    got = []
    for (plan, srcs, fresh, _) in cases:      # calls in a row on one stream
        dsts = fresh()
        rs.gather_broadcast_execute_static(plan, srcs, dsts)
        got.append(dsts)
    torch.cuda.synchronize()
    for spec, (_, _, _, want), ref, have in zip(SPECS, cases, expected, got):
        _check(have, want, (), f"{spec.name} static vs oracle")
        for a, b in zip(ref, have):
            assert torch.equal(a, b), f"{spec.name}: static and caller-scratch results differ"
    # and the first plan once more, after the later ones overwrote the shared arrays
    plan, srcs, fresh, want = cases[0]
    dsts = fresh()
    rs.gather_broadcast_execute_static(plan, srcs, dsts)
    torch.cuda.synchronize()
    _check(dsts, want, (), "qkv_small again")


def test_static_scratch_on_an_excluded_plan(oracle):
    """A plan that leaves a source replica and a destination rank out takes NULL for
    both, as gather_broadcast_execute does, and fills every other destination."""
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    dev = torch.device("cuda:0")
    spec = SPECS[0]
    src_gone, dst_gone = (3,), (5,)
    plan, srcs, fresh, want = _case(spec, dev, oracle, src_gone=src_gone, dst_gone=dst_gone)
    ref = _caller_scratch_result(plan, srcs, fresh, dev)
    for _ in range(2):                          # two calls in a row
        dsts = fresh()
        rs.gather_broadcast_execute_static(plan, srcs, dsts)
        torch.cuda.synchronize()
        _check(dsts, want, dst_gone, "excluded plan, static")
        for a, b in zip(ref, dsts):
            if a is not None:
                assert torch.equal(a, b)


def test_static_scratch_rejects_tensors_above_its_size():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    rows = rs.STATIC_SCRATCH_BYTES // (2 * 4096) + 1
    plan = rs.reshard_plan_create((rows, 4096), "bf16", (2,), ("S0",), (2,), ("S1",))
    with pytest.raises(rs.ReshardError) as ei:
        rs.gather_broadcast_execute_static(plan, [0x1000, 0x2000], [0x3000, 0x4000])
    assert ei.value.status == 2 and "static scratch" in str(ei.value)
    assert math.prod((rows, 4096)) * 2 > rs.STATIC_SCRATCH_BYTES
