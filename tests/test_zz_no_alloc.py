"""The allocation-free gather-and-broadcast entry point (needs a GB300).

gather_broadcast_execute_static serves callers that cannot call cudaMalloc (an
engine whose pool already owns the device memory, a path that must not trigger
the synchronisation an allocation can cause, a plugin given only its buffers):
its scratch and tables live in the library's static device arrays.  Here it is
called through the C ABI twice in a row, on two different plans, and each
result must equal, byte for byte, what gather_broadcast_execute produces with a
caller-owned scratch.  This file is collected last so that a failure here
cannot hide failures elsewhere; it also passes when run alone.
"""
import math

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
]


def _buffers(spec, dev):
    plan = rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                  spec.src_placements, spec.dst_mesh, spec.dst_placements)
    glob = global_tensor(spec, device=dev)
    srcs = []
    for r in range(plan.n_src):
        shp, off = rs.reshard_plan_local_shape(plan, 0, r)
        sl = tuple(slice(o, o + s) for o, s in zip(off, shp))
        srcs.append(glob[sl].contiguous())

    def fresh_dsts():
        out = []
        for r in range(plan.n_dst):
            shp, _ = rs.reshard_plan_local_shape(plan, 1, r)
            d = torch.empty(shp, dtype=glob.dtype, device=dev)
            if d.numel():
                d.view(-1).view(torch.uint8).fill_(0xA5)
            out.append(d)
        return out
    return plan, srcs, fresh_dsts


def _bytes(ts):
    return [t.reshape(-1).view(torch.uint8) for t in ts]


def test_static_scratch_matches_caller_scratch_on_two_calls():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    dev = torch.device("cuda:0")
    cases = [_buffers(spec, dev) for spec in SPECS]
    expected = []
    for (plan, srcs, fresh) in cases:
        dsts = fresh()
        G = rs.reshard_plan_stats(plan)["global_bytes"]
        scratch = torch.empty(G, dtype=torch.uint8, device=dev)
        rs.gather_broadcast_execute(plan, srcs, dsts, scratch, G)
        expected.append(dsts)
    torch.cuda.synchronize()
    got = []
    for (plan, srcs, fresh) in cases:      # two calls in a row on one stream
        dsts = fresh()
        rs.gather_broadcast_execute_static(plan, srcs, dsts)
        got.append(dsts)
    torch.cuda.synchronize()
    for want, have in zip(expected, got):
        for a, b in zip(_bytes(want), _bytes(have)):
            assert torch.equal(a, b)
    # and the first plan once more, after the second overwrote the shared arrays
    plan, srcs, fresh = cases[0]
    dsts = fresh()
    rs.gather_broadcast_execute_static(plan, srcs, dsts)
    torch.cuda.synchronize()
    for a, b in zip(_bytes(expected[0]), _bytes(dsts)):
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
