"""The multi-GPU partition's CUDA steps on one GB300 (needs a GPU).

Every GPU of a partition is emulated on cuda:0: each has its own source,
destination, send and receive buffers, its steps run through the C ABI
(reshard_partition_execute, the library's kernels), and each message is a
device-to-device copy from the sender's send buffer into the receiver's receive
buffer, in the library's schedule order on one stream.  No kernel waits on
another; the steps of the emulated GPUs simply run one after the other.  Every
destination byte is compared with the oracle (small cases) or with the slices
of the global tensor that the oracle's boxes give (the full FFN up projection).
"""
import math
import random

import numpy as np
import pytest
import torch

import dtensor_reshard_gb300 as rs
from inputs import TensorSpec, global_tensor, workload
from tests import helpers

pytestmark = pytest.mark.gpu


def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda:0")


def _emulate(oracle, spec, src_gpu, dst_gpu, dom, nchunks, misalign=0):
    dev = _cuda()
    glob = global_tensor(spec)
    host = helpers.scatter_with_oracle(oracle, glob, spec.src_mesh, spec.src_placements)
    plan = helpers.spec_plan(spec)
    part = rs.reshard_partition_create(plan, src_gpu, dst_gpu, dom, nchunks)
    G = len(dom)
    dboxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)

    def dev_bytes(n):
        # a payload that starts `misalign` bytes into its allocation
        base = torch.full((n + misalign + 16,), 0xA5, dtype=torch.uint8, device=dev)
        return base[misalign:misalign + n]
    srcs = [[None] * plan.n_src for _ in range(G)]
    dsts = [[None] * plan.n_dst for _ in range(G)]
    for r, h in enumerate(host):
        b = helpers.to_bytes(h)
        t = dev_bytes(b.size)
        if b.size:
            t.copy_(torch.from_numpy(b))
        srcs[src_gpu[r]][r] = t
    for r, (_, shp) in enumerate(dboxes):
        dsts[dst_gpu[r]][r] = dev_bytes(math.prod(shp) * spec.elem_bytes)
    info = [rs.reshard_partition_gpu(part, g) for g in range(G)]
    recv = [torch.zeros(max(1, i["recv_bytes"]), dtype=torch.uint8, device=dev) for i in info]
    send = [torch.zeros(max(1, i["send_bytes"]), dtype=torch.uint8, device=dev) for i in info]
    xfers = [rs.reshard_partition_transfers(part, g) for g in range(G)]
    for item in rs.partition_schedule(nchunks):
        if item[0] == "step":
            for g in range(G):
                rs.reshard_partition_execute(part, g, item[1], item[2], srcs[g], dsts[g],
                                             recv[g], send[g])
            continue
        rounds = set(item[1])
        for g in range(G):
            for x in xfers[g]:
                if x["dir"] != 0 or (x["chunk"], x["stage"]) not in rounds:
                    continue
                h = x["peer"]
                y = next(y for y in xfers[h] if y["dir"] == 1 and y["peer"] == g and
                         (y["chunk"], y["stage"]) == (x["chunk"], x["stage"]))
                assert y["bytes"] == x["bytes"]
                recv[h][y["offset"]:y["offset"] + y["bytes"]].copy_(
                    send[g][x["offset"]:x["offset"] + x["bytes"]])
    torch.cuda.synchronize()
    got = [dsts[dst_gpu[r]][r] for r in range(plan.n_dst)]
    assert rs.reshard_device_status() == 0, "a bounded wait ran out in a copy kernel"
    return part, glob, got


def _maps(kind, M, N, G):
    if kind == "colocated":
        return [r % G for r in range(M)], [r % G for r in range(N)]
    h = G // 2
    return [r % h for r in range(M)], [h + r % (G - h) for r in range(N)]


SMALL = [
    TensorSpec("w8x8", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",), init=("bits",), seed=1),
    TensorSpec("ragged3d", (37, 61, 229), "fp32", (2, 3), ("S2", "S0"), (5, 2), ("S1", "S2"),
               init=("bits",), seed=2),
    TensorSpec("odd_cols", (700, 1001), "bf16", (2, 3), ("R", "S1"), (4, 2), ("R", "S0"),
               init=("bits",), seed=3),
]


@pytest.mark.parametrize("i", range(len(SMALL)))
@pytest.mark.parametrize("kind", ["colocated", "disaggregated"])
@pytest.mark.parametrize("nchunks,misalign", [(1, 0), (3, 0), (2, 5)])
def test_partition_steps_match_oracle(oracle, i, kind, nchunks, misalign):
    spec = SMALL[i]
    plan = helpers.spec_plan(spec)
    G = 4
    src_gpu, dst_gpu = _maps(kind, plan.n_src, plan.n_dst, G)
    dom = [0, 0, 1, 1]
    _, glob, got = _emulate(oracle, spec, src_gpu, dst_gpu, dom, nchunks, misalign)
    src_bytes = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, src_bytes)
    for r, (g, w) in enumerate(zip(got, want)):
        assert np.array_equal(g.cpu().numpy(), w), f"{spec.name}: destination rank {r}"


@pytest.mark.parametrize("cfg", [3, 5])
def test_partition_reduced_workloads_on_the_gpu(oracle, cfg):
    w = workload(cfg, reduced=True)
    rng = random.Random(cfg)
    for spec in w.tensors[:3]:
        plan = helpers.spec_plan(spec)
        src_gpu = [rng.randrange(8) for _ in range(plan.n_src)]
        dst_gpu = [rng.randrange(8) for _ in range(plan.n_dst)]
        _, glob, got = _emulate(oracle, spec, src_gpu, dst_gpu, [g // 4 for g in range(8)], 2)
        src_bytes = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
            oracle, glob, spec.src_mesh, spec.src_placements)]
        want = helpers.expected_dst(oracle, spec, src_bytes)
        for r, (g, wnt) in enumerate(zip(got, want)):
            assert np.array_equal(g.cpu().numpy(), wnt), f"{spec.name}: destination rank {r}"


def test_partition_full_ffn_up(oracle):
    """The dense FFN up projection [14336, 4096] bf16, (DP2, TP4) -> (DP4, TP2), over 8
    emulated GPUs, training and generation ranks colocated, 2 chunks.  The domains take
    alternate GPUs, so each holds only half of the source's tensor-parallel shards and
    the rest must cross (domains of consecutive GPUs would each hold a whole replica)."""
    spec = workload(2).tensors[0]
    plan = helpers.spec_plan(spec)
    src_gpu, dst_gpu = _maps("colocated", plan.n_src, plan.n_dst, 8)
    dom = [g % 2 for g in range(8)]
    part, glob, got = _emulate(oracle, spec, src_gpu, dst_gpu, dom, 2)
    st = rs.reshard_partition_stats(part)
    assert st["inter_domain_bytes"] > 0 and st["intra_domain_bytes"] > 0
    whole = rs.reshard_partition_create(plan, src_gpu, dst_gpu, [g // 4 for g in range(8)], 2)
    assert rs.reshard_partition_stats(whole)["inter_domain_bytes"] == 0
    for r, (off, shp) in enumerate(oracle.boxes(spec.global_shape, spec.dst_mesh,
                                                spec.dst_placements)):
        want = helpers.to_bytes(helpers.slice_box(glob, off, shp))
        assert torch.equal(got[r].cpu(), torch.from_numpy(want)), f"destination rank {r}"
