"""The multi-GPU partition of a reshard, on the CPU (no GPU needed).

A partition cuts one plan by destination ownership over several GPUs in NVLink
domains.  Here every GPU's share runs on host buffers with the test CPU tile
executor, the messages are copied between the GPUs' send and receive buffers,
and every destination byte is compared with the oracle.  The routing rules are
checked against figures computed here from the layouts alone: bytes copied
locally, bytes that cross domains (each region at most once per receiving
domain) and bytes sent inside domains.
"""
import ctypes
import math
import random

import numpy as np
import pytest
import torch

import dtensor_reshard_gb300 as rs
from inputs import TensorSpec, global_tensor, workload
from tests import helpers
from tests import torch_chunk_layout as tcl


def _spec(gshape, dtype, sm, sp, dm, dp, seed=0):
    return TensorSpec(f"p{gshape}", tuple(gshape), dtype, tuple(sm), tuple(sp), tuple(dm),
                      tuple(dp), init=("bits",), seed=seed)


def _maps(kind, M, N, G, rng):
    if G == 1:
        return [0] * M, [0] * N
    if kind == "colocated":          # training and generation on the same GPUs
        return [r % G for r in range(M)], [r % G for r in range(N)]
    if kind == "disaggregated":      # sources on the first half of the GPUs
        h = G // 2
        return [r % h for r in range(M)], [h + r % (G - h) for r in range(N)]
    return [rng.randrange(G) for _ in range(M)], [rng.randrange(G) for _ in range(N)]


def emulate(oracle, spec, src_gpu, dst_gpu, gpu_domain, nchunks, plan=None):
    """Every GPU's share on the CPU, in lockstep; returns (partition, per-GPU buffers,
    write counts, expected destination bytes)."""
    glob = global_tensor(spec)
    src_bytes = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, src_bytes)
    plan = plan or helpers.spec_plan(spec)
    part = rs.reshard_partition_create(plan, src_gpu, dst_gpu, gpu_domain, nchunks)
    G = len(gpu_domain)
    state = [helpers.partition_gpu_buffers(part, g, src_bytes, [w.size for w in want], src_gpu,
                                           dst_gpu) for g in range(G)]
    xfers = [rs.reshard_partition_transfers(part, g) for g in range(G)]
    for item in rs.partition_schedule(nchunks):
        if item[0] == "step":
            for g in range(G):
                helpers.run_partition_step_cpu(part, g, item[1], item[2], *state[g])
            continue
        rounds = set(item[1])
        for g in range(G):
            for x in xfers[g]:
                if (x["chunk"], x["stage"]) not in rounds or x["dir"] != 0:
                    continue
                h = x["peer"]
                match = [y for y in xfers[h] if y["dir"] == 1 and y["peer"] == g and
                         (y["chunk"], y["stage"]) == (x["chunk"], x["stage"])]
                assert len(match) == 1 and match[0]["bytes"] == x["bytes"], (g, h, x)
                y = match[0]
                send, recv = state[g][0][-1], state[h][0][-2]
                assert x["offset"] + x["bytes"] <= send.size
                assert y["offset"] + y["bytes"] <= recv.size
                recv[y["offset"]:y["offset"] + y["bytes"]] = \
                    send[x["offset"]:x["offset"] + x["bytes"]]
    return part, state, want


def check_against_oracle(spec, part, state, want, dst_gpu):
    M, N = part.plan.n_src, part.plan.n_dst
    for r in range(N):
        bufs, writes = state[dst_gpu[r]]
        got = bufs[M + r]
        assert np.array_equal(got, want[r]), f"{spec.name}: destination rank {r} differs"
        assert (writes[M + r] == 1).all(), f"{spec.name}: destination rank {r} not written once"


def expected_routing(oracle, spec, src_gpu, dst_gpu, gpu_domain):
    """(local, inter, intra) bytes from the layouts and maps alone: a destination replica
    whose GPU holds a source replica of a region copies it locally; every other GPU that
    needs a region receives it once; a domain with no source replica of it receives it
    across domains exactly once, the rest of its GPUs inside the domain."""
    eb = spec.elem_bytes
    sb = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    db = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
    sclass, dclass = {}, {}
    for r, b in enumerate(sb):
        if math.prod(b[1]):
            sclass.setdefault(b, []).append(r)
    for r, b in enumerate(db):
        if math.prod(b[1]):
            dclass.setdefault(b, []).append(r)
    local = inter = intra = 0
    for (doff, dshp), dranks in dclass.items():
        for (soff, sshp), sranks in sclass.items():
            vol = 1
            for a, b, c, d in zip(doff, dshp, soff, sshp):
                vol *= max(0, min(a + b, c + d) - max(a, c))
            if vol == 0:
                continue
            have = {src_gpu[s] for s in sranks}
            need = {dst_gpu[r] for r in dranks}
            local += vol * eb * sum(1 for r in dranks if dst_gpu[r] in have)
            remote = need - have
            for dom in {gpu_domain[g] for g in remote}:
                n = sum(1 for g in remote if gpu_domain[g] == dom)
                if any(gpu_domain[g] == dom for g in have):
                    intra += vol * eb * n
                else:
                    inter += vol * eb
                    intra += vol * eb * (n - 1)
    return local, inter, intra


CASES = [
    _spec((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",), seed=1),            # the worked example
    _spec((37, 61, 29), "fp32", (2, 3), ("S2", "S0"), (5, 2), ("S1", "S2"), seed=2),
    _spec((96, 40), "bf16", (2, 4), ("R", "S0"), (4, 2), ("R", "S1"), seed=3),  # FFN-up shape
    _spec((64, 24), "fp16", (8,), ("S0",), (2, 4), ("S0", "R"), seed=4),         # HybridFlow
    _spec((16, 20, 14), "bf16", (1, 4, 2), ("R", "S0", "S1"), (2, 4), ("R", "S1"), seed=5),
    _spec((0, 7), "bf16", (2,), ("S0",), (3,), ("S1",), seed=6),                 # empty tensor
    _spec((3,), "fp32", (8,), ("S0",), (5,), ("S0",), seed=7),                   # empty shards
]


@pytest.mark.parametrize("i", range(len(CASES)))
@pytest.mark.parametrize("kind", ["colocated", "disaggregated", "random"])
@pytest.mark.parametrize("G,per_domain,nchunks", [(4, 2, 1), (4, 2, 3), (6, 3, 2), (3, 3, 1),
                                                  (1, 1, 1)])
def test_partition_matches_oracle(oracle, i, kind, G, per_domain, nchunks):
    spec = CASES[i]
    rng = random.Random(i * 100 + G)
    plan = helpers.spec_plan(spec)
    src_gpu, dst_gpu = _maps(kind, plan.n_src, plan.n_dst, G, rng)
    dom = [g // per_domain for g in range(G)]
    part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, nchunks, plan)
    check_against_oracle(spec, part, state, want, dst_gpu)
    st = rs.reshard_partition_stats(part)
    local, inter, intra = expected_routing(oracle, spec, src_gpu, dst_gpu, dom)
    assert (st["local_bytes"], st["inter_domain_bytes"], st["intra_domain_bytes"]) == \
        (local, inter, intra)
    assert st["ngpus"] == G and st["ndomains"] == len(set(dom))


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_partition_reduced_workloads(oracle, cfg):
    """The reduced configurations over 8 GPUs in 2 domains: training ranks on one domain's
    GPUs, generation ranks on the other's (disaggregated), and both colocated."""
    w = workload(cfg, reduced=True)
    rng = random.Random(cfg)
    for spec in w.tensors[:3]:
        plan = helpers.spec_plan(spec)
        for kind in ("colocated", "disaggregated"):
            src_gpu, dst_gpu = _maps(kind, plan.n_src, plan.n_dst, 8, rng)
            dom = [g // 4 for g in range(8)]
            part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, 2, plan)
            check_against_oracle(spec, part, state, want, dst_gpu)
            st = rs.reshard_partition_stats(part)
            assert (st["local_bytes"], st["inter_domain_bytes"], st["intra_domain_bytes"]) == \
                expected_routing(oracle, spec, src_gpu, dst_gpu, dom)


def test_partition_uneven_stress_reduced(oracle):
    w = workload(4, reduced=True)
    rng = random.Random(44)
    for spec in w.tensors[:12]:
        plan = helpers.spec_plan(spec)
        G = rng.choice((2, 4, 8))
        src_gpu, dst_gpu = _maps("random", plan.n_src, plan.n_dst, G, rng)
        dom = [g // 2 for g in range(G)]
        part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, rng.choice((1, 2)),
                                    plan)
        check_against_oracle(spec, part, state, want, dst_gpu)


def test_partition_random_small_layouts(oracle):
    rng = random.Random(9)
    layouts = {nd: [(m, p) for m in tcl.all_meshes(4) for p in tcl.all_placements(len(m), nd)]
               for nd in (1, 2, 3)}
    for k in range(150):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 7) for _ in range(nd))
        (sm, sp), (dm, dp) = rng.choice(layouts[nd]), rng.choice(layouts[nd])
        spec = _spec(gshape, rng.choice(("u8", "bf16", "fp32", "fp64")), sm, sp, dm, dp, seed=k)
        plan = helpers.spec_plan(spec)
        G = rng.randint(1, 5)
        src_gpu, dst_gpu = _maps("random", plan.n_src, plan.n_dst, G, rng)
        dom = [rng.randrange(2) for _ in range(G)]
        part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, rng.randint(1, 3), plan)
        check_against_oracle(spec, part, state, want, dst_gpu)
        assert (lambda s: (s["local_bytes"], s["inter_domain_bytes"], s["intra_domain_bytes"]))(
            rs.reshard_partition_stats(part)) == expected_routing(oracle, spec, src_gpu, dst_gpu,
                                                                  dom)


def test_partition_balances_senders_and_receivers(oracle):
    """Two source replicas in domain 0, four destination replicas in domain 1 (one GPU
    each): every region crosses once, the two source GPUs send about half each, the
    receiving GPUs take turns, and each receiver forwards to the other three."""
    spec = _spec((64, 256), "bf16", (2, 4), ("R", "S1"), (4,), ("R",), seed=11)
    plan = helpers.spec_plan(spec)
    # source rank (d, t) on GPU d (domain 0), destination replica r on GPU 2 + r (domain 1)
    src_gpu = [r // 4 for r in range(8)]
    dst_gpu = [2 + r for r in range(4)]
    dom = [0, 0, 1, 1, 1, 1]
    part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, 1, plan)
    check_against_oracle(spec, part, state, want, dst_gpu)
    st = rs.reshard_partition_stats(part)
    G = spec.global_bytes
    assert st["inter_domain_bytes"] == G            # the tensor crosses once
    assert st["intra_domain_bytes"] == 3 * G        # each piece forwarded to three GPUs
    sent = [rs.reshard_partition_gpu(part, g)["sent_inter_bytes"] for g in (0, 1)]
    assert sent[0] == sent[1] == G // 2
    got = [rs.reshard_partition_gpu(part, g)["recv_inter_bytes"] for g in range(2, 6)]
    assert got == [G // 4] * 4


def test_partition_pipeline_chunks_and_slots(oracle):
    """Chunks split the crossing bytes evenly and alternate between two buffer slots."""
    spec = _spec((120, 64), "fp32", (4,), ("S0",), (4,), ("S1",), seed=12)
    plan = helpers.spec_plan(spec)
    src_gpu, dst_gpu, dom = [0, 1, 2, 3], [3, 2, 1, 0], [0, 0, 1, 1]
    one = rs.reshard_partition_create(plan, src_gpu, dst_gpu, dom, 1)
    four = rs.reshard_partition_create(plan, src_gpu, dst_gpu, dom, 4)
    assert rs.reshard_partition_stats(four)["nslots"] == 2
    for g in range(4):
        a, b = rs.reshard_partition_gpu(one, g), rs.reshard_partition_gpu(four, g)
        # two slots of about a quarter each (three regions of 30 rows cut 7 + 8 + 7 + 8)
        assert b["recv_bytes"] <= 2 * (a["recv_bytes"] // 4 + 64 + 64)
        per_chunk = {}
        for x in rs.reshard_partition_transfers(four, g):
            if x["dir"] == 1:
                per_chunk[x["chunk"]] = per_chunk.get(x["chunk"], 0) + x["bytes"]
        assert len(per_chunk) == 4 and max(per_chunk.values()) - min(per_chunk.values()) <= 128
    part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, 4, plan)
    check_against_oracle(spec, part, state, want, dst_gpu)


def test_partition_excluded_ranks(oracle):
    """A plan that leaves out a source replica and a destination rank: the gone ranks get
    no buffers, the others are filled from the surviving replicas."""
    spec = _spec((48, 30), "bf16", (2, 2), ("R", "S0"), (3, 2), ("R", "S1"), seed=13)
    base = helpers.spec_plan(spec)
    plan = rs.reshard_plan_exclude(base, src_gone=[1], dst_gone=[4])
    src_gpu, dst_gpu, dom = [0, 1, 2, 3], [0, 1, 2, 3, -1, 1], [0, 0, 1, 1]
    part, state, want = emulate(oracle, spec, src_gpu, dst_gpu, dom, 1, plan)
    for r in range(plan.n_dst):
        if r == 4:
            continue
        bufs, writes = state[dst_gpu[r]]
        assert np.array_equal(bufs[plan.n_src + r], want[r]), r
    for g in range(4):
        for t in rs.reshard_partition_program(part, g, rs.STEP_PACK, 0)[0]:
            assert t["src_buf"] != 1


def test_partition_argument_checks():
    plan = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_partition_create(plan, [0, 2], [0, 1, 0, 1], [0, 0])   # gpu out of range
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_partition_create(plan, [0, 1], [0, 1, 0, 1], [0, -1])  # negative domain
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_partition_create(plan, [0, 1], [0, 1, 0, 1], [0, 0], nchunks=0)
    assert e.value.status == 1
    inplace = rs.reshard_plan_create_inplace((64, 16), "fp32", (8,), ("S0",), (2, 4),
                                             ("S0", "R"), src_alias=list(range(8)))
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_partition_create(inplace, list(range(8)), list(range(8)), [0] * 8)
    assert e.value.status == 2
    part = rs.reshard_partition_create(plan, [0, 1], [0, 1, 0, 1], [0, 0])
    with pytest.raises(rs.ReshardError):
        rs.reshard_partition_program(part, 2, rs.STEP_LOCAL)
    with pytest.raises(rs.ReshardError):
        rs.reshard_partition_program(part, 0, rs.STEP_PACK, 1)       # chunk out of range
    # NULL for a source rank this GPU reads: rejected before any device work
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_partition_execute(part, 0, rs.STEP_LOCAL, 0, [None, None],
                                     [0x1000, None, 0x2000, None], 0x3000, 0x4000)
    assert e.value.status == 1
    stale = part.handle
    rs.reshard_partition_destroy(part)
    out = rs.reshard_partition_stats_t()
    assert rs._lib.reshard_partition_stats(stale, ctypes.byref(out)) == 6   # use after destroy
    assert rs._lib.reshard_partition_destroy(stale) == 6
