"""GPU parity: the CUDA path against the CPU oracle, bit for bit (needs a GB300).

Every call goes through the C ABI (via the ctypes binding).  Destination
buffers sit between guard bands that must come back untouched.  Sizes the
oracle finishes in seconds are compared in full; the full-size workloads are
compared on oracle-sampled elements and, in full, against the slices of the
global tensor given by the oracle's boxes.
"""
import math
import random

import numpy as np
import pytest
import torch

import dtensor_reshard_gb300 as rs
from inputs import TensorSpec, global_tensor, uneven_stress, workload
from tests import helpers

pytestmark = pytest.mark.gpu

GUARD = 512
GUARD_BYTE = 0x5C
FILL_BYTE = 0xA5


def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda:0")


class Guarded:
    """A device byte buffer with guard bands; ``ptr`` is the payload's address."""

    def __init__(self, nbytes, misalign=0, fill=FILL_BYTE):
        self.n = int(nbytes)
        self.lead = GUARD + misalign
        self.buf = torch.full((self.lead + self.n + GUARD,), GUARD_BYTE, dtype=torch.uint8,
                              device="cuda")
        if self.n:
            self.buf[self.lead:self.lead + self.n].fill_(fill)
        self.ptr = self.buf.data_ptr() + self.lead if self.n else None

    def payload(self):
        return self.buf[self.lead:self.lead + self.n]

    def guards_intact(self):
        head = self.buf[:self.lead]
        tail = self.buf[self.lead + self.n:]
        return bool((head == GUARD_BYTE).all()) and bool((tail == GUARD_BYTE).all())


def _upload(arrs, misalign=0):
    out = []
    for a in arrs:
        g = Guarded(a.size, misalign)
        if a.size:
            g.payload().copy_(torch.from_numpy(a).cuda())
        out.append(g)
    return out


def run_and_compare(oracle, spec, kernel=rs.KERNEL_FANOUT, misalign=0, stream=None,
                    path="reshard", dst_misalign=None, expect_path=None):
    _cuda()
    glob = global_tensor(spec)
    srcs = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, srcs)
    dsrc = _upload(srcs, misalign)
    ddst = [Guarded(w.size, misalign if dst_misalign is None else dst_misalign(r))
            for r, w in enumerate(want)]
    plan = helpers.spec_plan(spec)
    sptr = [g.ptr for g in dsrc]
    dptr = [g.ptr for g in ddst]
    scratch = None
    if expect_path is not None:
        assert rs.reshard_plan_path(plan, sptr, dptr, kernel)[0] == expect_path
    if path == "reshard":
        rs.reshard_execute_ex(plan, sptr, dptr, kernel, stream)
    else:
        scratch = Guarded(spec.global_bytes, misalign)
        rs.gather_broadcast_execute(plan, sptr, dptr, scratch.ptr, spec.global_bytes, stream)
    torch.cuda.synchronize()
    for r, (g, w) in enumerate(zip(ddst, want)):
        got = g.payload().cpu().numpy()
        if not np.array_equal(got, w):
            bad = np.flatnonzero(got != w)
            raise AssertionError(f"{spec.name} dst rank {r}: {bad.size} bytes differ, "
                                 f"first at {bad[0]} (kernel {kernel}, path {path})")
        assert g.guards_intact(), f"guard band overwritten at dst rank {r}"
    for r, g in enumerate(dsrc):
        assert g.payload().cpu().numpy().tobytes() == srcs[r].tobytes(), "source modified"
        assert g.guards_intact()
    if scratch is not None:
        assert np.array_equal(scratch.payload().cpu().numpy(), helpers.to_bytes(glob))
        assert scratch.guards_intact()
    assert rs.reshard_device_status() == 0, "a bounded wait ran out in a copy kernel"


# ---------------------------------------------------------------------- reduced workloads
@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
@pytest.mark.parametrize("kernel", [rs.KERNEL_FANOUT, rs.KERNEL_BOXCOPY])
def test_reduced_workloads(oracle, cfg, kernel):
    for spec in workload(cfg, reduced=True).tensors:
        run_and_compare(oracle, spec, kernel=kernel)


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_reduced_workloads_gather_broadcast(oracle, cfg):
    for spec in workload(cfg, reduced=True).tensors:
        run_and_compare(oracle, spec, path="gather_broadcast")


def test_uneven_stress_reduced(oracle):
    for spec in workload(4, reduced=True).tensors:
        run_and_compare(oracle, spec)
        run_and_compare(oracle, spec, kernel=rs.KERNEL_BOXCOPY)


def test_worked_example_blocks(oracle):
    """Each destination of the 8x8 example holds rows 0-3 of source 0 and rows 4-7 of
    source 1 at columns 2j..2j+1 (two 4x2 blocks)."""
    spec = workload(1).tensors[0]
    run_and_compare(oracle, spec)
    glob = global_tensor(spec).cuda()
    srcs = [glob[:4].contiguous(), glob[4:].contiguous()]
    dsts = [torch.empty(8, 2, dtype=glob.dtype, device="cuda") for _ in range(4)]
    plan = helpers.spec_plan(spec)
    rs.reshard_execute(plan, srcs, dsts)
    torch.cuda.synchronize()
    for j in range(4):
        assert torch.equal(dsts[j][:4], srcs[0][:, 2 * j:2 * j + 2])
        assert torch.equal(dsts[j][4:], srcs[1][:, 2 * j:2 * j + 2])


# ---------------------------------------------------------------------- edge cases
def _spec(gshape, dtype, sm, sp, dm, dp, seed=0):
    return TensorSpec("edge", tuple(gshape), dtype, tuple(sm), tuple(sp), tuple(dm), tuple(dp),
                      init=("bits",), seed=seed)


EDGE = [
    _spec((0, 7), "bf16", (2,), ("S0",), (3,), ("S1",)),              # empty tensor
    _spec((3,), "fp32", (8,), ("S0",), (5,), ("S0",)),                # more ranks than elements
    _spec((1,), "u8", (1,), ("R",), (4,), ("R",)),                    # one byte, fan-out 4
    _spec((5, 3), "bf16", (4,), ("S0",), (2, 2), ("S1", "S0")),       # ragged + empty shards
    _spec((1000, 37), "bf16", (3,), ("S1",), (7,), ("S0",)),          # odd bf16 rows
    _spec((4097, 3), "u8", (5,), ("S0",), (2,), ("S1",)),             # 1-byte rows
    _spec((37, 11, 13), "fp16", (2, 3), ("S2", "S1"), (3, 2), ("S1", "S2")),  # 3-D planes
    _spec((3, 5, 7, 9), "fp64", (2,), ("S3",), (2, 2), ("S1", "S3")),  # 4-D
    _spec((64, 4096), "bf16", (2,), ("S0",), (64,), ("R",)),          # fan-out 64
    _spec((300, 1000), "bf16", (1,), ("R",), (300,), ("R",)),         # fan-out 300 > group max
    _spec((512,), "fp32", (510,), ("S0",), (513,), ("S0",)),          # M + N + 1 = 1024
    _spec((2, 70000), "bf16", (2,), ("S1",), (2,), ("S0",)),          # 70 KB runs inside rows
    _spec((16, 3, 100000), "fp32", (2, 2), ("S0", "S2"), (4,), ("S2",)),  # long rows, planes
]


@pytest.mark.parametrize("i", range(len(EDGE)))
def test_edge_cases(oracle, i):
    spec = EDGE[i]
    run_and_compare(oracle, spec)
    run_and_compare(oracle, spec, kernel=rs.KERNEL_BOXCOPY)
    if spec.global_bytes:
        run_and_compare(oracle, spec, path="gather_broadcast")


@pytest.mark.parametrize("misalign", [1, 2, 4, 8])
def test_misaligned_buffers(oracle, misalign):
    """Base pointers off the 16-byte grid take the narrower vector paths."""
    for spec in (workload(2, reduced=True).tensors[0], EDGE[4], EDGE[6]):
        run_and_compare(oracle, spec, misalign=misalign)


@pytest.mark.parametrize("kernel", [rs.KERNEL_FANOUT, rs.KERNEL_BOXCOPY])
def test_destinations_with_different_alignments(oracle, kernel):
    """Replicas whose buffers differ in address mod 16 (one fan-out group)."""
    for spec in (_spec((300, 97), "bf16", (2,), ("S0",), (2, 3), ("R", "S1")),
                 _spec((7, 4099), "u8", (3,), ("S1",), (5,), ("R",)),
                 _spec((64, 1024), "fp32", (4,), ("S0",), (8,), ("R",))):
        run_and_compare(oracle, spec, kernel=kernel, misalign=3, dst_misalign=lambda r: r % 16)


def test_nan_payloads_and_negative_zero_survive(oracle):
    spec = _spec((257, 129), "fp32", (2, 2), ("S0", "R"), (3,), ("S1",), seed=77)
    run_and_compare(oracle, spec)


def test_runs_on_a_side_stream(oracle):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_and_compare(oracle, workload(2, reduced=True).tensors[0], stream=s)


def test_repeated_execution_is_stable(oracle):
    spec = workload(3, reduced=True).tensors[0]
    for _ in range(3):
        run_and_compare(oracle, spec)


def test_execute_after_destroy_is_rejected():
    _cuda()
    plan = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    h = plan.handle
    rs.reshard_plan_destroy(plan)
    import ctypes
    assert rs._lib.reshard_execute(ctypes.c_void_p(h), None, None, None) == 6


def test_replan_after_rank_removal(oracle):
    """Membership change = destroy + re-create with the shrunken mesh (planned on the host)."""
    spec = workload(2, reduced=True).tensors[0]
    run_and_compare(oracle, spec)
    shrunk = TensorSpec(spec.name, spec.global_shape, spec.dtype, spec.src_mesh,
                        spec.src_placements, (3, 2), spec.dst_placements, init=spec.init,
                        seed=spec.seed)
    run_and_compare(oracle, shrunk)


# ---------------------------------------------------------------------- full sizes
def _full_size_check(oracle, spec, samples=4000, kernel=rs.KERNEL_FANOUT, seed=0):
    """Full-size run: every destination shard equals the global tensor cut by the oracle's
    box, and oracle_source_of agrees on sampled elements."""
    dev = _cuda()
    glob = global_tensor(spec, device=dev)
    src_boxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    dst_boxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
    srcs = [helpers.slice_box(glob, o, s) for o, s in src_boxes]
    dsts = [torch.empty(s, dtype=glob.dtype, device=dev) for _, s in dst_boxes]
    for d in dsts:
        if d.numel():
            d.view(-1).view(torch.uint8).fill_(FILL_BYTE)
    plan = helpers.spec_plan(spec)
    rs.reshard_execute_ex(plan, srcs, dsts, kernel)
    torch.cuda.synchronize()
    for r, (o, s) in enumerate(dst_boxes):
        if math.prod(s):
            want = helpers.slice_box(glob, o, s)
            assert torch.equal(dsts[r].reshape(-1).view(torch.uint8),
                               want.reshape(-1).view(torch.uint8)), (spec.name, r)
    del glob
    rng = random.Random(seed)
    nonempty = [r for r, (_, s) in enumerate(dst_boxes) if math.prod(s)]
    ivt = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[spec.elem_bytes]
    by_rank = {}
    for _ in range(samples if nonempty else 0):
        r = rng.choice(nonempty)
        e = rng.randrange(math.prod(dst_boxes[r][1]))
        s, j = oracle.source_of(spec.global_shape, spec.src_mesh, spec.src_placements,
                                spec.dst_mesh, spec.dst_placements, r, e)
        by_rank.setdefault((r, s), []).append((e, j))
    for (r, s), pairs in by_rank.items():
        e = torch.tensor([p[0] for p in pairs], device=dev)
        j = torch.tensor([p[1] for p in pairs], device=dev)
        got = dsts[r].reshape(-1).view(ivt)[e]
        want = srcs[s].reshape(-1).view(ivt)[j]
        assert torch.equal(got, want), (spec.name, r, s)


def test_full_ffn_up_against_full_oracle(oracle):
    """Dense FFN up-projection at its full size, compared byte for byte with the oracle."""
    spec = workload(2).tensors[0]
    run_and_compare(oracle, spec)


@pytest.mark.parametrize("idx", [0, 2])
def test_full_hybridflow_layer(oracle, idx):
    _full_size_check(oracle, workload(3).tensors[idx])


@pytest.mark.parametrize("idx", [0, 2, 3, 4])
def test_full_moe_refit(oracle, idx):
    spec = workload(5).tensors[idx]
    if spec.path == "gather_broadcast":
        dev = _cuda()
        glob = global_tensor(spec, device=dev)
        src_boxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
        dst_boxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
        srcs = [helpers.slice_box(glob, o, s) for o, s in src_boxes]
        dsts = [torch.empty(s, dtype=glob.dtype, device=dev) for _, s in dst_boxes]
        scratch = torch.empty(spec.global_bytes, dtype=torch.uint8, device=dev)
        plan = helpers.spec_plan(spec)
        rs.gather_broadcast_execute(plan, srcs, dsts, scratch, spec.global_bytes)
        torch.cuda.synchronize()
        assert torch.equal(scratch, glob.reshape(-1).view(torch.uint8))
        for r, (o, s) in enumerate(dst_boxes):
            assert torch.equal(dsts[r].reshape(-1).view(torch.uint8),
                               helpers.slice_box(glob, o, s).reshape(-1).view(torch.uint8))
    else:
        _full_size_check(oracle, spec)


def test_full_moe_refit_as_one_batch_launch(oracle):
    """The bench's launch form at full size: the three expert tensors of the MoE refit as one
    batch launch (one launch class); every destination shard equals the global tensor cut by
    the oracle's box, and the oracle's owning-source rule agrees on sampled elements."""
    dev = _cuda()
    specs = [t for t in workload(5).tensors if t.path == "reshard"]
    assert len(specs) == 3
    cases = []
    for spec in specs:
        glob = global_tensor(spec, device=dev)
        src_boxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
        dst_boxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
        srcs = [helpers.slice_box(glob, o, sh).contiguous() for o, sh in src_boxes]
        del glob
        dsts = [torch.empty(sh, dtype=srcs[0].dtype, device=dev) for _, sh in dst_boxes]
        for d in dsts:
            d.view(-1).view(torch.uint8).fill_(FILL_BYTE)
        cases.append((spec, helpers.spec_plan(spec), src_boxes, dst_boxes, srcs, dsts))
    batch = rs.reshard_batch_create([c[1] for c in cases])
    assert rs.reshard_batch_classes(batch) == (1, [0, 0, 0])
    rs.reshard_batch_execute(batch, [c[4] for c in cases], [c[5] for c in cases])
    torch.cuda.synchronize()
    assert rs.reshard_device_status() == 0
    rng = random.Random(5)
    for spec, plan, src_boxes, dst_boxes, srcs, dsts in cases:
        # full comparison: re-assemble the global tensor from the sources, cut each box
        glob = torch.empty(spec.global_shape, dtype=srcs[0].dtype, device=dev)
        for (o, sh), x in zip(src_boxes, srcs):
            glob[tuple(slice(a, a + n) for a, n in zip(o, sh))] = x
        for r, (o, sh) in enumerate(dst_boxes):
            assert torch.equal(dsts[r].reshape(-1).view(torch.uint8),
                               helpers.slice_box(glob, o, sh).reshape(-1).view(torch.uint8)), (
                spec.name, r)
        del glob
        ivt = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[spec.elem_bytes]
        for _ in range(500):
            r = rng.randrange(len(dst_boxes))
            e = rng.randrange(math.prod(dst_boxes[r][1]))
            src, j = oracle.source_of(spec.global_shape, spec.src_mesh, spec.src_placements,
                                      spec.dst_mesh, spec.dst_placements, r, e)
            assert int(dsts[r].reshape(-1).view(ivt)[e]) == int(srcs[src].reshape(-1).view(ivt)[j])


@pytest.mark.parametrize("n", [3_000_000_000, 3_000_000_001])
@pytest.mark.parametrize("kernel", [rs.KERNEL_FANOUT, rs.KERNEL_BOXCOPY])
def test_offsets_beyond_4gib(oracle, n, kernel):
    """A 6 GB bf16 vector held whole by one rank, split four ways: the last shards start
    more than 4 GiB into the source buffer.  The even length keeps every piece 16-byte
    aligned (TMA path); the odd one leaves 2-byte alignment (realigning path)."""
    spec = TensorSpec("big", (n,), "bf16", (1,), ("R",), (4,), ("S0",), init=("bits",),
                      seed=n % 1000)
    plan = helpers.spec_plan(spec)
    assert rs.reshard_plan_local_shape(plan, 1, 3)[1][0] * 2 > (1 << 32)
    _full_size_check(oracle, spec, samples=2000, kernel=kernel)


def test_full_uneven_stress_sampled(oracle):
    for spec in workload(4).tensors:
        _full_size_check(oracle, spec, samples=300)


# ---------------------------------------------------------------------- in place
def run_inplace(oracle, spec, alias, kernel=rs.KERNEL_FANOUT):
    _cuda()
    glob = global_tensor(spec)
    sboxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    srcs = [helpers.to_bytes(helpers.slice_box(glob, o, s)) for o, s in sboxes]
    want = helpers.expected_dst(oracle, spec, srcs)
    plan = rs.reshard_plan_create_inplace(spec.global_shape, spec.dtype, spec.src_mesh,
                                          spec.src_placements, spec.dst_mesh, spec.dst_placements,
                                          alias)
    ddst = [Guarded(w.size) for w in want]
    sptr, own = [], []
    for s in range(spec.n_src):
        d, off = rs.reshard_plan_alias(plan, s)
        n = srcs[s].size
        if d >= 0 and n:
            ddst[d].payload()[off:off + n].copy_(torch.from_numpy(srcs[s]).cuda())
            sptr.append(ddst[d].ptr + off)
        else:
            g = Guarded(n)
            if n:
                g.payload().copy_(torch.from_numpy(srcs[s]).cuda())
            own.append(g)
            sptr.append(g.ptr)
    rs.reshard_execute_ex(plan, sptr, [g.ptr for g in ddst], kernel)
    torch.cuda.synchronize()
    for r, (g, w) in enumerate(zip(ddst, want)):
        assert np.array_equal(g.payload().cpu().numpy(), w), (spec.name, r, kernel)
        assert g.guards_intact()
    for g in own:
        assert g.guards_intact()
    assert rs.reshard_device_status() == 0
    return rs.reshard_plan_stats(plan)


@pytest.mark.parametrize("kernel", [rs.KERNEL_FANOUT, rs.KERNEL_BOXCOPY])
def test_inplace_hybridflow_divisible(oracle, kernel):
    spec = TensorSpec("hf", (2048, 819), "bf16", (8,), ("S0",), (2, 4), ("S0", "R"),
                      init=("bits",), seed=31)
    st = run_inplace(oracle, spec, list(range(8)), kernel)
    assert st["inplace_bytes"] == spec.global_bytes


@pytest.mark.parametrize("kernel", [rs.KERNEL_FANOUT, rs.KERNEL_BOXCOPY])
def test_inplace_reduced_and_random(oracle, kernel):
    for spec in workload(3, reduced=True).tensors:
        run_inplace(oracle, spec, helpers.pick_aliases(oracle, spec), kernel)
    rng = random.Random(41)
    n = 0
    while n < 40:
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 40) for _ in range(nd))
        sm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        dm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        sp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in sm)
        dp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in dm)
        spec = _spec(gshape, rng.choice(("bf16", "fp32", "u8")), sm, sp, dm, dp, seed=n)
        alias = helpers.pick_aliases(oracle, spec, rng)
        if all(a < 0 for a in alias):
            continue
        run_inplace(oracle, spec, alias, kernel)
        n += 1


def test_full_hybridflow_layer_inplace(oracle):
    """Full-size gate projection, in place: every generation buffer starts out holding its
    own training shard and must end up equal to its slice of the global tensor."""
    dev = _cuda()
    spec = workload(3).tensors[0]
    glob = global_tensor(spec, device=dev)
    dboxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
    sboxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    plan = rs.reshard_plan_create_inplace(spec.global_shape, spec.dtype, spec.src_mesh,
                                          spec.src_placements, spec.dst_mesh, spec.dst_placements,
                                          list(range(8)))
    dsts = [torch.empty(s, dtype=glob.dtype, device=dev) for _, s in dboxes]
    for d in dsts:
        d.view(-1).view(torch.uint8).fill_(FILL_BYTE)
    sptr = []
    for s, (o, shp) in enumerate(sboxes):
        d, off = rs.reshard_plan_alias(plan, s)
        piece = helpers.slice_box(glob, o, shp).reshape(-1).view(torch.uint8)
        flat = dsts[d].reshape(-1).view(torch.uint8)
        flat[off:off + piece.numel()].copy_(piece)
        sptr.append(dsts[d].data_ptr() + off)
    rs.reshard_execute(plan, sptr, dsts)
    torch.cuda.synchronize()
    for r, (o, s) in enumerate(dboxes):
        assert torch.equal(dsts[r].reshape(-1).view(torch.uint8),
                           helpers.slice_box(glob, o, s).reshape(-1).view(torch.uint8)), r
    assert rs.reshard_device_status() == 0


# ---------------------------------------------------------------------- batches
def _batch_case(oracle, specs, misalign=0):
    plans, sptrs, dptrs, want, keep = [], [], [], [], []
    for spec in specs:
        glob = global_tensor(spec)
        srcs = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
            oracle, glob, spec.src_mesh, spec.src_placements)]
        w = helpers.expected_dst(oracle, spec, srcs)
        ds = _upload(srcs, misalign)
        dd = [Guarded(x.size, misalign) for x in w]
        plans.append(helpers.spec_plan(spec))
        sptrs.append([g.ptr for g in ds])
        dptrs.append([g.ptr for g in dd])
        want.append(w)
        keep.append((ds, dd))
    return plans, sptrs, dptrs, want, keep


@pytest.mark.parametrize("misalign", [0, 2])
def test_batch_of_plans(oracle, misalign):
    """One launch for several tensors (aligned), or one plan at a time (misaligned)."""
    specs = list(workload(3, reduced=True).tensors) + list(
        t for t in workload(5, reduced=True).tensors if t.path == "reshard")
    plans, sptrs, dptrs, want, keep = _batch_case(oracle, specs, misalign)
    batch = rs.reshard_batch_create(plans)
    for _ in range(2):
        rs.reshard_batch_execute(batch, sptrs, dptrs)
    torch.cuda.synchronize()
    for (ds, dd), w in zip(keep, want):
        for g, x in zip(dd, w):
            assert np.array_equal(g.payload().cpu().numpy(), x)
            assert g.guards_intact()
    assert rs.reshard_device_status() == 0


@pytest.mark.parametrize("misalign", [0, 2, 3])
def test_batch_of_mixed_classes(oracle, misalign):
    """Uneven tensors of every copy path batched together: one launch per class of plans
    that take the same kernel, classes whose buffers are less aligned than assumed run plan
    by plan; every destination byte and guard band matches the oracle."""
    specs = list(uneven_stress(n=24, seed=4242, max_dim=2000, max_numel=1 << 19,
                               max_bytes=64 << 20, name="mix").tensors)
    plans, sptrs, dptrs, want, keep = _batch_case(oracle, specs, misalign)
    batch = rs.reshard_batch_create(plans)
    n, per = rs.reshard_batch_classes(batch)
    assert n >= 3 and n == len({c for c in per if c >= 0})
    for _ in range(2):
        rs.reshard_batch_execute(batch, sptrs, dptrs)
    torch.cuda.synchronize()
    for (ds, dd), w in zip(keep, want):
        for g, x in zip(dd, w):
            assert np.array_equal(g.payload().cpu().numpy(), x)
            assert g.guards_intact()
    assert rs.reshard_device_status() == 0


def test_batch_with_inplace_plan(oracle):
    spec = TensorSpec("hf", (2048, 264), "bf16", (8,), ("S0",), (2, 4), ("S0", "R"),
                      init=("bits",), seed=77)
    glob = global_tensor(spec)
    sboxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    srcs = [helpers.to_bytes(helpers.slice_box(glob, o, s)) for o, s in sboxes]
    want = helpers.expected_dst(oracle, spec, srcs)
    p_in = rs.reshard_plan_create_inplace(spec.global_shape, spec.dtype, spec.src_mesh,
                                          spec.src_placements, spec.dst_mesh,
                                          spec.dst_placements, list(range(8)))
    dd = [Guarded(x.size) for x in want]
    sp = []
    for s in range(8):
        d, off = rs.reshard_plan_alias(p_in, s)
        dd[d].payload()[off:off + srcs[s].size].copy_(torch.from_numpy(srcs[s]).cuda())
        sp.append(dd[d].ptr + off)
    other = workload(2, reduced=True).tensors[0]
    plans2, sptrs2, dptrs2, want2, keep2 = _batch_case(oracle, [other])
    batch = rs.reshard_batch_create([p_in] + plans2)
    rs.reshard_batch_execute(batch, [sp] + sptrs2, [[g.ptr for g in dd]] + dptrs2)
    torch.cuda.synchronize()
    for g, x in zip(dd, want):
        assert np.array_equal(g.payload().cpu().numpy(), x)
    for g, x in zip(keep2[0][1], want2[0]):
        assert np.array_equal(g.payload().cpu().numpy(), x)


# ---------------------------------------------------------------------- CUDA graphs
def test_cuda_graph_capture_and_replay(oracle):
    """A refit step recorded once into a CUDA graph replays exactly, and picks up new source
    values written into the same buffers (plans uploaded and kernels warmed up first)."""
    dev = _cuda()
    specs = list(workload(3, reduced=True).tensors[:3]) + [
        t for t in workload(5, reduced=True).tensors if t.path == "reshard"]
    cases = []
    for spec in specs:
        plan = helpers.spec_plan(spec)
        rs.reshard_plan_upload(plan)
        boxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
        srcs = [torch.empty(s, dtype=torch.bfloat16, device=dev) for _, s in boxes]
        dboxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
        dsts = [torch.empty(s, dtype=torch.bfloat16, device=dev) for _, s in dboxes]
        cases.append((spec, plan, boxes, srcs, dsts))

    def load(seed_shift):
        wants = []
        for spec, plan, boxes, srcs, dsts in cases:
            sp = TensorSpec(spec.name, spec.global_shape, spec.dtype, spec.src_mesh,
                            spec.src_placements, spec.dst_mesh, spec.dst_placements,
                            init=("bits",), seed=spec.seed + seed_shift)
            glob = global_tensor(sp)
            host = [helpers.slice_box(glob, o, s) for o, s in boxes]
            for d, h in zip(srcs, host):
                d.copy_(h)
            wants.append(helpers.expected_dst(oracle, sp, [helpers.to_bytes(h) for h in host]))
            for d in dsts:
                d.view(-1).view(torch.uint8).fill_(FILL_BYTE)
        torch.cuda.synchronize()
        return wants

    def step(stream):
        for spec, plan, boxes, srcs, dsts in cases:
            rs.reshard_execute(plan, srcs, dsts, stream)

    wants = load(0)
    step(torch.cuda.current_stream())          # warm-up: first launches outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    for shift in (0, 1000):
        wants = load(shift)
        graph.replay()
        torch.cuda.synchronize()
        for (spec, plan, boxes, srcs, dsts), want in zip(cases, wants):
            for d, w in zip(dsts, want):
                assert np.array_equal(helpers.to_bytes(d), w), (spec.name, shift)
    assert rs.reshard_device_status() == 0


def test_streams_and_graph_replay_beside_eager_launches(oracle):
    """Work-queue kernels on four streams at once, then a captured reshard replayed on one
    stream while the stream it was captured on keeps launching (more launches than a round
    of the device's work-queue slots): every destination byte is exact."""
    dev = _cuda()
    specs = [
        _spec((256, 64, 96), "fp32", (2, 2), ("S0", "S2"), (4,), ("S1",), seed=10),  # TMA fan-out
        _spec((2000, 1001), "bf16", (3,), ("S0",), (2,), ("S1",), seed=11),          # staged
        _spec((1500, 777), "fp16", (2,), ("S1",), (3,), ("S0",), seed=12),           # staged
        _spec((1000, 257), "fp16", (5,), ("S0",), (4,), ("R",), seed=13)]            # TMA fan-out
    for spec in specs:
        p = helpers.spec_plan(spec)
        assert rs.reshard_plan_path(p, [1 << 20] * p.n_src, [1 << 24] * p.n_dst)[0] in (
            "tma_fanout", "staged", "staged_bulk"), spec
    cases = []
    for spec in specs:
        glob = global_tensor(TensorSpec(spec.name, spec.global_shape, spec.dtype, spec.src_mesh,
                                        spec.src_placements, spec.dst_mesh, spec.dst_placements,
                                        init=("bits",), seed=spec.seed))
        boxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
        host = [helpers.slice_box(glob, o, sh) for o, sh in boxes]
        want = helpers.expected_dst(oracle, spec, [helpers.to_bytes(h) for h in host])
        srcs = [h.to(dev) for h in host]
        dboxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
        dsts = [torch.empty(sh, dtype=host[0].dtype, device=dev) for _, sh in dboxes]
        plan = helpers.spec_plan(spec)
        rs.reshard_plan_upload(plan)
        cases.append((spec, plan, srcs, dsts, want))

    def clear():
        for _, _, _, dsts, _ in cases:
            for d in dsts:
                d.view(-1).view(torch.uint8).fill_(FILL_BYTE)
        torch.cuda.synchronize()

    def check(which):
        torch.cuda.synchronize()
        for i in which:
            spec, _, _, dsts, want = cases[i]
            for d, w in zip(dsts, want):
                assert np.array_equal(helpers.to_bytes(d), w), spec.name
        assert rs.reshard_device_status() == 0

    clear()
    streams = [torch.cuda.Stream() for _ in cases]
    for _ in range(20):
        for (spec, plan, srcs, dsts, _), st in zip(cases, streams):
            rs.reshard_execute(plan, srcs, dsts, st)
    check(range(len(cases)))

    clear()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rs.reshard_execute(cases[0][1], cases[0][2], cases[0][3], torch.cuda.current_stream())
    eager, replay = torch.cuda.Stream(), torch.cuda.Stream()
    _, plan1, srcs1, dsts1, _ = cases[3]
    for k in range(1100):
        rs.reshard_execute(plan1, srcs1, dsts1, eager)
        if k % 50 == 0:
            with torch.cuda.stream(replay):
                graph.replay()
    check([0, 3])


def _driver_streams():
    """cuStreamCreate / cuStreamDestroy from the driver library: torch.cuda.Stream() hands
    out streams from a small pool, and these tests need genuinely new streams."""
    import ctypes
    lib = ctypes.CDLL("libcuda.so.1")
    lib.cuStreamCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint]
    lib.cuStreamCreate.restype = ctypes.c_int
    lib.cuStreamDestroy_v2.argtypes = [ctypes.c_void_p]
    lib.cuStreamDestroy_v2.restype = ctypes.c_int

    def create():
        h = ctypes.c_void_p()
        assert lib.cuStreamCreate(ctypes.byref(h), 1) == 0   # CU_STREAM_NON_BLOCKING
        return h.value

    def destroy(h):
        assert lib.cuStreamDestroy_v2(h) == 0
    return create, destroy


def test_work_queue_slots_pass_between_streams(oracle):
    """More streams than the device has work-queue slots (1024): 1500 streams created,
    used once and destroyed one after another, then 1100 live streams whose launches all
    wait behind one long kernel, so that no slot is idle when the later streams ask for
    one.  Every launch writes its own destinations, and each is exact."""
    dev = _cuda()
    specs = [_spec((64, 32, 96), "fp32", (2, 2), ("S0", "S2"), (4,), ("S1",), seed=14),
             _spec((600, 1001), "bf16", (3,), ("S0",), (2,), ("S1",), seed=15)]
    cases = []
    for spec, path in zip(specs, ("tma_fanout", "staged")):
        glob = global_tensor(spec)
        boxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
        host = [helpers.slice_box(glob, o, sh) for o, sh in boxes]
        want = helpers.expected_dst(oracle, spec, [helpers.to_bytes(h) for h in host])
        srcs = [h.to(dev) for h in host]
        plan = helpers.spec_plan(spec)
        wants = [torch.from_numpy(w).to(dev) for w in want]

        def new_dsts(wants=wants):
            return [torch.full_like(w, FILL_BYTE) for w in wants]
        assert rs.reshard_plan_path(plan, srcs, new_dsts())[0] == path, spec.name
        cases.append((plan, srcs, wants, new_dsts))
    create, destroy = _driver_streams()

    # streams created and destroyed one after another; each checks its own launches
    bad = torch.zeros((), dtype=torch.int64, device=dev)
    dsts = [c[3]() for c in cases]
    for k in range(1500):
        h = create()
        st = torch.cuda.ExternalStream(h)
        st.wait_stream(torch.cuda.current_stream())   # one stream after the other
        with torch.cuda.stream(st):
            for (plan, srcs, wants, _), d in zip(cases, dsts):
                for t in d:
                    t.fill_(FILL_BYTE)
                rs.reshard_execute(plan, srcs, d, st)
                for t, w in zip(d, wants):
                    bad += (t != w).sum()
        torch.cuda.current_stream().wait_stream(st)
        destroy(h)
    torch.cuda.synchronize()
    assert int(bad) == 0
    assert rs.reshard_device_status() == 0

    # live streams beyond the slot count, all held back behind one long kernel
    plan, srcs, wants, new_dsts = cases[0]
    outs = [new_dsts() for _ in range(1100)]
    torch.cuda.synchronize()
    gate = torch.cuda.Stream()
    with torch.cuda.stream(gate):
        torch.cuda._sleep(1_000_000_000)          # about half a second of one SM
    opened = torch.cuda.Event()
    opened.record(gate)
    handles = []
    for d in outs:
        h = create()
        st = torch.cuda.ExternalStream(h)
        st.wait_event(opened)
        rs.reshard_execute(plan, srcs, d, st)
        handles.append(h)
    torch.cuda.synchronize()
    for k, d in enumerate(outs):
        for t, w in zip(d, wants):
            assert torch.equal(t, w), f"stream {k}"
    for h in handles:
        destroy(h)
    assert rs.reshard_device_status() == 0


# ---------------------------------------------------------------------- transpose blocks
TRANSPOSE_CASES = [
    _spec((74, 65, 1721), "fp16", (61,), ("S2",), (3,), ("R",), seed=1),        # gather, R=3
    _spec((1338, 65), "fp16", (18,), ("S0",), (38,), ("S1",), seed=2),          # scatter, 2-4 B
    _spec((900, 7, 23), "bf16", (2, 5), ("R", "S2"), (2,), ("R",), seed=3),     # gather, R=2
    _spec((300, 40), "u8", (1,), ("R",), (40,), ("S1",), seed=4),               # scatter, 1 B
    _spec((40, 45, 17), "fp32", (6,), ("S0",), (17,), ("S2",), seed=5),         # scatter 3-D
    _spec((4097, 20), "u8", (20,), ("S1",), (4,), ("R",), seed=6),              # gather, 1 B, R=4
    _spec((40, 451, 715), "bf16", (6,), ("S0",), (45,), ("S2",), seed=7),       # scatter, 32 B
    _spec((2000, 288), "bf16", (18,), ("S1",), (4,), ("S0",), seed=8),          # gather, 32 B, R=1
    _spec((50, 553, 122), "bf16", (32,), ("S2",), (16,), ("S1",), seed=9),      # gather, planes
    _spec((30, 40, 300), "bf16", (4,), ("S1",), (20,), ("S2",), seed=10),       # scatter, planes
    _spec((3, 400, 1416), "bf16", (42,), ("S2",), (5,), ("S1",), seed=11),      # gather, 68 B
    _spec((520, 583, 3), "fp16", (1,), ("S1",), (45,), ("S2",), seed=12),       # de-interleave
    _spec((700, 3), "fp16", (1,), ("R",), (2,), ("S1",), seed=13),              # 4 + 2 bytes
    # gathers whose whole image is under one or two 16-byte granules: no bulk copy
    # of an aligned middle, or one of a single granule, beside the threads' bytes
    _spec((2, 6), "u8", (6,), ("S1",), (2,), ("R",), seed=14),
    _spec((5, 6), "u8", (6,), ("S1",), (3,), ("R",), seed=15),
]


@pytest.mark.parametrize("i", range(len(TRANSPOSE_CASES)))
@pytest.mark.parametrize("misalign", [0, 3])
def test_transpose_blocks(oracle, i, misalign):
    spec = TRANSPOSE_CASES[i]
    blocks, _ = rs.reshard_plan_transposes(helpers.spec_plan(spec), rs.PROGRAM_FANOUT)
    assert blocks, "layout expected to use transpose blocks"
    run_and_compare(oracle, spec, misalign=misalign)
    run_and_compare(oracle, spec, misalign=misalign, dst_misalign=lambda r: (r * 5) % 16)


# ---------------------------------------------------------------------- assemble, then replicate
# Column bands of 632-byte rows (off the 16-byte grid) gathered into 9 and into 15 replicas:
# the first step assembles the shard in one replica, the second copies it as one run to the
# others (TMA fan-out when the buffers are aligned, the vector kernel otherwise).
ASSEMBLE_CASES = [
    _spec((600, 2200), "fp32", (14,), ("S1",), (9,), ("R",), seed=21),
    _spec((393, 8780), "fp32", (56,), ("S1",), (15,), ("R",), seed=22),
    _spec((2, 300, 4424), "bf16", (2, 14), ("R", "S2"), (3, 12), ("S0", "R"), seed=23),
    # 6 replicas (the smallest fan-out that is assembled) of 770-byte column bands
    _spec((300, 6538), "bf16", (17,), ("S1",), (6,), ("R",), seed=24),
]


@pytest.mark.parametrize("i", range(len(ASSEMBLE_CASES)))
@pytest.mark.parametrize("misalign", [0, 3])
def test_assemble_then_replicate(oracle, i, misalign):
    spec = ASSEMBLE_CASES[i]
    plan = helpers.spec_plan(spec)
    st = rs.reshard_plan_stats(plan)
    assert st["assembled_classes"] >= 1 and st["n_replicate_tiles"] >= 1
    run_and_compare(oracle, spec, misalign=misalign)
    run_and_compare(oracle, spec, misalign=misalign, dst_misalign=lambda r: (r * 4) % 16)


# ---------------------------------------------------------------------- staged realigning copy
# One case per way the TMA-staged realigning kernel stages and stores a chunk;
# each asserts the path the execution takes, then checks every byte.
STAGED_CASES = [
    # runs, one replica
    ("runs", _spec((2000, 1301), "bf16", (3,), ("S0",), (2,), ("S0",), seed=11), "staged"),
    # rows that follow one another in the source: one bulk copy per chunk
    ("contiguous_rows", _spec((3000, 1203), "bf16", (4,), ("S1",), (3,), ("S0",), seed=12),
     "staged"),
    # short rows apart in the source: 16-byte cp.async copies into row slots
    ("short_rows", _spec((2400, 1203), "bf16", (3,), ("S0",), (2,), ("S1",), seed=13), "staged"),
    # rows of 5 KB apart in the source: one bulk copy per row slot
    ("long_rows", _spec((800, 5001), "bf16", (3,), ("S0",), (2,), ("S1",), seed=14), "staged"),
    # rows of 30 KB: pieces of a row per chunk
    ("row_pieces", _spec((300, 30001), "bf16", (3,), ("S0",), (2,), ("S1",), seed=15), "staged"),
    # 3-D tiles with planes
    ("planes", _spec((6, 500, 701), "bf16", (2,), ("S2",), (3,), ("S1",), seed=16), "staged"),
]


@pytest.mark.parametrize("misalign", [0, 3])
@pytest.mark.parametrize("i", range(len(STAGED_CASES)))
def test_staged_realign_paths(oracle, i, misalign):
    name, spec, want = STAGED_CASES[i]
    run_and_compare(oracle, spec, misalign=misalign, expect_path=want)


# Two replicas of a 52.8 MB bf16 tensor in 16 MB runs: bulk stores from the
# output stage when the replicas share their address mod 16 (aligned or not),
# per-replica realignment in registers when they do not.
BULK_SPEC = _spec((4400, 6001), "bf16", (3,), ("S0",), (2,), ("R",), seed=17)


@pytest.mark.parametrize("dst_mis,want", [
    (lambda r: 0, "staged_bulk"),
    (lambda r: 6, "staged_bulk"),
    (lambda r: (r * 5) % 16, "staged"),
], ids=["aligned", "congruent_misaligned", "incongruent"])
def test_staged_realign_fanout(oracle, dst_mis, want):
    run_and_compare(oracle, BULK_SPEC, misalign=0, dst_misalign=dst_mis, expect_path=want)


# Short rows (32..511 bytes) off the 16-byte grid, one replica or replicas at one
# address mod 16: the element kernel at the rows' common width.
SHORT_ROW_CASES = [
    # a column re-split of 2-byte elements: pieces of up to 160 bytes from 1-2 sources
    ("resplit", _spec((731, 397), "fp16", (5,), ("S1",), (6,), ("S1",), seed=21)),
    # 3-D tiles with planes (an innermost split into a middle-dim split)
    ("planes", _spec((40, 60, 301), "fp16", (3,), ("S2",), (4,), ("S1",), seed=22)),
    # rows of 474-480 bytes and 2-byte pieces beside them
    ("long_short", _spec((300, 957), "bf16", (4,), ("S1",), (2,), ("S1",), seed=23)),
    # 4-byte elements in rows of up to 448 bytes
    ("fp32", _spec((500, 1003), "fp32", (7,), ("S1",), (9,), ("S1",), seed=24)),
    # three replicas of every destination piece
    ("fanout", _spec((900, 397), "fp16", (5,), ("S1",), (3, 2), ("R", "S1"), seed=25)),
    # 410-byte rows from 818-byte source rows: every pair of source and destination
    # offsets mod 16
    ("all_offsets", _spec((1433, 409), "bf16", (4,), ("S0",), (2,), ("S1",), seed=26)),
]


@pytest.mark.parametrize("misalign", [0, 3])
@pytest.mark.parametrize("i", range(len(SHORT_ROW_CASES)))
def test_short_unaligned_rows(oracle, i, misalign):
    name, spec = SHORT_ROW_CASES[i]
    run_and_compare(oracle, spec, misalign=misalign, expect_path="vector")


@pytest.mark.parametrize("i", [0, 1, 5])
def test_short_unaligned_rows_every_destination_offset(oracle, i):
    """Destination rank r starts r bytes past its alignment: every destination
    offset mod 16 against every source offset."""
    _, spec = SHORT_ROW_CASES[i]
    run_and_compare(oracle, spec, misalign=0, dst_misalign=lambda r: r % 16,
                    expect_path="vector")


def test_short_rows_with_incongruent_replicas(oracle):
    _, spec = SHORT_ROW_CASES[4]
    run_and_compare(oracle, spec, misalign=0, dst_misalign=lambda r: (r * 6) % 16,
                    expect_path="vector")


def test_small_misaligned_fanout_uses_register_realign(oracle):
    spec = _spec((2000, 1301), "bf16", (3,), ("S0",), (2,), ("R",), seed=18)
    run_and_compare(oracle, spec, misalign=3, expect_path="realign")


# ---------------------------------------------------------------------- membership change
@pytest.mark.parametrize("kernel", [rs.KERNEL_FANOUT, rs.KERNEL_BOXCOPY])
@pytest.mark.parametrize("misalign", [0, 2])
def test_excluded_ranks_get_null_buffers(oracle, kernel, misalign):
    """A source replica and a destination rank leave: the derived plan reads the other
    replica, leaves the gone destination alone (NULL pointers for both) and is exact."""
    _cuda()
    spec = workload(2, reduced=True).tensors[0]
    src_gone, dst_gone = [1], [3]
    glob = global_tensor(spec)
    srcs = [helpers.to_bytes(x) for x in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, srcs)
    ds = _upload(srcs, misalign)
    dd = [Guarded(w.size, misalign) for w in want]
    plan = rs.reshard_plan_exclude(helpers.spec_plan(spec), src_gone, dst_gone)
    sptr = [None if r in src_gone else g.ptr for r, g in enumerate(ds)]
    dptr = [None if r in dst_gone else g.ptr for r, g in enumerate(dd)]
    rs.reshard_execute_ex(plan, sptr, dptr, kernel)
    torch.cuda.synchronize()
    for r, (g, w) in enumerate(zip(dd, want)):
        got = g.payload().cpu().numpy()
        if r in dst_gone:
            assert (got == FILL_BYTE).all(), "a gone destination was written"
        else:
            assert np.array_equal(got, w), r
        assert g.guards_intact()
    assert rs.reshard_device_status() == 0


# ---------------------------------------------------------------------- whole-model refit
@pytest.mark.parametrize("mode", ["one_stream", "batch", "lanes", "both"])
@pytest.mark.parametrize("misalign", [0, 2])
def test_refit_hybrid_routes(oracle, mode, misalign):
    """The reduced MoE model in one reshard_refit_execute: expert weights on the reshard
    route (one launch per plan, one batch launch, or spread over side streams), attention
    and norm weights on gather-and-broadcast (the configuration's split), one shared
    scratch; every byte checked."""
    _cuda()
    w = workload(5, reduced=True)
    plans, sptrs, dptrs, wants, keep = [], [], [], [], []
    for spec in w.tensors:
        glob = global_tensor(spec)
        srcs = [helpers.to_bytes(x) for x in helpers.scatter_with_oracle(
            oracle, glob, spec.src_mesh, spec.src_placements)]
        want = helpers.expected_dst(oracle, spec, srcs)
        ds = _upload(srcs, misalign)
        dd = [Guarded(x.size, misalign) for x in want]
        plans.append(helpers.spec_plan(spec))
        sptrs.append([g.ptr for g in ds])
        dptrs.append([g.ptr for g in dd])
        wants.append(want)
        keep.append((ds, dd))
    routes = [rs.ROUTE_GATHER_BROADCAST if spec.path == "gather_broadcast" else rs.ROUTE_AUTO
              for spec in w.tensors]
    assert rs.ROUTE_GATHER_BROADCAST in routes and rs.ROUTE_AUTO in routes
    refit = rs.reshard_refit_create(plans, routes, batch=mode in ("batch", "both"),
                                    lanes=mode in ("lanes", "both"))
    got_routes, need = rs.reshard_refit_info(refit)
    assert got_routes == [rs.ROUTE_RESHARD if r == rs.ROUTE_AUTO else r for r in routes]
    scratch = Guarded(need, misalign)
    rs.reshard_refit_execute(refit, sptrs, dptrs, scratch.ptr, need)
    torch.cuda.synchronize()
    for spec, want, (ds, dd) in zip(w.tensors, wants, keep):
        for g, x in zip(dd, want):
            assert np.array_equal(g.payload().cpu().numpy(), x), spec.name
            assert g.guards_intact()
    assert scratch.guards_intact()
    assert rs.reshard_device_status() == 0


def _refit_set(oracle, w, misalign=0):
    plans, sptrs, dptrs, wants, keep = [], [], [], [], []
    for spec in w.tensors:
        glob = global_tensor(spec)
        srcs = [helpers.to_bytes(x) for x in helpers.scatter_with_oracle(
            oracle, glob, spec.src_mesh, spec.src_placements)]
        want = helpers.expected_dst(oracle, spec, srcs)
        ds = _upload(srcs, misalign)
        dd = [Guarded(x.size, misalign) for x in want]
        plans.append(helpers.spec_plan(spec))
        sptrs.append([g.ptr for g in ds])
        dptrs.append([g.ptr for g in dd])
        wants.append(want)
        keep.append((ds, dd))
    return plans, sptrs, dptrs, wants, keep


def _check_refit_set(w, wants, keep):
    for spec, want, (ds, dd) in zip(w.tensors, wants, keep):
        for r, (g, x) in enumerate(zip(dd, want)):
            assert np.array_equal(g.payload().cpu().numpy(), x), (spec.name, r)
            assert g.guards_intact()


@pytest.mark.parametrize("batch", [False, True])
@pytest.mark.parametrize("misalign", [0, 3])
def test_refit_lanes_uneven_set(oracle, misalign, batch):
    """The 60 reduced uneven-stress tensors (every copy kernel, many tiny launches) in one
    refit spread over the side streams (with batch, the TMA fan-out plans as one batch unit),
    executed twice on a non-default stream; every byte of every destination checked against
    the oracle after each execution."""
    _cuda()
    w = workload(4, reduced=True)
    plans, sptrs, dptrs, wants, keep = _refit_set(oracle, w, misalign)
    refit = rs.reshard_refit_create(plans, lanes=True, batch=batch)
    s = torch.cuda.Stream()
    for _ in range(2):
        for ds, dd in keep:
            for g in dd:
                g.payload().fill_(FILL_BYTE)
        torch.cuda.synchronize()
        rs.reshard_refit_execute(refit, sptrs, dptrs, None, 0, s)
        s.synchronize()
        _check_refit_set(w, wants, keep)
    assert rs.reshard_device_status() == 0


def test_refit_lanes_in_cuda_graph(oracle):
    """A lanes refit captured into a CUDA graph from one stream (the side streams fork from
    and join back into the capture) and replayed twice; every byte checked after each."""
    _cuda()
    w = workload(4, reduced=True)
    keep_w = type(w)(w.name, w.tensors[:24], w.note)
    plans, sptrs, dptrs, wants, keep = _refit_set(oracle, keep_w)
    refit = rs.reshard_refit_create(plans, lanes=True)
    s = torch.cuda.Stream()
    rs.reshard_refit_execute(refit, sptrs, dptrs, None, 0, s)  # first use uploads the plans
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rs.reshard_refit_execute(refit, sptrs, dptrs, None, 0, s)
    for _ in range(2):
        for ds, dd in keep:
            for x in dd:
                x.payload().fill_(FILL_BYTE)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        _check_refit_set(keep_w, wants, keep)
    assert rs.reshard_device_status() == 0


def test_refit_lanes_refuse_a_foreign_capture(oracle):
    """While a capture that took in a lanes execution is open, the side streams belong to
    it: a lanes execution from another stream is refused (UNSUPPORTED, nothing enqueued),
    and runs normally once the capture has ended."""
    _cuda()
    w = workload(4, reduced=True)
    wa = type(w)(w.name, w.tensors[:6], w.note)
    wb = type(w)(w.name, w.tensors[6:12], w.note)
    pa, sa, da, want_a, keep_a = _refit_set(oracle, wa)
    pb, sb, db, want_b, keep_b = _refit_set(oracle, wb)
    ra = rs.reshard_refit_create(pa, lanes=True)
    rb = rs.reshard_refit_create(pb, lanes=True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    rs.reshard_refit_execute(ra, sa, da, None, 0, s1)  # first use uploads the plans
    rs.reshard_refit_execute(rb, sb, db, None, 0, s2)
    torch.cuda.synchronize()
    for ds, dd in keep_a + keep_b:
        for x in dd:
            x.payload().fill_(FILL_BYTE)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1, capture_error_mode="thread_local"):
        rs.reshard_refit_execute(ra, sa, da, None, 0, s1)
        with pytest.raises(rs.ReshardError) as e:
            rs.reshard_refit_execute(rb, sb, db, None, 0, s2)
        assert e.value.status == 2
    torch.cuda.synchronize()
    for ds, dd in keep_b:                      # the refused execution wrote nothing
        for x in dd:
            assert (x.payload().cpu().numpy() == FILL_BYTE).all()
    g.replay()
    rs.reshard_refit_execute(rb, sb, db, None, 0, s2)
    torch.cuda.synchronize()
    _check_refit_set(wa, want_a, keep_a)
    _check_refit_set(wb, want_b, keep_b)
    assert rs.reshard_device_status() == 0


# ---------------------------------------------------------------------- concurrency
def test_first_use_from_several_host_threads(oracle):
    """Eight host threads execute one fresh plan at once (each into its own buffers): the
    plan's first upload is serialised and every result is exact."""
    import threading
    _cuda()
    spec = workload(2, reduced=True).tensors[0]
    glob = global_tensor(spec)
    srcs = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, srcs)
    plan = helpers.spec_plan(spec)
    dsrc = _upload(srcs)
    outs = [[Guarded(w.size) for w in want] for _ in range(8)]
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            rs.reshard_execute(plan, [g.ptr for g in dsrc], [g.ptr for g in outs[i]], s)
            s.synchronize()
        except Exception as e:  # noqa: BLE001 - collected and asserted below
            errors.append(e)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for dd in outs:
        for g, w in zip(dd, want):
            assert np.array_equal(g.payload().cpu().numpy(), w)


def test_two_plans_on_two_streams(oracle):
    _cuda()
    a, b = workload(3, reduced=True).tensors[:2]
    cases = []
    for spec in (a, b):
        glob = global_tensor(spec)
        srcs = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
            oracle, glob, spec.src_mesh, spec.src_placements)]
        want = helpers.expected_dst(oracle, spec, srcs)
        cases.append((helpers.spec_plan(spec), _upload(srcs), [Guarded(w.size) for w in want],
                      want, torch.cuda.Stream()))
    for _ in range(3):
        for plan, ds, dd, _, st in cases:
            rs.reshard_execute(plan, [g.ptr for g in ds], [g.ptr for g in dd], st)
    torch.cuda.synchronize()
    for _, _, dd, want, _ in cases:
        for g, w in zip(dd, want):
            assert np.array_equal(g.payload().cpu().numpy(), w)
