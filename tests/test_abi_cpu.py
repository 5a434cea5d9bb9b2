"""The C ABI without a GPU: the library loads, exports every declared symbol, and its
host-side entry points (planning, queries, argument checks, handle checks) behave."""
import ctypes
import math
import os
import re

import pytest

import dtensor_reshard_gb300 as rs
from inputs import workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "reshard.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("reshard_plan_create", "reshard_execute", "gather_broadcast_execute",
                     "reshard_plan_local_shape", "reshard_plan_stats", "reshard_plan_destroy",
                     "reshard_last_error"):
        assert required in names, required


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(rs.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_struct_layouts_match_header():
    assert ctypes.sizeof(rs.reshard_tile_t) == 64
    assert ctypes.sizeof(rs.reshard_mesh_t) == 40
    assert ctypes.sizeof(rs.reshard_placement_t) == 8


def _create(gshape, dtype, sm, sp, dm, dp):
    shape = (ctypes.c_int64 * max(1, len(gshape)))(*gshape)
    h = ctypes.c_void_p()
    st = rs._lib.reshard_plan_create(shape, len(gshape), dtype, ctypes.byref(rs._mesh(sm)),
                                     rs._placements(sp), ctypes.byref(rs._mesh(dm)),
                                     rs._placements(dp), ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("args,status", [
    (((8, 8), 1, (2,), ("S0",), (4,), ("S2",)), 1),           # shard dim out of range
    (((8, 8), 99, (2,), ("S0",), (4,), ("S1",)), 1),          # unknown dtype
    (((8, 8), 1, (0,), ("S0",), (4,), ("S1",)), 1),           # mesh size 0
    (((8, -1), 1, (2,), ("S0",), (4,), ("S1",)), 1),          # negative extent
    (((1, 2, 3, 4, 5), 1, (2,), ("S0",), (4,), ("S1",)), 2),  # tensor ndim 5
    (((8, 8), 1, (1, 1, 1, 1, 1), ("R",) * 5, (4,), ("S1",)), 2),  # mesh ndim 5
    (((8, 8), 1, (2,), ((7, 0),), (4,), ("S1",)), 2),         # Partial-like placement kind
])
def test_plan_create_rejects_bad_arguments(args, status):
    st, h = _create(*args)
    assert st == status, rs.reshard_last_error()
    assert not h.value
    assert rs.reshard_last_error()


def test_null_out_plan_and_null_shape():
    assert rs._lib.reshard_plan_create(None, 2, 1, None, None, None, None, None) == 1
    h = ctypes.c_void_p()
    assert rs._lib.reshard_plan_create(None, 2, 1, None, None, None, None, ctypes.byref(h)) == 1


def test_handle_checks_after_destroy():
    st, h = _create((8, 8), 1, (2,), ("S0",), (4,), ("S1",))
    assert st == 0
    assert rs._lib.reshard_plan_destroy(h) == 0
    assert rs._lib.reshard_plan_destroy(h) == 6
    s = rs.reshard_stats_t()
    assert rs._lib.reshard_plan_stats(h, ctypes.byref(s)) == 6
    assert rs._lib.reshard_execute(h, None, None, None) == 6
    assert rs._lib.reshard_plan_stats(None, ctypes.byref(s)) == 6
    # a pointer that was never a plan
    bogus = ctypes.c_void_p(ctypes.addressof(s))
    assert rs._lib.reshard_plan_stats(bogus, ctypes.byref(s)) == 6


def test_execute_argument_checks_before_any_device_work():
    p = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    srcs = (ctypes.c_void_p * 2)(None, 0x1000)   # NULL for a non-empty source shard
    dsts = (ctypes.c_void_p * 4)(0x2000, 0x3000, 0x4000, 0x5000)
    assert rs._lib.reshard_execute(p, srcs, dsts, None) == 1
    assert "source" in rs.reshard_last_error()
    assert rs._lib.reshard_execute(p, None, dsts, None) == 1
    assert rs._lib.reshard_execute_ex(p, srcs, dsts, 7, None) == 1
    full = 0x9000
    assert rs._lib.gather_broadcast_execute(p, srcs, dsts, full, 64, None) == 1  # scratch < G
    assert rs._lib.gather_broadcast_execute(p, srcs, dsts, None, 1 << 20, None) == 1


def test_too_many_ranks_for_execution_is_unsupported():
    p = rs.reshard_plan_create((4096,), "fp32", (1024,), ("S0",), (4,), ("S0",))
    srcs = (ctypes.c_void_p * 1024)(*([0x1000] * 1024))
    dsts = (ctypes.c_void_p * 4)(*([0x2000] * 4))
    assert rs._lib.reshard_execute(p, srcs, dsts, None) == 2


def test_local_shape_matches_oracle(oracle):
    for cfg in (1, 2, 3, 5):
        for spec in workload(cfg).tensors[:4]:
            p = rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                       spec.src_placements, spec.dst_mesh, spec.dst_placements)
            for side, mesh, pl in ((0, spec.src_mesh, spec.src_placements),
                                   (1, spec.dst_mesh, spec.dst_placements)):
                for r in range(math.prod(mesh)):
                    shp, off = rs.reshard_plan_local_shape(p, side, r)
                    assert (off, shp) == oracle.resolve(spec.global_shape, mesh, pl, r)
            with pytest.raises(rs.ReshardError):
                rs.reshard_plan_local_shape(p, 2, 0)
            with pytest.raises(rs.ReshardError):
                rs.reshard_plan_local_shape(p, 0, spec.n_src)


def test_stats_of_the_large_workloads():
    """Byte accounting at the full sizes (planning only, no device memory)."""
    w = workload(3)
    G = sum(t.global_bytes for t in w.tensors)
    D = 0
    for spec in w.tensors:
        s = rs.reshard_plan_stats(rs.reshard_plan_create(
            spec.global_shape, spec.dtype, spec.src_mesh, spec.src_placements, spec.dst_mesh,
            spec.dst_placements))
        assert s["region_bytes"] == s["global_bytes"] == spec.global_bytes
        assert s["fanout_read_bytes"] == spec.global_bytes
        assert s["fanout_write_bytes"] == s["dst_bytes"] == 4 * spec.global_bytes
        assert s["boxcopy_read_bytes"] == s["boxcopy_write_bytes"] == s["dst_bytes"]
        assert s["gb_read_bytes"] == s["gb_write_bytes"] == s["global_bytes"] + s["dst_bytes"]
        assert s["max_fanout"] == 4 and s["n_regions"] == 8
        D += s["dst_bytes"]
    assert G == 11_274_289_152 and D == 4 * G  # 24 x 28672 x 8192 x 2 bytes


def test_version_string():
    assert "sm_103a" in rs.reshard_version()


def test_batch_host_checks():
    import ctypes as C
    a = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    b = rs.reshard_plan_create((16,), "fp32", (4,), ("S0",), (2,), ("S0",))
    batch = rs.reshard_batch_create([a, b])
    # a plan destroyed behind the batch's back is detected before any device work
    rs.reshard_plan_destroy(b)
    sa = (C.POINTER(C.c_void_p) * 2)(C.cast(rs._ptr_array([1, 2]), C.POINTER(C.c_void_p)),
                                      C.cast(rs._ptr_array([1] * 4), C.POINTER(C.c_void_p)))
    da = (C.POINTER(C.c_void_p) * 2)(C.cast(rs._ptr_array([3] * 4), C.POINTER(C.c_void_p)),
                                      C.cast(rs._ptr_array([4, 5]), C.POINTER(C.c_void_p)))
    assert rs._lib.reshard_batch_execute(batch, sa, da, None) == 6
    rs.reshard_batch_destroy(batch)
    assert rs._lib.reshard_batch_destroy(C.c_void_p(0)) == 6
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_batch_create([b])
    assert e.value.status == 6
    # a plan with more ranks than one launch can address
    big = rs.reshard_plan_create((8192,), "fp32", (512,), ("S0",), (512,), ("S0",))
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_batch_create([big])
    assert e.value.status == 2
    # plans that only together exceed one launch's buffer table go to two launches
    wide = [rs.reshard_plan_create((4800,), "fp32", (300,), ("S0",), (300,), ("S0",))
            for _ in range(2)]
    assert rs.reshard_batch_classes(rs.reshard_batch_create(wide)) == (2, [0, 1])


def test_batch_classes():
    """Plans go into launch classes by the kernel they take with aligned buffers."""
    aligned = rs.reshard_plan_create((64, 64), "fp32", (2,), ("S0",), (4,), ("S0",))
    aligned2 = rs.reshard_plan_create((128, 32), "bf16", (4,), ("S1",), (2,), ("S1",))
    odd = rs.reshard_plan_create((7, 9), "bf16", (2,), ("S0",), (3,), ("S1",))
    odd2 = rs.reshard_plan_create((5, 11), "bf16", (3,), ("S1",), (2,), ("S0",))
    empty = rs.reshard_plan_create((0, 8), "fp32", (2,), ("S0",), (2,), ("S0",))
    batch = rs.reshard_batch_create([aligned, odd, empty, aligned2, odd2])
    n, per = rs.reshard_batch_classes(batch)
    assert per[2] == -1                      # nothing to copy
    assert per[0] == per[3] == 0             # 16-byte runs: one TMA fan-out launch
    assert per[1] != per[0] and per[4] != per[0]
    assert n == len({c for c in per if c >= 0})
    # the same plans in one class each when batched alone
    assert rs.reshard_batch_classes(rs.reshard_batch_create([odd])) == (1, [0])


def _fake_ptrs(plan, side, n, mis):
    """Distinct 256-byte aligned fake addresses + mis(rank); NULL for empty shards."""
    out = []
    for r in range(n):
        shp, _ = rs.reshard_plan_local_shape(plan, side, r)
        out.append(0 if 0 in shp else ((r + 1 + 4096 * side) << 24) + mis(r))
    return out


@pytest.mark.parametrize("gshape,dtype,sm,sp,dm,dp,smis,dmis,kernel,want", [
    # 16-byte aligned: TMA fan-out, or the 16-byte vector kernel for box copies
    ((1024, 1024), "bf16", (2,), ("S0",), (4,), ("S1",), 0, 0, 0, ("tma_fanout", 16)),
    ((1024, 1024), "bf16", (2,), ("S0",), (4,), ("S1",), 0, 0, 1, ("vector", 16)),
    # one replica, long rows, 2-byte or 1-byte alignment: staged realigning copy
    ((2000, 1301), "bf16", (3,), ("S0",), (2,), ("S0",), 0, 0, 0, ("staged", 2)),
    ((2000, 1301), "bf16", (3,), ("S0",), (2,), ("S0",), 3, 3, 0, ("staged", 1)),
    # one replica, 8-byte alignment: element kernel
    ((6971, 7418), "fp32", (49,), ("S1",), (10,), ("S1",), 0, 0, 0, ("vector", 8)),
    # one replica at 4-byte alignment: the staged kernel for long runs of a large
    # program, the element kernel for rows of 1372 bytes
    ((880, 3593, 34), "fp16", (1,), ("R",), (15,), ("S0",), 0, 0, 0, ("staged", 4)),
    ((6401, 8213), "fp32", (7,), ("S0",), (24,), ("S1",), 0, 0, 0, ("vector", 4)),
    # narrow rows (< 32 bytes): element kernel
    ((1000, 37), "bf16", (3,), ("S1",), (7,), ("S0",), 0, 0, 0, ("vector", 2)),
    # short rows (32..511 bytes) off the 16-byte grid: element kernel (a thread per
    # element column, stepping down the rows, was measured faster than 16-byte
    # granules realigned per row)
    ((731, 397), "fp16", (5,), ("S1",), (6,), ("S1",), 0, 0, 0, ("vector", 2)),
    ((731, 397), "fp16", (5,), ("S1",), (6,), ("S1",), 3, 3, 0, ("vector", 1)),
    ((900, 397), "fp16", (5,), ("S1",), (3, 2), ("R", "S1"), 0, 5, 0, ("vector", 1)),
    # fan-out, small or not in wide rows: register realigning kernel
    ((2000, 1301), "bf16", (3,), ("S0",), (2,), ("R",), 3, 3, 0, ("realign", 1)),
    # fan-out of 52.8 MB in 16 MB runs: bulk stores, unless the replicas differ mod 16
    ((4400, 6001), "bf16", (3,), ("S0",), (2,), ("R",), 0, 6, 0, ("staged_bulk", 2)),
    ((4400, 6001), "bf16", (3,), ("S0",), (2,), ("R",), 0, 5, 0, ("staged", 1)),
])
def test_plan_path_dispatch_rule(gshape, dtype, sm, sp, dm, dp, smis, dmis, kernel, want):
    p = rs.reshard_plan_create(gshape, dtype, sm, sp, dm, dp)
    src = _fake_ptrs(p, 0, p.n_src, lambda r: smis)
    # dmis == 5: replica r sits 5 * r bytes past its alignment (incongruent replicas)
    dst = _fake_ptrs(p, 1, p.n_dst, (lambda r: 5 * r) if dmis == 5 else (lambda r: dmis))
    assert rs.reshard_plan_path(p, src, dst, kernel) == want


def test_plan_path_argument_checks():
    p = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    src = _fake_ptrs(p, 0, 2, lambda r: 0)
    dst = _fake_ptrs(p, 1, 4, lambda r: 0)
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_path(p, src, dst, 7)
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_path(p, [None, src[1]], dst)
    assert e.value.status == 1
    empty = rs.reshard_plan_create((0, 7), "bf16", (2,), ("S0",), (3,), ("S1",))
    assert rs.reshard_plan_path(empty, [None, None], [None] * 3) == ("none", 1)
    out = ctypes.c_int32(-1)
    assert rs._lib.reshard_plan_path(p, rs._ptr_array(src), rs._ptr_array(dst), 0, None,
                                     ctypes.byref(out)) == 0
    assert out.value == rs.reshard_plan_path(p, src, dst)[1] == 4  # 4-byte rows


def test_refit_routes_and_host_checks():
    a = rs.reshard_plan_create((64, 64), "bf16", (2,), ("S0",), (4,), ("S1",))
    b = rs.reshard_plan_create((300, 7), "fp32", (3,), ("S1",), (2,), ("S0",))
    c = rs.reshard_plan_create((5,), "bf16", (1,), ("R",), (2,), ("R",))
    refit = rs.reshard_refit_create([a, b, c], [rs.ROUTE_AUTO, rs.ROUTE_GATHER_BROADCAST,
                                                rs.ROUTE_RESHARD])
    routes, scratch = rs.reshard_refit_info(refit)
    assert routes == [rs.ROUTE_RESHARD, rs.ROUTE_GATHER_BROADCAST, rs.ROUTE_RESHARD]
    assert scratch == 300 * 7 * 4          # the gathered tensor's global bytes
    assert rs.reshard_refit_info(rs.reshard_refit_create([a, c]))[1] == 0
    srcs = [_fake_ptrs(p, 0, p.n_src, lambda r: 0) for p in (a, b, c)]
    dsts = [_fake_ptrs(p, 1, p.n_dst, lambda r: 0) for p in (a, b, c)]
    with pytest.raises(rs.ReshardError) as e:          # no scratch for the gathered tensor
        rs.reshard_refit_execute(refit, srcs, dsts, None, 0)
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:          # scratch too small
        rs.reshard_refit_execute(refit, srcs, dsts, 0x10000, scratch - 1)
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_refit_create([a], [7])
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:
        rs._check(rs._lib.reshard_refit_create((ctypes.c_void_p * 1)(a.handle), None, 1, 8,
                                               ctypes.byref(ctypes.c_void_p())), "create")
    assert e.value.status == 1
    rs.reshard_plan_destroy(c)                          # a plan destroyed behind its back
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_refit_execute(refit, srcs, dsts, 0x10000, scratch)
    assert e.value.status == 6
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_refit_create([a, c])
    assert e.value.status == 6
    rs.reshard_refit_destroy(refit)
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_refit_destroy(refit)
    assert e.value.status == 6
    assert rs._lib.reshard_refit_destroy(ctypes.c_void_p(0)) == 6


def test_refit_batch_limit_is_reported():
    # plans that only together exceed one launch's buffer table: the batch splits them
    wide = [rs.reshard_plan_create((4096,), "fp32", (256,), ("S0",), (256,), ("S0",))
            for _ in range(2)]
    rs.reshard_refit_create(wide, batch=True)
    # a plan that alone exceeds it cannot be batched (nor executed)
    big = [rs.reshard_plan_create((8192,), "fp32", (512,), ("S0",), (512,), ("S0",))]
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_refit_create(big, batch=True)
    assert e.value.status == 2
    rs.reshard_refit_create(big, batch=False)


def test_binding_constants_come_from_the_header():
    """The binding's sizes are the header's (no hand copies that could drift)."""
    text = open(HEADER).read()

    def define(name):
        m = re.search(r"#define\s+" + name + r"\s+\(?(\d+)[uUlL]*(?:\s*<<\s*(\d+))?", text)
        assert m, name
        return int(m.group(1)) << int(m.group(2) or 0)
    assert rs.STATIC_SCRATCH_BYTES == define("RESHARD_STATIC_SCRATCH_BYTES") == 64 << 20
    assert rs.STATIC_TABLE_BYTES == define("RESHARD_STATIC_TABLE_BYTES") == 1 << 20
    assert rs.MAX_EXEC_BUFFERS == define("RESHARD_MAX_EXEC_BUFFERS")
    assert rs.MAX_TENSOR_NDIM == define("RESHARD_MAX_TENSOR_NDIM")
    assert rs.MAX_MESH_NDIM == define("RESHARD_MAX_MESH_NDIM")
    assert rs.REFIT_NUM_LANES == define("RESHARD_REFIT_NUM_LANES")


def _static_table_bytes(plan):
    """Bytes the gather and slice tables take in the static table array (256-byte slots)."""
    def a256(x):
        return (x + 255) // 256 * 256
    end = 0
    for prog in (rs.PROGRAM_GATHER, rs.PROGRAM_SLICE):
        tiles, prefix, goff, gbuf = rs.reshard_plan_program(plan, prog)
        p = a256(end + 64 * len(tiles))
        g = a256(p + 8 * len(prefix))
        b = a256(g + 4 * len(goff))
        end = a256(b + 2 * len(gbuf))
    return end


def test_static_entry_point_host_checks():
    """Every rejection of gather_broadcast_execute_static happens before device work."""
    # a 4-D tensor whose gather needs one tile per outermost index: 1.1 MiB of tables
    # for a 0.5 MiB tensor
    p = rs.reshard_plan_create((2048, 4, 4, 4), "fp32", (2, 2, 2), ("S1", "S2", "S3"),
                               (2,), ("S0",))
    assert rs.reshard_plan_stats(p)["global_bytes"] <= rs.STATIC_SCRATCH_BYTES
    assert _static_table_bytes(p) > rs.STATIC_TABLE_BYTES
    srcs = (ctypes.c_void_p * 8)(*([0x1000] * 8))
    dsts = (ctypes.c_void_p * 2)(0x2000, 0x3000)
    assert rs._lib.gather_broadcast_execute_static(p, srcs, dsts, None) == 2
    assert "static table" in rs.reshard_last_error()
    # half the outer extent fits
    q = rs.reshard_plan_create((1024, 4, 4, 4), "fp32", (2, 2, 2), ("S1", "S2", "S3"),
                               (2,), ("S0",))
    assert _static_table_bytes(q) <= rs.STATIC_TABLE_BYTES
    # the global tensor above the scratch
    rows = rs.STATIC_SCRATCH_BYTES // (2 * 4096) + 1
    big = rs.reshard_plan_create((rows, 4096), "bf16", (2,), ("S0",), (2,), ("S1",))
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    assert rs._lib.gather_broadcast_execute_static(big, two, two, None) == 2
    assert "static scratch" in rs.reshard_last_error()
    # pointer checks are the library's own: NULL for a non-empty shard, bad handle
    w = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    nul = (ctypes.c_void_p * 2)(None, 0x1000)
    four = (ctypes.c_void_p * 4)(0x2000, 0x3000, 0x4000, 0x5000)
    assert rs._lib.gather_broadcast_execute_static(w, nul, four, None) == 1
    assert "source" in rs.reshard_last_error()
    assert rs._lib.gather_broadcast_execute_static(w, None, four, None) == 1
    assert rs._lib.gather_broadcast_execute_static(None, two, four, None) == 6


def test_static_entry_point_checks_inplace_aliases():
    """An in-place plan's source pointers must alias the destinations, as elsewhere."""
    # generation rank 4t+d holds training shards 4t..4t+3; training shard s lives in rank s
    p = rs.reshard_plan_create_inplace((64, 16), "fp32", (8,), ("S0",), (2, 4), ("S0", "R"),
                                       src_alias=list(range(8)))
    n_src, n_dst = p.n_src, p.n_dst
    srcs = (ctypes.c_void_p * n_src)(*[0x10000 * (i + 1) for i in range(n_src)])
    dsts = (ctypes.c_void_p * n_dst)(*[0x1000000 * (i + 1) for i in range(n_dst)])
    assert rs._lib.gather_broadcast_execute_static(p, srcs, dsts, None) == 1
    assert "in-place" in rs.reshard_last_error()
