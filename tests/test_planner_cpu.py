"""The planner's copy programs, executed on the CPU by a test-only tile executor and
compared with the oracle; invariants of the tiles and of the replica choice."""
import math
import random

import numpy as np
import pytest
import torch

import dtensor_reshard_gb300 as rs
from inputs import TensorSpec, global_tensor, workload
from tests import helpers
from tests import torch_chunk_layout as tcl


def _case(gshape, dtype, sm, sp, dm, dp, seed):
    return TensorSpec("case", tuple(gshape), dtype, tuple(sm), tuple(sp), tuple(dm), tuple(dp),
                      init=("bits",), seed=seed)


def _check_spec(oracle, spec, programs=(0, 1)):
    glob = global_tensor(spec)
    srcs = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, srcs)
    plan = helpers.spec_plan(spec)
    for program in programs:
        dsts = [np.full(w.size, 0xA5, dtype=np.uint8) for w in want]
        bufs = [s.copy() for s in srcs] + dsts + [np.zeros(0, dtype=np.uint8)]
        writes = helpers.run_program_cpu(plan, program, bufs)
        M = spec.n_src
        for r, w in enumerate(want):
            assert np.array_equal(bufs[M + r], w), (spec, program, r)
            assert (writes[M + r] == 1).all(), ("each dst byte written exactly once", spec, r)
        for s in range(M):
            assert not writes[s].any(), "sources must not be written"
    # gather-and-broadcast: gather covers the full tensor once, slice fills every dst
    G = spec.global_bytes
    dsts = [np.full(w.size, 0x5A, dtype=np.uint8) for w in want]
    bufs = [s.copy() for s in srcs] + dsts + [np.zeros(G, dtype=np.uint8)]
    wg = helpers.run_program_cpu(plan, rs.PROGRAM_GATHER, bufs)
    assert (wg[-1] == 1).all()
    assert np.array_equal(bufs[-1], helpers.to_bytes(glob))
    ws = helpers.run_program_cpu(plan, rs.PROGRAM_SLICE, bufs)
    for r, w in enumerate(want):
        assert np.array_equal(bufs[spec.n_src + r], w)
        assert (ws[spec.n_src + r] == 1).all()
    return plan


def test_worked_example_programs(oracle):
    _check_spec(oracle, workload(1).tensors[0])


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_reduced_workloads(oracle, cfg):
    w = workload(cfg, reduced=True)
    for spec in w.tensors[:4]:
        _check_spec(oracle, spec)


@pytest.mark.parametrize("case,transposed", [
    # 45 pieces of 32 bytes cut out of 1430-byte rows: transpose blocks
    (((6, 40, 715), "bf16", (6,), ("S0",), (45,), ("S2",)), True),
    # 18 narrow sources of 32 bytes into one destination replica: transpose blocks
    (((200, 288), "bf16", (18,), ("S1",), (4,), ("S0",)), True),
    # 3-D gather: 31 narrow sources of 8 bytes whose rows break into planes of 8 rows
    (((10, 30, 122), "bf16", (32,), ("S2",), (4,), ("S1",)), True),
    # 3-D scatter: 20 pieces of 30 bytes into destinations cut along the middle dim too
    (((10, 40, 300), "bf16", (4,), ("S1",), (20,), ("S2",)), True),
    # scatter of pieces of 34 bytes: per-piece copies
    (((6, 40, 765), "bf16", (6,), ("S0",), (45,), ("S2",)), False),
    # gather of 42 pieces of 68 bytes into 2832-byte rows (7 per block), 3-D: transposed
    (((3, 40, 1416), "bf16", (42,), ("S2",), (5,), ("S1",)), True),
    # gather of 46 pieces of 206 bytes: too wide
    (((40, 4717), "bf16", (46,), ("S1",), (1,), ("S1",)), False),
    # gather of 32 pieces of 128 bytes into 4 KB rows: transposed
    (((40, 1024), "fp32", (32,), ("S1",), (4,), ("S0",)), True),
    # gather of 80 pieces of 128 bytes into 10 KB rows (two per block): per-piece copies
    (((40, 2560), "fp32", (80,), ("S1",), (4,), ("S0",)), False),
    # a 3-way de-interleave of 6-byte rows: transposed
    (((200, 50, 3), "fp16", (1,), ("S1",), (45,), ("S2",)), True),
    # a 2-way de-interleave of 6-byte rows into pieces of 4 and 2 bytes: transposed
    (((200, 50, 3), "fp16", (1,), ("S1",), (2,), ("S2",)), True),
    # 8 pieces of 4 bytes out of 32-byte rows (too few): per-piece copies
    (((60, 50, 8), "fp32", (8,), ("S0",), (17,), ("S2",)), False),
])
def test_transpose_rule_for_narrow_pieces(oracle, case, transposed):
    """Narrow innermost pieces (at least 16 of them, at most 32 bytes per row, or up to 128
    bytes gathered into rows short enough for four per block, or any pieces scattered out of
    rows of at most 8 bytes) are regrouped into transpose blocks, in planes of rows where the rows do not collapse into one level; wider or fewer
    pieces stay per-piece tiles.  Either way the program, executed on the
    CPU, reproduces the oracle."""
    spec = _case(*case, seed=9)
    plan = _check_spec(oracle, spec)
    blocks, _ = rs.reshard_plan_transposes(plan, rs.PROGRAM_FANOUT)
    assert bool(blocks) == transposed
    # a block flagged as having the previous block's shape has it: same wide side,
    # direction, rows and segments (widths, columns, narrow sides), other offsets
    blocks, segs = rs.reshard_plan_transposes(plan, rs.PROGRAM_FANOUT)
    flagged = 0
    for i, b in enumerate(blocks):
        if not b["flags"] & 1:
            continue
        flagged += 1
        assert i > 0
        a = blocks[i - 1]
        for f in ("wide", "direction", "row_bytes", "nrows", "seg_count"):
            assert a[f] == b[f], (i, f)
        for k in range(b["seg_count"]):
            x, y = segs[a["seg_begin"] + k], segs[b["seg_begin"] + k]
            assert (x["width"], x["col"], x["narrow"]) == (y["width"], y["col"], y["narrow"])
            if b["flags"] & 2:   # follows: offsets advanced by the previous block's rows
                assert y["narrow_off"] == x["narrow_off"] + a["nrows"] * x["width"]
        if b["flags"] & 2:
            assert b["wide_off"] == a["wide_off"] + a["nrows"] * a["row_bytes"]
    if blocks:
        assert flagged >= len(blocks) // 2 or len(blocks) < 4
    # transpose blocks are a fan-out device only: the box-copy, gather, slice and
    # replicate programs (which the allocation-free entry point runs from tables at
    # explicit addresses) stay tiles alone
    for prog in (rs.PROGRAM_BOXCOPY, rs.PROGRAM_GATHER, rs.PROGRAM_SLICE, rs.PROGRAM_REPLICATE):
        blocks, segs = rs.reshard_plan_transposes(plan, prog)
        assert not blocks and not segs, prog


@pytest.mark.parametrize("case,assembled", [
    # 14 column bands of 632 bytes (off the 16-byte grid) into 9 replicas: assembled
    (((60, 2200), "fp32", (14,), ("S1",), (9,), ("R",)), 1),
    # two destination classes of 12 replicas each, bands of 632 bytes in 3-D: assembled
    (((2, 30, 4424), "bf16", (2, 14), ("R", "S2"), (2, 12), ("S0", "R")), 2),
    # 6 replicas: assembled; 5: too few
    (((60, 2200), "fp32", (14,), ("S1",), (6,), ("R",)), 1),
    (((60, 2200), "fp32", (14,), ("S1",), (5,), ("R",)), 0),
    # bands of 640 bytes, on the 16-byte grid: the TMA fan-out takes them directly
    (((60, 2240), "fp32", (14,), ("S1",), (9,), ("R",)), 0),
    # one source region per shard (a replicated tensor): nothing to assemble
    (((60, 2201), "fp32", (3,), ("R",), (9,), ("R",)), 0),
])
def test_assemble_then_replicate(oracle, case, assembled):
    """Destination shards that many replicas need, cut from pieces off the 16-byte grid, are
    assembled in their first replica and then copied as one run to the others: every byte
    written once, the oracle's result, and traffic G + D plus one read per assembled shard."""
    spec = _case(*case, seed=5)
    plan = _check_spec(oracle, spec)
    st = rs.reshard_plan_stats(plan)
    assert st["assembled_classes"] == assembled
    tiles, _, goff, gbuf = rs.reshard_plan_program(plan, rs.PROGRAM_REPLICATE)
    assert len(tiles) == st["n_replicate_tiles"] == assembled
    M = spec.n_src
    shard = 0
    for t in tiles:
        first = t["src_buf"] - M
        others = [b - M for b in gbuf[goff[t["dst_group"]]:goff[t["dst_group"] + 1]]]
        assert first not in others
        shp, _ = rs.reshard_plan_local_shape(plan, 1, first)
        assert t["row_bytes"] == math.prod(shp) * spec.elem_bytes and t["src_off"] == 0
        for r in others:
            assert rs.reshard_plan_local_shape(plan, 1, r) == rs.reshard_plan_local_shape(
                plan, 1, first)
        shard += t["row_bytes"]
    assert st["fanout_read_bytes"] == st["global_bytes"] + shard
    assert st["fanout_write_bytes"] == st["dst_bytes"]


def test_uneven_stress_reduced(oracle):
    for spec in workload(4, reduced=True).tensors:
        _check_spec(oracle, spec)


def test_bruteforce_small_layouts(oracle):
    rng = random.Random(17)
    layouts = {nd: [(m, p) for m in tcl.all_meshes(4) for p in tcl.all_placements(len(m), nd)]
               for nd in (1, 2, 3)}
    for i in range(400):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(0 if rng.random() < 0.05 else 1, 7) for _ in range(nd))
        (sm, sp), (dm, dp) = rng.choice(layouts[nd]), rng.choice(layouts[nd])
        dtype = rng.choice(("u8", "bf16", "fp32", "fp64"))
        _check_spec(oracle, _case(gshape, dtype, sm, sp, dm, dp, seed=i))


def test_four_dim_tensors(oracle):
    rng = random.Random(5)
    for i in range(40):
        gshape = tuple(rng.randint(1, 5) for _ in range(4))
        sm = tuple(rng.randint(1, 3) for _ in range(rng.randint(1, 3)))
        dm = tuple(rng.randint(1, 3) for _ in range(rng.randint(1, 3)))
        sp = tuple(rng.choice(["R", "S0", "S1", "S2", "S3"]) for _ in sm)
        dp = tuple(rng.choice(["R", "S0", "S1", "S2", "S3"]) for _ in dm)
        _check_spec(oracle, _case(gshape, "fp16", sm, sp, dm, dp, seed=100 + i))


def test_unit_prefix_matches_tile_units():
    spec = workload(5, reduced=True).tensors[2]
    plan = helpers.spec_plan(spec)
    for program in range(4):
        tiles, prefix, _, _ = rs.reshard_plan_program(plan, program)
        assert prefix[0] == 0
        for i, t in enumerate(tiles):
            assert prefix[i + 1] - prefix[i] == rs.reshard_tile_units(t) > 0


def test_tiles_sorted_by_destination():
    spec = workload(5, reduced=True).tensors[0]
    plan = helpers.spec_plan(spec)
    tiles, _, goff, gbuf = rs.reshard_plan_program(plan, rs.PROGRAM_FANOUT)
    keys = [(gbuf[goff[t["dst_group"]]], t["dst_off"]) for t in tiles]
    assert keys == sorted(keys)


def test_replica_load_balance():
    """Greedy largest-first: within a source class, replica loads differ by at most one region."""
    rng = random.Random(9)
    checked = 0
    for i in range(300):
        nd = rng.choice((1, 2))
        gshape = tuple(rng.randint(1, 40) for _ in range(nd))
        sm = (rng.randint(2, 4), rng.randint(1, 4))
        sp = ("R", f"S{rng.randrange(nd)}")
        dm = (rng.randint(1, 8),)
        dp = (f"S{rng.randrange(nd)}",)
        plan = rs.reshard_plan_create(gshape, "bf16", sm, sp, dm, dp)
        tiles, _, goff, _ = rs.reshard_plan_program(plan, rs.PROGRAM_FANOUT)
        load = {}
        for t in tiles:
            b = t["row_bytes"] * t["nrows"] * t["nplanes"]
            load[t["src_buf"]] = load.get(t["src_buf"], 0) + b
        # group source ranks by their box (replicas)
        classes = {}
        for r in range(math.prod(sm)):
            shp, off = rs.reshard_plan_local_shape(plan, 0, r)
            classes.setdefault((shp, off), []).append(r)
        # largest region = largest source box x destination box intersection
        biggest = 0
        for r in range(math.prod(dm)):
            dshp, doff = rs.reshard_plan_local_shape(plan, 1, r)
            for (sshp, soff) in classes:
                v = 2
                for a, b, c, d in zip(soff, sshp, doff, dshp):
                    v *= max(0, min(a + b, c + d) - max(a, c))
                biggest = max(biggest, v)
        for ranks in classes.values():
            if len(ranks) < 2:
                continue
            loads = [load.get(r, 0) for r in ranks]
            assert max(loads) - min(loads) <= biggest, (gshape, sm, sp, dm, dp, loads)
            checked += 1
    assert checked > 100


def test_fanout_groups_hybridflow():
    """Training TP8 -> (TP2, DP4): each region is one fan-out record to 4 replicas."""
    spec = workload(3).tensors[0]
    plan = helpers.spec_plan(spec)
    tiles, _, goff, gbuf = rs.reshard_plan_program(plan, rs.PROGRAM_FANOUT)
    sizes = {goff[g + 1] - goff[g] for g in range(len(goff) - 1)}
    assert sizes == {4}
    st = rs.reshard_plan_stats(plan)
    assert st["fanout_read_bytes"] == spec.global_bytes
    assert st["fanout_write_bytes"] == 4 * spec.global_bytes
    # every region is one contiguous 58.7 MB run, cut into run tiles
    assert all(t["nrows"] == 1 and t["nplanes"] == 1 for t in tiles)
    assert sum(t["row_bytes"] for t in tiles) == spec.global_bytes


def test_moe_down_is_strided_rows():
    """Down projection [E, 7168, 2048] Shard(ffn): 512-byte rows at a 2 KiB source stride."""
    spec = workload(5).tensors[2]
    plan = helpers.spec_plan(spec)
    tiles, _, goff, _ = rs.reshard_plan_program(plan, rs.PROGRAM_FANOUT)
    assert all(t["row_bytes"] == 512 and t["src_row_stride"] == 2048
               and t["dst_row_stride"] == 512 for t in tiles)
    assert {goff[g + 1] - goff[g] for g in range(len(goff) - 1)} == {2}


def test_planner_scale_pages_layout():
    """The pages' TP4 x PP8 x EP16 -> TP8 x DP16 layout (512 -> 128 ranks), planning only."""
    gshape = (128, 2048, 7168)
    plan = rs.reshard_plan_create(gshape, "bf16", (4, 8, 16), ("S1", "R", "S0"), (8, 16),
                                  ("S1", "R"))
    st = rs.reshard_plan_stats(plan)
    G = math.prod(gshape) * 2
    assert st["region_bytes"] == G
    assert st["dst_bytes"] == 16 * G
    assert st["n_src_ranks"] == 512 and st["n_dst_ranks"] == 128
    assert st["planner_ns"] < 2e9


def test_empty_and_degenerate_layouts(oracle):
    # zero-size tensor, more ranks than elements, size-1 meshes
    for spec in (_case((0, 5), "bf16", (2,), ("S0",), (3,), ("S1",), 1),
                 _case((3,), "fp32", (8,), ("S0",), (5,), ("S0",), 2),
                 _case((5, 1), "bf16", (1, 1), ("R", "S1"), (1,), ("R",), 3),
                 _case((1, 1, 1), "u8", (2, 2), ("S0", "S2"), (3,), ("S1",), 4)):
        _check_spec(oracle, spec)


# ------------------------------------------------------------------------------ in place
def _inplace_cpu(oracle, spec, alias):
    glob = global_tensor(spec)
    sboxes = oracle.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    dboxes = oracle.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
    srcs = [helpers.to_bytes(helpers.slice_box(glob, o, s)) for o, s in sboxes]
    want = helpers.expected_dst(oracle, spec, srcs)
    plan = rs.reshard_plan_create_inplace(spec.global_shape, spec.dtype, spec.src_mesh,
                                          spec.src_placements, spec.dst_mesh,
                                          spec.dst_placements, alias)
    M = spec.n_src
    for program in (rs.PROGRAM_FANOUT, rs.PROGRAM_BOXCOPY):
        dsts = [np.full(w.size, 0xA5, dtype=np.uint8) for w in want]
        views = []
        for s, a in enumerate(alias):
            d, off = rs.reshard_plan_alias(plan, s)
            if a >= 0 and srcs[s].size:
                assert d == a and off == helpers.alias_offset_bytes(sboxes[s], dboxes[a],
                                                                    spec.elem_bytes)
                v = dsts[a][off:off + srcs[s].size]
                v[:] = srcs[s]
                views.append(v)
            else:
                views.append(srcs[s].copy())
        bufs = views + dsts + [np.zeros(0, dtype=np.uint8)]
        writes = helpers.run_program_cpu(plan, program, bufs)
        for r, w in enumerate(want):
            assert np.array_equal(dsts[r], w), (spec, program, r)
            assert (writes[M + r] <= 1).all()
        # no copy writes a byte that is a source of the same execution
        for s, a in enumerate(alias):
            if a >= 0 and srcs[s].size:
                _, off = rs.reshard_plan_alias(plan, s)
                assert not writes[M + a][off:off + srcs[s].size].any()
    st = rs.reshard_plan_stats(plan)
    assert st["fanout_write_bytes"] + st["inplace_bytes"] == st["dst_bytes"]
    return st


def test_inplace_hybridflow(oracle):
    """Strided generation ranks: every training shard is already inside its rank's
    generation shard, so a quarter of the destination bytes are never written."""
    for spec in workload(3, reduced=False).tensors[:1] + (
            TensorSpec("hf", (64, 24), "bf16", (8,), ("S0",), (2, 4), ("S0", "R"),
                       init=("bits",), seed=3),):
        if spec.numel > 1 << 22:
            plan = rs.reshard_plan_create_inplace(spec.global_shape, spec.dtype, spec.src_mesh,
                                                  spec.src_placements, spec.dst_mesh,
                                                  spec.dst_placements, list(range(8)))
            st = rs.reshard_plan_stats(plan)
            assert st["inplace_bytes"] == spec.global_bytes
            assert st["fanout_write_bytes"] == 3 * spec.global_bytes
            continue
        st = _inplace_cpu(oracle, spec, list(range(8)))
        assert st["inplace_bytes"] == spec.global_bytes


def test_inplace_random_layouts(oracle):
    rng = random.Random(23)
    done = 0
    for i in range(400):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 9) for _ in range(nd))
        sm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        dm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        sp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in sm)
        dp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in dm)
        spec = _case(gshape, "bf16", sm, sp, dm, dp, seed=i)
        alias = helpers.pick_aliases(oracle, spec, rng)
        if all(a < 0 for a in alias):
            continue
        _inplace_cpu(oracle, spec, alias)
        done += 1
    assert done > 50


def test_inplace_rejects_impossible_aliases():
    # source rank 0 (rows 0-3) is not inside destination rank 1 (rows 4-7)
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_create_inplace((8, 8), "bf16", (2,), ("S0",), (2,), ("S0",), [1, -1])
    assert e.value.status == 3
    # a 4x4 corner inside the full 8x8 matrix: inside, but not one contiguous range
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_create_inplace((8, 8), "bf16", (2, 2), ("S0", "S1"), (1,), ("R",),
                                       [0, -1, -1, -1])
    assert e.value.status == 3
    with pytest.raises(rs.ReshardError):
        rs.reshard_plan_create_inplace((8, 8), "bf16", (2,), ("S0",), (2,), ("S0",), [5, -1])


def test_inplace_execute_requires_aliased_pointers():
    import ctypes
    plan = rs.reshard_plan_create_inplace((8, 8), "bf16", (2,), ("S0",), (2, 2), ("S0", "R"),
                                          [0, 2])
    dsts = [0x10000, 0x20000, 0x30000, 0x40000]
    # source 1 sits inside destination 2 at its offset; source 0 points elsewhere
    srcs = [0x90000, 0x30000 + rs.reshard_plan_alias(plan, 1)[1]]
    rc = rs._lib.reshard_execute(plan, rs._ptr_array(srcs), rs._ptr_array(dsts), None)
    assert rc == 1 and "in-place" in rs.reshard_last_error()
    del ctypes


# ---------------------------------------------------------------------- membership change
def _check_excluded(oracle, spec, src_gone, dst_gone):
    """Run the derived plan's programs on the CPU with zero-length buffers for the gone
    ranks (any access to one fails the executor's bounds check); every remaining
    destination must match the oracle and be written exactly once."""
    glob = global_tensor(spec)
    srcs = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
        oracle, glob, spec.src_mesh, spec.src_placements)]
    want = helpers.expected_dst(oracle, spec, srcs)
    plan = rs.reshard_plan_exclude(helpers.spec_plan(spec), src_gone, dst_gone)
    M = spec.n_src
    empty = np.zeros(0, dtype=np.uint8)
    for program in (rs.PROGRAM_FANOUT, rs.PROGRAM_BOXCOPY):
        bufs = ([empty if s in src_gone else srcs[s].copy() for s in range(M)] +
                [empty if r in dst_gone else np.full(w.size, 0xA5, dtype=np.uint8)
                 for r, w in enumerate(want)] + [empty])
        writes = helpers.run_program_cpu(plan, program, bufs)
        for r, w in enumerate(want):
            if r in dst_gone:
                continue
            assert np.array_equal(bufs[M + r], w), (spec.name, program, r)
            assert (writes[M + r] == 1).all()
    # gather-and-broadcast: the slice of every remaining destination is exact
    bufs = ([empty if s in src_gone else srcs[s].copy() for s in range(M)] +
            [empty if r in dst_gone else np.zeros(w.size, dtype=np.uint8)
             for r, w in enumerate(want)] + [np.zeros(spec.global_bytes, dtype=np.uint8)])
    helpers.run_program_cpu(plan, rs.PROGRAM_GATHER, bufs)
    helpers.run_program_cpu(plan, rs.PROGRAM_SLICE, bufs)
    for r, w in enumerate(want):
        if r not in dst_gone:
            assert np.array_equal(bufs[M + r], w), (spec.name, "gather-broadcast", r)
    return plan


def _shard_bytes(plan, side, ranks, spec):
    return sum(math.prod(rs.reshard_plan_local_shape(plan, side, r)[0]) for r in ranks) * \
        spec.elem_bytes


def test_exclude_source_replicas_rebalances(oracle):
    # FFN up (reduced): every source box has two replicas (DP2)
    spec = workload(2, reduced=True).tensors[0]
    base = helpers.spec_plan(spec)
    plan = _check_excluded(oracle, spec, src_gone=[0, 5], dst_gone=[])
    s0, s1 = rs.reshard_plan_stats(base), rs.reshard_plan_stats(plan)
    assert s1["fanout_read_bytes"] == s0["fanout_read_bytes"]     # still read once
    assert s1["src_bytes"] == s0["src_bytes"] - _shard_bytes(base, 0, [0, 5], spec)
    tiles, _, _, _ = rs.reshard_plan_program(plan, rs.PROGRAM_FANOUT)
    assert {t["src_buf"] for t in tiles}.isdisjoint({0, 5})


def test_exclude_destination_ranks(oracle):
    spec = workload(2, reduced=True).tensors[0]
    base = helpers.spec_plan(spec)
    plan = _check_excluded(oracle, spec, src_gone=[], dst_gone=[1, 6])
    s0, s1 = rs.reshard_plan_stats(base), rs.reshard_plan_stats(plan)
    assert s1["dst_bytes"] == s0["dst_bytes"] - _shard_bytes(base, 1, [1, 6], spec)
    assert s1["fanout_write_bytes"] == s1["dst_bytes"]


def test_exclude_both_sides_random(oracle):
    rng = random.Random(77)
    for i in range(12):
        spec = _case((rng.randint(1, 40), rng.randint(1, 40)), "bf16", (2, 2),
                     ("R", rng.choice(["S0", "S1"])), (3,), (rng.choice(["R", "S0", "S1"]),),
                     seed=900 + i)
        src_gone = [rng.choice([0, 1])] if rng.random() < 0.7 else []   # one replica of a pair
        dst_gone = [rng.randrange(3)] if rng.random() < 0.5 else []
        _check_excluded(oracle, spec, src_gone, dst_gone)


def test_exclude_without_a_remaining_source_is_unsupported():
    p = rs.reshard_plan_create((8, 8), "bf16", (2,), ("S0",), (4,), ("S1",))
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_exclude(p, [1])
    assert e.value.status == 2
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_exclude(p, [2])
    assert e.value.status == 1
    with pytest.raises(rs.ReshardError) as e:
        rs.reshard_plan_exclude(p, [], [4])
    assert e.value.status == 1


def test_rank_rejoining_restores_the_plan():
    spec = workload(2, reduced=True).tensors[0]
    base = helpers.spec_plan(spec)
    gone = rs.reshard_plan_exclude(base, [0], [2])
    back = rs.reshard_plan_exclude(gone, [], [])
    for program in range(4):
        a, pa, _, _ = rs.reshard_plan_program(base, program)
        b, pb, _, _ = rs.reshard_plan_program(back, program)
        assert [dict(t) for t in a] == [dict(t) for t in b] and list(pa) == list(pb)
    assert rs.reshard_plan_stats(back)["dst_bytes"] == rs.reshard_plan_stats(base)["dst_bytes"]


def test_exclude_drops_aliases_of_gone_ranks(oracle):
    spec = workload(3, reduced=True).tensors[0]
    alias = helpers.pick_aliases(oracle, spec)
    s = next(i for i, d in enumerate(alias) if d >= 0)
    base = rs.reshard_plan_create_inplace(spec.global_shape, spec.dtype, spec.src_mesh,
                                          spec.src_placements, spec.dst_mesh,
                                          spec.dst_placements, alias)
    plan = rs.reshard_plan_exclude(base, [], [alias[s]])
    assert rs.reshard_plan_alias(plan, s)[0] == -1
    assert rs.reshard_plan_alias(base, s)[0] == alias[s]
