"""Test helpers: scattering with the oracle's layout, a CPU executor of plan tiles.

The CPU tile executor is test code that runs the library's copy programs on
host byte buffers, so planner mistakes show up without a GPU.  It is never used
by the library or the benchmark.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import dtensor_reshard_gb300 as rs


def oracle_boxes(o, gshape, mesh, placements):
    return o.boxes(gshape, mesh, placements)


def slice_box(t: torch.Tensor, off, shp) -> torch.Tensor:
    """Contiguous local shard of a global tensor for a box (offset, shape)."""
    if math.prod(shp) == 0:
        return t.new_empty(tuple(shp))
    sl = tuple(slice(a, a + b) for a, b in zip(off, shp))
    return t[sl].contiguous()


def to_bytes(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous().cpu()
    if t.numel() == 0:
        return np.zeros(0, dtype=np.uint8)
    return t.view(torch.uint8).reshape(-1).numpy().copy()


def scatter_with_oracle(o, glob: torch.Tensor, mesh, placements):
    """Source shards (contiguous tensors) of ``glob`` under a layout, by the oracle's boxes."""
    gshape = tuple(glob.shape)
    return [slice_box(glob, off, shp) for off, shp in oracle_boxes(o, gshape, mesh, placements)]


def expected_dst(o, spec, src_bytes):
    """Oracle's destination byte buffers for a TensorSpec-like object."""
    return o.reshard(spec.global_shape, spec.elem_bytes, spec.src_mesh, spec.src_placements,
                     spec.dst_mesh, spec.dst_placements, src_bytes)


def run_program_cpu(plan, program, bufs):
    """Execute one copy program of ``plan`` on host buffers (list of uint8 arrays).

    ``bufs`` is the buffer table [sources..., destinations..., scratch].  Returns,
    per buffer, a count array of how many times each byte was written.
    """
    writes = [np.zeros(b.size, dtype=np.int32) for b in bufs]
    _run_tiles_cpu(plan, program, bufs, writes)
    run_transposes_cpu(plan, program, bufs, writes)
    if program == rs.PROGRAM_FANOUT:
        # second step: destination shards assembled in one replica, copied to the others
        _run_tiles_cpu(plan, rs.PROGRAM_REPLICATE, bufs, writes)
    return writes


def _run_tiles_cpu(plan, program, bufs, writes):
    tiles, prefix, goff, gbuf = rs.reshard_plan_program(plan, program)
    for t in tiles:
        src = bufs[t["src_buf"]]
        for g in range(goff[t["dst_group"]], goff[t["dst_group"] + 1]):
            di = gbuf[g]
            dst = bufs[di]
            for p in range(t["nplanes"]):
                for r in range(t["nrows"]):
                    so = t["src_off"] + p * t["src_plane_stride"] + r * t["src_row_stride"]
                    do = t["dst_off"] + p * t["dst_plane_stride"] + r * t["dst_row_stride"]
                    n = t["row_bytes"]
                    assert 0 <= so and so + n <= src.size, ("source out of bounds", t)
                    assert 0 <= do and do + n <= dst.size, ("destination out of bounds", t)
                    dst[do:do + n] = src[so:so + n]
                    writes[di][do:do + n] += 1


def run_transposes_cpu(plan, program, bufs, writes):
    """Execute a program's transpose blocks on host buffers (test only)."""
    blocks, segs = rs.reshard_plan_transposes(plan, program)
    _, _, goff, gbuf = rs.reshard_plan_program(plan, program)
    for b in blocks:
        L, nr = b["row_bytes"], b["nrows"]
        for k in range(b["seg_begin"], b["seg_begin"] + b["seg_count"]):
            sg = segs[k]
            w, col = sg["width"], sg["col"]
            if b["direction"] == 0:   # narrow source -> wide destination group
                src = bufs[sg["narrow"]][sg["narrow_off"]:sg["narrow_off"] + nr * w]
                assert src.size == nr * w, ("source out of bounds", b, sg)
                for di in gbuf[goff[b["wide"]]:goff[b["wide"] + 1]]:
                    lo = b["wide_off"]
                    assert lo >= 0 and lo + nr * L <= bufs[di].size, ("dst out of bounds", b)
                    bufs[di][lo:lo + nr * L].reshape(nr, L)[:, col:col + w] = src.reshape(nr, w)
                    writes[di][lo:lo + nr * L].reshape(nr, L)[:, col:col + w] += 1
            else:                      # wide source -> narrow destination group
                lo = b["wide_off"]
                wide = bufs[b["wide"]][lo:lo + nr * L]
                assert wide.size == nr * L, ("source out of bounds", b)
                piece = wide.reshape(nr, L)[:, col:col + w].reshape(-1)
                for di in gbuf[goff[sg["narrow"]]:goff[sg["narrow"] + 1]]:
                    o = sg["narrow_off"]
                    assert o >= 0 and o + nr * w <= bufs[di].size, ("dst out of bounds", sg)
                    bufs[di][o:o + nr * w] = piece
                    writes[di][o:o + nr * w] += 1


def spec_plan(spec):
    return rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                  spec.src_placements, spec.dst_mesh, spec.dst_placements)


def contiguous_inside(src_box, dst_box):
    """True when src_box lies in dst_box as one contiguous range of dst's row-major layout."""
    (so, ss), (do, ds) = src_box, dst_box
    if math.prod(ss) == 0:
        return False
    for a, b, c, d in zip(so, ss, do, ds):
        if a < c or a + b > c + d:
            return False
    k0 = next((k for k, e in enumerate(ss) if e != 1), len(ss))
    return all(ss[k] == ds[k] for k in range(k0 + 1, len(ss)))


def alias_offset_bytes(src_box, dst_box, elem_bytes):
    (so, _), (do, ds) = src_box, dst_box
    strides = [math.prod(ds[k + 1:]) for k in range(len(ds))]
    return sum((a - c) * st for a, c, st in zip(so, do, strides)) * elem_bytes


def pick_aliases(o, spec, rng=None):
    """A valid in-place alias map (first containing destination rank, or -1)."""
    sb = o.boxes(spec.global_shape, spec.src_mesh, spec.src_placements)
    db = o.boxes(spec.global_shape, spec.dst_mesh, spec.dst_placements)
    out = []
    for s in range(len(sb)):
        cands = [d for d in range(len(db)) if contiguous_inside(sb[s], db[d])]
        if not cands or (rng is not None and rng.random() < 0.25):
            out.append(-1)
        else:
            out.append(cands[0] if rng is None else rng.choice(cands))
    return out


# ------------------------------------------------------------------ partition on the CPU
def run_tile_list_cpu(tiles, goff, gbuf, bufs, writes):
    """Execute a list of tiles (as the program views give them) on host buffers."""
    for t in tiles:
        src = bufs[t["src_buf"]]
        for g in range(goff[t["dst_group"]], goff[t["dst_group"] + 1]):
            di = gbuf[g]
            dst = bufs[di]
            for p in range(t["nplanes"]):
                for r in range(t["nrows"]):
                    so = t["src_off"] + p * t["src_plane_stride"] + r * t["src_row_stride"]
                    do = t["dst_off"] + p * t["dst_plane_stride"] + r * t["dst_row_stride"]
                    n = t["row_bytes"]
                    assert src is not None and dst is not None, ("buffer not on this gpu", t)
                    assert 0 <= so and so + n <= src.size, ("source out of bounds", t)
                    assert 0 <= do and do + n <= dst.size, ("destination out of bounds", t)
                    dst[do:do + n] = src[so:so + n]
                    writes[di][do:do + n] += 1


def partition_gpu_buffers(part, gpu, src_bytes, dst_sizes, src_gpu, dst_gpu):
    """Host buffer table [sources..., destinations..., receive, send] of one GPU: only the
    ranks on that GPU get buffers (others None)."""
    info = rs.reshard_partition_gpu(part, gpu)
    srcs = [src_bytes[r].copy() if src_gpu[r] == gpu else None for r in range(len(src_bytes))]
    dsts = [np.full(n, 0xA5, dtype=np.uint8) if dst_gpu[r] == gpu else None
            for r, n in enumerate(dst_sizes)]
    recv = np.zeros(info["recv_bytes"], dtype=np.uint8)
    send = np.zeros(info["send_bytes"], dtype=np.uint8)
    bufs = srcs + dsts + [recv, send]
    writes = [np.zeros(b.size, dtype=np.int32) if b is not None else None for b in bufs]
    return bufs, writes


def run_partition_step_cpu(part, gpu, step, chunk, bufs, writes):
    tiles, _, goff, gbuf = rs.reshard_partition_program(part, gpu, step, chunk)
    run_tile_list_cpu(tiles, goff, gbuf, bufs, writes)
