"""Shard layouts built from torch.chunk alone -- an independent check of the oracle.

DTensor's Shard(d) places the pieces of ``torch.chunk`` on the ranks of a mesh
dim, and trailing ranks that ``torch.chunk`` gives no piece receive an empty
shard.  Applying ``torch.chunk`` mesh dim by mesh dim (dim 0 outermost) to a
tensor of global indices therefore yields every rank's shard without any of the
oracle's index arithmetic.  These helpers are test code; they never touch the
oracle or the library.
"""
from __future__ import annotations

import itertools
import math

import torch


def coords(mesh, rank):
    out = []
    for m in reversed(mesh):
        out.append(rank % m)
        rank //= m
    return tuple(reversed(out))


def index_lists(gshape, mesh, placements, rank):
    """Per tensor dim, the global indices that ``rank`` holds (a 1-D tensor)."""
    idx = [torch.arange(n) for n in gshape]
    c = coords(mesh, rank)
    for md, p in enumerate(placements):
        if p == "R":
            continue
        d = int(p[1:])
        pieces = torch.chunk(idx[d], mesh[md]) if idx[d].numel() else ()
        idx[d] = pieces[c[md]] if c[md] < len(pieces) else idx[d][idx[d].numel():]
    return idx


def box(gshape, mesh, placements, rank):
    """(offset, shape) as DTensor reports them (empty dim -> offset = global extent)."""
    idx = index_lists(gshape, mesh, placements, rank)
    sharded = {int(p[1:]) for p in placements if p != "R"}
    off, shp = [], []
    for d, ix in enumerate(idx):
        n = ix.numel()
        if n:
            assert torch.equal(ix, torch.arange(int(ix[0]), int(ix[0]) + n)), "non-contiguous"
            off.append(int(ix[0]))
        else:
            off.append(gshape[d] if d in sharded else 0)
        shp.append(n)
    return tuple(off), tuple(shp)


def local_shard(global_t, mesh, placements, rank):
    """The rank's local shard of a global tensor, contiguous (torch.chunk slicing)."""
    idx = index_lists(tuple(global_t.shape), mesh, placements, rank)
    t = global_t
    for d, ix in enumerate(idx):
        t = t.index_select(d, ix)
    return t.contiguous()


def all_meshes(max_ranks=4, max_ndim=3):
    out = []
    for nd in range(1, max_ndim + 1):
        for mesh in itertools.product(range(1, max_ranks + 1), repeat=nd):
            if math.prod(mesh) <= max_ranks:
                out.append(mesh)
    return out


def all_placements(mesh_ndim, tensor_ndim):
    opts = ["R"] + [f"S{d}" for d in range(tensor_ndim)]
    return list(itertools.product(opts, repeat=mesh_ndim))
