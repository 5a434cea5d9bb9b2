"""CPU oracle of the DTensor-to-DTensor reshard -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check of ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never calls it,
and it shares no code with the library: the arithmetic lives in ``oracle.c``
(plain C, compiled with gcc), this module only marshals arguments.

What the oracle computes is the plain definition of a reshard (see the header
of ``oracle.c``): every destination element is copied from the first source
shard, in flat rank order, whose box holds its global index.  Source:
"Accelerating Reinforcement Learning Weight Refit with the Reshard
Collective" (news.bpdata.com summary, sections on the DTensor reformulation
and on the Reshard collective; techfeed.io summary, the 8x8 example).

Placements are given as strings, ``"R"`` for Replicate and ``"S<d>"`` for
Shard(d); buffers are 1-D ``numpy.uint8`` arrays holding the row-major local
shard of each rank.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

_I64P = ctypes.POINTER(ctypes.c_int64)
_I32P = ctypes.POINTER(ctypes.c_int32)


def build(plant: int = 0, out: str | None = None) -> str:
    """Compile oracle.c into a shared library with gcc and return its path.

    ``plant`` selects one deliberately planted mistake (tests only, see
    oracle.c); 0 builds the real oracle.
    """
    out = out or LIB_PATH
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", SOURCE, "-o", out]
    if plant:
        cmd.insert(1, f"-DORACLE_PLANT={int(plant)}")
    subprocess.run(cmd, check=True)
    return out


def shard_dims(placements: Sequence[str]) -> list[int]:
    """Encode placement strings as one int per mesh dim (-1 = Replicate)."""
    out = []
    for p in placements:
        if p == "R":
            out.append(-1)
        elif isinstance(p, str) and p.startswith("S"):
            out.append(int(p[1:]))
        else:
            raise ValueError(f"unsupported placement {p!r}")
    return out


def _arr64(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def _arr32(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


class OracleError(RuntimeError):
    pass


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str = LIB_PATH):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_resolve.argtypes = [ctypes.c_int32, _I64P, ctypes.c_int32, _I64P, _I32P,
                                       ctypes.c_int64, _I64P, _I64P]
        lib.oracle_resolve.restype = ctypes.c_int
        lib.oracle_reshard.argtypes = [ctypes.c_int32, _I64P, ctypes.c_int64,
                                       ctypes.c_int32, _I64P, _I32P,
                                       ctypes.c_int32, _I64P, _I32P,
                                       ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.c_int64, ctypes.c_int64]
        lib.oracle_reshard.restype = ctypes.c_int
        lib.oracle_source_of.argtypes = [ctypes.c_int32, _I64P,
                                         ctypes.c_int32, _I64P, _I32P,
                                         ctypes.c_int32, _I64P, _I32P,
                                         ctypes.c_int64, ctypes.c_int64, _I64P, _I64P]
        lib.oracle_source_of.restype = ctypes.c_int
        lib.oracle_gather_full.argtypes = [ctypes.c_int32, _I64P, ctypes.c_int64,
                                           ctypes.c_int32, _I64P, _I32P,
                                           ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
        lib.oracle_gather_full.restype = ctypes.c_int
        lib.oracle_reshard_elems.argtypes = [ctypes.c_int32, _I64P, ctypes.c_int64,
                                             ctypes.c_int32, _I64P, _I32P,
                                             ctypes.c_int32, _I64P, _I32P,
                                             ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_reshard_elems.restype = ctypes.c_int
        self.lib = lib

    # -- layout --------------------------------------------------------------------------
    def resolve(self, gshape, mesh, placements, rank):
        """(offset, shape) of one flat rank's local shard, as tuples."""
        nd = len(gshape)
        off = (ctypes.c_int64 * nd)()
        shp = (ctypes.c_int64 * nd)()
        rc = self.lib.oracle_resolve(nd, _arr64(gshape), len(mesh), _arr64(mesh),
                                     _arr32(shard_dims(placements)), int(rank), off, shp)
        if rc:
            raise OracleError(f"oracle_resolve failed ({rc})")
        return tuple(off), tuple(shp)

    def boxes(self, gshape, mesh, placements):
        n = int(np.prod(mesh))
        return [self.resolve(gshape, mesh, placements, r) for r in range(n)]

    # -- data ----------------------------------------------------------------------------
    def reshard(self, gshape, elem_bytes, src_mesh, src_pl, dst_mesh, dst_pl,
                src_bufs: Sequence[np.ndarray], dst_ranks: Sequence[int] | None = None):
        """Expected destination buffers (uint8 arrays) for the given dst ranks."""
        nd = len(gshape)
        ndst = int(np.prod(dst_mesh))
        ranks = list(range(ndst)) if dst_ranks is None else [int(r) for r in dst_ranks]
        srcs = [np.ascontiguousarray(b, dtype=np.uint8) for b in src_bufs]
        src_ptrs = (ctypes.c_void_p * max(1, len(srcs)))(
            *[b.ctypes.data if b.size else None for b in srcs])
        outs = []
        for r in ranks:
            _, shp = self.resolve(gshape, dst_mesh, dst_pl, r)
            out = np.zeros(int(np.prod(shp)) * elem_bytes, dtype=np.uint8)
            dst_ptrs = (ctypes.c_void_p * 1)(out.ctypes.data if out.size else None)
            rc = self.lib.oracle_reshard(nd, _arr64(gshape), int(elem_bytes),
                                         len(src_mesh), _arr64(src_mesh),
                                         _arr32(shard_dims(src_pl)),
                                         len(dst_mesh), _arr64(dst_mesh),
                                         _arr32(shard_dims(dst_pl)),
                                         src_ptrs, dst_ptrs, r, r + 1)
            if rc:
                raise OracleError(f"oracle_reshard failed ({rc}) for dst rank {r}")
            outs.append(out)
        return outs

    def reshard_elems(self, gshape, elem_bytes, src_mesh, src_pl, dst_mesh, dst_pl, src_ptrs,
                      dst_ptr, dst_rank, e_begin, e_end):
        """Elements [e_begin, e_end) of one destination rank, on raw host pointers.

        ``src_ptrs`` are host addresses of the source shards (ints or None),
        ``dst_ptr`` the host address of the rank's whole local shard.
        """
        sp = (ctypes.c_void_p * max(1, len(src_ptrs)))(*src_ptrs)
        rc = self.lib.oracle_reshard_elems(len(gshape), _arr64(gshape), int(elem_bytes),
                                           len(src_mesh), _arr64(src_mesh),
                                           _arr32(shard_dims(src_pl)),
                                           len(dst_mesh), _arr64(dst_mesh),
                                           _arr32(shard_dims(dst_pl)),
                                           sp, dst_ptr, int(dst_rank), int(e_begin), int(e_end))
        if rc:
            raise OracleError(f"oracle_reshard_elems failed ({rc})")

    def source_of(self, gshape, src_mesh, src_pl, dst_mesh, dst_pl, dst_rank, dst_linear):
        """(src rank, src linear element index) that supplies one dst element."""
        s = ctypes.c_int64()
        j = ctypes.c_int64()
        rc = self.lib.oracle_source_of(len(gshape), _arr64(gshape),
                                       len(src_mesh), _arr64(src_mesh),
                                       _arr32(shard_dims(src_pl)),
                                       len(dst_mesh), _arr64(dst_mesh),
                                       _arr32(shard_dims(dst_pl)),
                                       int(dst_rank), int(dst_linear),
                                       ctypes.byref(s), ctypes.byref(j))
        if rc:
            raise OracleError(f"oracle_source_of failed ({rc})")
        return s.value, j.value

    def gather_full(self, gshape, elem_bytes, src_mesh, src_pl, src_bufs):
        """The full global tensor (uint8) assembled from the source shards."""
        srcs = [np.ascontiguousarray(b, dtype=np.uint8) for b in src_bufs]
        src_ptrs = (ctypes.c_void_p * max(1, len(srcs)))(
            *[b.ctypes.data if b.size else None for b in srcs])
        out = np.zeros(int(np.prod(gshape)) * elem_bytes, dtype=np.uint8)
        rc = self.lib.oracle_gather_full(len(gshape), _arr64(gshape), int(elem_bytes),
                                         len(src_mesh), _arr64(src_mesh),
                                         _arr32(shard_dims(src_pl)), src_ptrs,
                                         out.ctypes.data if out.size else None)
        if rc:
            raise OracleError(f"oracle_gather_full failed ({rc})")
        return out


_CACHE: dict[str, Oracle] = {}


def load(path: str | None = None) -> Oracle:
    """The real oracle, compiled on first use if the library is missing or stale."""
    path = path or LIB_PATH
    if path == LIB_PATH and (not os.path.exists(path)
                             or os.path.getmtime(path) < os.path.getmtime(SOURCE)):
        build()
    if path not in _CACHE:
        _CACHE[path] = Oracle(path)
    return _CACHE[path]
