"""Python binding of libreshard.so: a GB300 (sm_103a) DTensor-to-DTensor reshard.

The functions below carry the names of the C entry points declared in
``include/reshard.h`` and only marshal arguments: every step of the reshard
(layout resolution, intersection, planning, copying) runs inside the library.
Device pointers may be passed as integers or as any object with a
``data_ptr()`` method (e.g. a CUDA ``torch.Tensor``); streams as integers, as
objects with a ``cuda_stream`` attribute, or None (legacy default stream).

Placements are strings, ``"R"`` for Replicate and ``"S<d>"`` for Shard(d), or
(kind, dim) tuples.  There is no CPU fallback: importing this package raises if
the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libreshard.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "reshard.h")


def header_defines(path: str = HEADER_PATH) -> dict:
    """Integer macros ``RESHARD_*`` of the library's header, by name.

    Values are plain integers or ``(a << b)`` shifts, with C integer suffixes.
    """
    out = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"\s*#define\s+(RESHARD_\w+)\s+\(?\s*(\d+)[uUlL]*"
                         r"(?:\s*<<\s*(\d+))?\s*\)?", line)
            if m:
                v = int(m.group(2))
                out[m.group(1)] = v << int(m.group(3)) if m.group(3) else v
    return out


_DEFINES = header_defines()
MAX_TENSOR_NDIM = _DEFINES["RESHARD_MAX_TENSOR_NDIM"]
MAX_MESH_NDIM = _DEFINES["RESHARD_MAX_MESH_NDIM"]
MAX_EXEC_BUFFERS = _DEFINES["RESHARD_MAX_EXEC_BUFFERS"]

DTYPES = {"u8": 0, "bf16": 1, "fp16": 2, "fp32": 3, "i32": 4, "fp64": 5, "i64": 6}
ELEM_BYTES = {"u8": 1, "bf16": 2, "fp16": 2, "fp32": 4, "i32": 4, "fp64": 8, "i64": 8}

OK = 0
STATUS = {0: "RESHARD_OK", 1: "RESHARD_ERR_INVALID_ARG", 2: "RESHARD_ERR_UNSUPPORTED",
          3: "RESHARD_ERR_SHAPE", 4: "RESHARD_ERR_CUDA", 5: "RESHARD_ERR_NO_MEMORY",
          6: "RESHARD_ERR_BAD_HANDLE"}

KERNEL_FANOUT = 0
KERNEL_BOXCOPY = 1
PROGRAM_FANOUT, PROGRAM_BOXCOPY, PROGRAM_GATHER, PROGRAM_SLICE, PROGRAM_REPLICATE = 0, 1, 2, 3, 4


class reshard_placement_t(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("dim", ctypes.c_int32)]


class reshard_mesh_t(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * MAX_MESH_NDIM)]


class reshard_stats_t(ctypes.Structure):
    _fields_ = [("global_bytes", ctypes.c_int64), ("src_bytes", ctypes.c_int64),
                ("dst_bytes", ctypes.c_int64), ("n_src_ranks", ctypes.c_int64),
                ("n_dst_ranks", ctypes.c_int64), ("n_src_classes", ctypes.c_int64),
                ("n_dst_classes", ctypes.c_int64), ("n_regions", ctypes.c_int64),
                ("region_bytes", ctypes.c_int64), ("n_tiles", ctypes.c_int64 * 4),
                ("fanout_read_bytes", ctypes.c_int64), ("fanout_write_bytes", ctypes.c_int64),
                ("boxcopy_read_bytes", ctypes.c_int64), ("boxcopy_write_bytes", ctypes.c_int64),
                ("gb_read_bytes", ctypes.c_int64), ("gb_write_bytes", ctypes.c_int64),
                ("max_replica_read_bytes", ctypes.c_int64), ("max_fanout", ctypes.c_int64),
                ("planner_ns", ctypes.c_int64), ("inplace_bytes", ctypes.c_int64),
                ("assembled_classes", ctypes.c_int64), ("n_replicate_tiles", ctypes.c_int64)]

    def as_dict(self) -> dict:
        out = {}
        for name, _ in self._fields_:
            v = getattr(self, name)
            out[name] = list(v) if name == "n_tiles" else int(v)
        return out


class reshard_tile_t(ctypes.Structure):
    _fields_ = [("src_off", ctypes.c_int64), ("dst_off", ctypes.c_int64),
                ("src_row_stride", ctypes.c_int64), ("dst_row_stride", ctypes.c_int64),
                ("src_plane_stride", ctypes.c_int64), ("dst_plane_stride", ctypes.c_int64),
                ("row_bytes", ctypes.c_uint32), ("nrows", ctypes.c_uint32),
                ("nplanes", ctypes.c_uint32), ("src_buf", ctypes.c_uint16),
                ("dst_group", ctypes.c_uint16)]


assert ctypes.sizeof(reshard_tile_t) == 64


class reshard_tblock_t(ctypes.Structure):
    _fields_ = [("wide_off", ctypes.c_int64), ("row_bytes", ctypes.c_uint32),
                ("nrows", ctypes.c_uint32), ("seg_begin", ctypes.c_uint32),
                ("seg_count", ctypes.c_uint32), ("wide", ctypes.c_uint16),
                ("direction", ctypes.c_uint16), ("flags", ctypes.c_uint32)]


class reshard_tseg_t(ctypes.Structure):
    _fields_ = [("narrow_off", ctypes.c_int64), ("width", ctypes.c_uint32),
                ("col", ctypes.c_uint32), ("narrow", ctypes.c_uint16), ("pad16", ctypes.c_uint16),
                ("pad32", ctypes.c_uint32)]


assert ctypes.sizeof(reshard_tblock_t) == 32 and ctypes.sizeof(reshard_tseg_t) == 24


class reshard_xfer_t(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int32), ("stage", ctypes.c_int32), ("peer", ctypes.c_int32),
                ("dir", ctypes.c_int32), ("offset", ctypes.c_int64), ("bytes", ctypes.c_int64)]


class reshard_partition_gpu_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "send_bytes", "recv_bytes", "local_bytes", "sent_inter_bytes", "sent_intra_bytes",
        "recv_inter_bytes", "recv_intra_bytes", "n_xfers")]


class reshard_partition_stats_t(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int32) for n in ("ngpus", "ndomains", "nchunks", "nslots")] +
                [(n, ctypes.c_int64) for n in (
                    "local_bytes", "inter_domain_bytes", "intra_domain_bytes",
                    "max_gpu_send_bytes", "max_gpu_recv_bytes", "n_pieces", "n_messages",
                    "planner_ns")])


assert ctypes.sizeof(reshard_xfer_t) == 32


class ReshardError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    i64p = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "reshard_plan_create": ([i64p, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.POINTER(reshard_mesh_t),
                                 ctypes.POINTER(reshard_placement_t),
                                 ctypes.POINTER(reshard_mesh_t),
                                 ctypes.POINTER(reshard_placement_t), vpp], ctypes.c_int),
        "reshard_plan_create_inplace": ([i64p, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.POINTER(reshard_mesh_t),
                                         ctypes.POINTER(reshard_placement_t),
                                         ctypes.POINTER(reshard_mesh_t),
                                         ctypes.POINTER(reshard_placement_t), i64p, vpp],
                                        ctypes.c_int),
        "reshard_plan_alias": ([vp, ctypes.c_int64, i64p, i64p], ctypes.c_int),
        "reshard_batch_create": ([ctypes.POINTER(vp), ctypes.c_int32, vpp], ctypes.c_int),
        "reshard_batch_execute": ([vp, ctypes.POINTER(vpp), ctypes.POINTER(vpp), vp],
                                  ctypes.c_int),
        "reshard_batch_destroy": ([vp], ctypes.c_int),
        "reshard_batch_classes": ([vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
                                  ctypes.c_int),
        "reshard_refit_create": ([ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                  ctypes.c_uint32, vpp], ctypes.c_int),
        "reshard_refit_info": ([vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_uint64)],
                               ctypes.c_int),
        "reshard_refit_execute": ([vp, ctypes.POINTER(vpp), ctypes.POINTER(vpp), vp, ctypes.c_size_t,
                                   vp], ctypes.c_int),
        "reshard_refit_destroy": ([vp], ctypes.c_int),
        "reshard_plan_upload": ([vp], ctypes.c_int),
        "reshard_execute": ([vp, vpp, vpp, vp], ctypes.c_int),
        "reshard_execute_ex": ([vp, vpp, vpp, ctypes.c_int32, vp], ctypes.c_int),
        "reshard_plan_exclude": ([vp, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                  ctypes.POINTER(ctypes.c_int64), ctypes.c_int32, vpp], ctypes.c_int),
        "reshard_plan_path": ([vp, vpp, vpp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                               ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
        "gather_broadcast_execute": ([vp, vpp, vpp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "gather_broadcast_execute_static": ([vp, vpp, vpp, vp], ctypes.c_int),
        "reshard_device_status": ([ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
        "reshard_selftest_wait_timeout": ([ctypes.c_uint32, vp], ctypes.c_int),
        "reshard_plan_local_shape": ([vp, ctypes.c_int32, ctypes.c_int64, i64p, i64p],
                                     ctypes.c_int),
        "reshard_plan_stats": ([vp, ctypes.POINTER(reshard_stats_t)], ctypes.c_int),
        "reshard_plan_program": ([vp, ctypes.c_int32,
                                  ctypes.POINTER(ctypes.POINTER(reshard_tile_t)), i64p,
                                  ctypes.POINTER(i64p),
                                  ctypes.POINTER(ctypes.POINTER(ctypes.c_uint32)),
                                  ctypes.POINTER(ctypes.POINTER(ctypes.c_uint16)), i64p],
                                 ctypes.c_int),
        "reshard_tile_units": ([ctypes.POINTER(reshard_tile_t)], ctypes.c_int64),
        "reshard_plan_transposes": ([vp, ctypes.c_int32,
                                     ctypes.POINTER(ctypes.POINTER(reshard_tblock_t)), i64p,
                                     ctypes.POINTER(ctypes.POINTER(reshard_tseg_t)), i64p],
                                    ctypes.c_int),
        "reshard_plan_destroy": ([vp], ctypes.c_int),
        "reshard_partition_create": ([vp, ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                      ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, vpp],
                                     ctypes.c_int),
        "reshard_partition_stats": ([vp, ctypes.POINTER(reshard_partition_stats_t)], ctypes.c_int),
        "reshard_partition_gpu": ([vp, ctypes.c_int32, ctypes.POINTER(reshard_partition_gpu_t)],
                                  ctypes.c_int),
        "reshard_partition_transfers": ([vp, ctypes.c_int32,
                                         ctypes.POINTER(ctypes.POINTER(reshard_xfer_t)), i64p],
                                        ctypes.c_int),
        "reshard_partition_program": ([vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(ctypes.POINTER(reshard_tile_t)), i64p,
                                       ctypes.POINTER(i64p),
                                       ctypes.POINTER(ctypes.POINTER(ctypes.c_uint32)),
                                       ctypes.POINTER(ctypes.POINTER(ctypes.c_uint16)), i64p],
                                      ctypes.c_int),
        "reshard_partition_execute": ([vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vpp,
                                       vpp, vp, vp, vp], ctypes.c_int),
        "reshard_partition_destroy": ([vp], ctypes.c_int),
        "reshard_last_error": ([], ctypes.c_char_p),
        "reshard_version": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library_path() -> str:
    return LIB_PATH


def reshard_last_error() -> str:
    return _lib.reshard_last_error().decode()


def reshard_version() -> str:
    return _lib.reshard_version().decode()


def _check(status: int, where: str):
    if status != OK:
        raise ReshardError(status, where, reshard_last_error())


# ------------------------------------------------------------------------ marshalling
def placement(p) -> tuple:
    """(kind, dim) of a placement given as "R", "S<d>" or a (kind, dim) tuple."""
    if isinstance(p, str):
        if p == "R":
            return (0, 0)
        if p.startswith("S"):
            return (1, int(p[1:]))
        raise ValueError(f"unknown placement {p!r}")
    kind, dim = p
    return (int(kind), int(dim))


def _mesh(mesh: Sequence[int]) -> reshard_mesh_t:
    m = reshard_mesh_t()
    m.ndim = len(mesh)
    for i, s in enumerate(list(mesh)[:MAX_MESH_NDIM]):
        m.shape[i] = int(s)
    return m


def _placements(pls) -> ctypes.Array:
    arr = (reshard_placement_t * max(1, len(pls)))()
    for i, p in enumerate(pls):
        arr[i].kind, arr[i].dim = placement(p)
    return arr


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr()) or None
    return int(x) or None


def _ptr_array(xs) -> ctypes.Array:
    return (ctypes.c_void_p * max(1, len(xs)))(*[_ptr(x) for x in xs])


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream) or None
    return int(s) or None


class Plan:
    """Owning wrapper of a reshard_plan_t handle."""

    def __init__(self, handle: int, global_shape, dtype, src_mesh, src_placements, dst_mesh,
                 dst_placements):
        self.handle = handle
        self.global_shape = tuple(int(s) for s in global_shape)
        self.dtype = dtype
        self.src_mesh, self.src_placements = tuple(src_mesh), tuple(src_placements)
        self.dst_mesh, self.dst_placements = tuple(dst_mesh), tuple(dst_placements)
        self.n_src = math.prod(self.src_mesh)
        self.n_dst = math.prod(self.dst_mesh)

    @property
    def _as_parameter_(self):
        if not self.handle:
            raise ReshardError(6, "plan", "plan already destroyed")
        return ctypes.c_void_p(self.handle)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                _lib.reshard_plan_destroy(ctypes.c_void_p(h))
            except Exception:  # noqa: BLE001 - interpreter shutdown
                pass
            self.handle = None


# ------------------------------------------------------------------------ entry points
def reshard_plan_create(global_shape, dtype, src_mesh, src_placements, dst_mesh,
                        dst_placements) -> Plan:
    shape = (ctypes.c_int64 * max(1, len(global_shape)))(*[int(s) for s in global_shape])
    h = ctypes.c_void_p()
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    st = _lib.reshard_plan_create(shape, len(global_shape), dt, ctypes.byref(_mesh(src_mesh)),
                                  _placements(src_placements), ctypes.byref(_mesh(dst_mesh)),
                                  _placements(dst_placements), ctypes.byref(h))
    _check(st, "reshard_plan_create")
    return Plan(h.value, global_shape, dtype, src_mesh, src_placements, dst_mesh, dst_placements)


def reshard_plan_exclude(plan: Plan, src_gone=(), dst_gone=()) -> Plan:
    """A plan with plan's layouts in which exactly the listed source and destination ranks
    are gone (never read / never written; their pointers may be None)."""
    sa = (ctypes.c_int64 * max(1, len(src_gone)))(*[int(r) for r in src_gone])
    da = (ctypes.c_int64 * max(1, len(dst_gone)))(*[int(r) for r in dst_gone])
    h = ctypes.c_void_p()
    _check(_lib.reshard_plan_exclude(plan, sa, len(src_gone), da, len(dst_gone),
                                     ctypes.byref(h)), "reshard_plan_exclude")
    return Plan(h.value, plan.global_shape, plan.dtype, plan.src_mesh, plan.src_placements,
                plan.dst_mesh, plan.dst_placements)


def reshard_plan_create_inplace(global_shape, dtype, src_mesh, src_placements, dst_mesh,
                                dst_placements, src_alias) -> Plan:
    """In-place plan: src_alias[s] = destination rank whose buffer holds source shard s (-1:
    none).  Executions need src_ptrs[s] = dst_ptrs[src_alias[s]] + reshard_plan_alias offset."""
    shape = (ctypes.c_int64 * max(1, len(global_shape)))(*[int(s) for s in global_shape])
    alias = (ctypes.c_int64 * max(1, len(src_alias)))(*[int(a) for a in src_alias])
    h = ctypes.c_void_p()
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    st = _lib.reshard_plan_create_inplace(shape, len(global_shape), dt,
                                          ctypes.byref(_mesh(src_mesh)),
                                          _placements(src_placements),
                                          ctypes.byref(_mesh(dst_mesh)),
                                          _placements(dst_placements), alias, ctypes.byref(h))
    _check(st, "reshard_plan_create_inplace")
    return Plan(h.value, global_shape, dtype, src_mesh, src_placements, dst_mesh, dst_placements)


def reshard_plan_alias(plan: Plan, src_rank: int):
    """(destination rank or -1, byte offset) where source rank src_rank lives."""
    d = ctypes.c_int64()
    o = ctypes.c_int64()
    _check(_lib.reshard_plan_alias(plan, int(src_rank), ctypes.byref(d), ctypes.byref(o)),
           "reshard_plan_alias")
    return d.value, o.value


class Batch:
    """Owning wrapper of a reshard_batch_t (keeps its plans alive)."""

    def __init__(self, handle: int, plans):
        self.handle = handle
        self.plans = list(plans)

    @property
    def _as_parameter_(self):
        if not self.handle:
            raise ReshardError(6, "batch", "batch already destroyed")
        return ctypes.c_void_p(self.handle)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                _lib.reshard_batch_destroy(ctypes.c_void_p(h))
            except Exception:  # noqa: BLE001 - interpreter shutdown
                pass
            self.handle = None


def reshard_batch_create(plans) -> Batch:
    arr = (ctypes.c_void_p * len(plans))(*[p.handle for p in plans])
    h = ctypes.c_void_p()
    _check(_lib.reshard_batch_create(arr, len(plans), ctypes.byref(h)), "reshard_batch_create")
    return Batch(h.value, plans)


def reshard_batch_execute(batch: Batch, src_ptrs_per_plan, dst_ptrs_per_plan, stream=None):
    """src_ptrs_per_plan[i] / dst_ptrs_per_plan[i]: plan i's pointer lists."""
    srcs = [_ptr_array(x) for x in src_ptrs_per_plan]
    dsts = [_ptr_array(x) for x in dst_ptrs_per_plan]
    sa = (ctypes.POINTER(ctypes.c_void_p) * len(srcs))(
        *[ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)) for a in srcs])
    da = (ctypes.POINTER(ctypes.c_void_p) * len(dsts))(
        *[ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)) for a in dsts])
    _check(_lib.reshard_batch_execute(batch, sa, da, _stream(stream)), "reshard_batch_execute")


def reshard_batch_classes(batch: Batch):
    """(number of launch classes, class of each plan or -1 for a plan with nothing to copy)."""
    n = ctypes.c_int32()
    per = (ctypes.c_int32 * len(batch.plans))()
    _check(_lib.reshard_batch_classes(batch, ctypes.byref(n), per), "reshard_batch_classes")
    return int(n.value), [int(x) for x in per]


def reshard_batch_destroy(batch: Batch):
    if not batch.handle:
        raise ReshardError(6, "reshard_batch_destroy", "batch already destroyed")
    st = _lib.reshard_batch_destroy(batch)
    batch.handle = None
    _check(st, "reshard_batch_destroy")


ROUTE_AUTO, ROUTE_RESHARD, ROUTE_GATHER_BROADCAST = 0, 1, 2
REFIT_BATCH = _DEFINES["RESHARD_REFIT_BATCH"]
REFIT_LANES = _DEFINES["RESHARD_REFIT_LANES"]
REFIT_NUM_LANES = _DEFINES["RESHARD_REFIT_NUM_LANES"]


class Refit:
    """Owning wrapper of a reshard_refit_t (keeps its plans alive)."""

    def __init__(self, handle, plans):
        self.handle = handle
        self.plans = list(plans)

    @property
    def _as_parameter_(self):
        if not self.handle:
            raise ReshardError(6, "refit", "refit already destroyed")
        return ctypes.c_void_p(self.handle)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                _lib.reshard_refit_destroy(ctypes.c_void_p(h))
            except Exception:  # noqa: BLE001 - interpreter shutdown
                pass
            self.handle = None


def _nested(ptr_lists):
    arrs = [_ptr_array(x) for x in ptr_lists]
    out = (ctypes.POINTER(ctypes.c_void_p) * len(arrs))(
        *[ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)) for a in arrs])
    return out, arrs


def reshard_refit_create(plans, routes=None, batch: bool = False, lanes: bool = False) -> Refit:
    """One refit over plans; routes[i] in ROUTE_* (None: AUTO for every plan).
    batch: the reshard group in as few launches as a batch makes; lanes: the reshard
    group spread over REFIT_NUM_LANES side streams (with batch as well, the plans a
    batch merges into one launch run as one unit on one lane)."""
    arr = (ctypes.c_void_p * len(plans))(*[p.handle for p in plans])
    ra = None if routes is None else (ctypes.c_int32 * len(plans))(*[int(r) for r in routes])
    h = ctypes.c_void_p()
    flags = (REFIT_BATCH if batch else 0) | (REFIT_LANES if lanes else 0)
    _check(_lib.reshard_refit_create(arr, ra, len(plans), flags, ctypes.byref(h)),
           "reshard_refit_create")
    return Refit(h.value, plans)


def reshard_refit_info(refit: Refit):
    """(resolved routes, scratch bytes needed)."""
    routes = (ctypes.c_int32 * len(refit.plans))()
    sb = ctypes.c_uint64()
    _check(_lib.reshard_refit_info(refit, routes, ctypes.byref(sb)), "reshard_refit_info")
    return [int(r) for r in routes], int(sb.value)


def reshard_refit_execute(refit: Refit, src_ptrs_per_plan, dst_ptrs_per_plan, scratch=None,
                          scratch_bytes: int = 0, stream=None):
    sa, keep_s = _nested(src_ptrs_per_plan)
    da, keep_d = _nested(dst_ptrs_per_plan)
    if scratch is not None and not scratch_bytes and hasattr(scratch, "numel"):
        scratch_bytes = scratch.numel() * scratch.element_size()
    _check(_lib.reshard_refit_execute(refit, sa, da, _ptr(scratch), int(scratch_bytes),
                                      _stream(stream)), "reshard_refit_execute")


def reshard_refit_destroy(refit: Refit):
    if not refit.handle:
        raise ReshardError(6, "reshard_refit_destroy", "refit already destroyed")
    st = _lib.reshard_refit_destroy(refit)
    refit.handle = None
    _check(st, "reshard_refit_destroy")


def reshard_plan_upload(plan: Plan):
    _check(_lib.reshard_plan_upload(plan), "reshard_plan_upload")


def reshard_execute(plan: Plan, src_ptrs, dst_ptrs, stream=None):
    _check(_lib.reshard_execute(plan, _ptr_array(src_ptrs), _ptr_array(dst_ptrs),
                                _stream(stream)), "reshard_execute")


def reshard_execute_ex(plan: Plan, src_ptrs, dst_ptrs, kernel: int, stream=None):
    _check(_lib.reshard_execute_ex(plan, _ptr_array(src_ptrs), _ptr_array(dst_ptrs),
                                   int(kernel), _stream(stream)), "reshard_execute_ex")


PATHS = {0: "none", 1: "vector", 2: "tma_fanout", 3: "realign", 4: "staged", 5: "staged_bulk"}


def reshard_plan_path(plan: Plan, src_ptrs, dst_ptrs, kernel: int = 0):
    """(path name, access width in bytes) that reshard_execute_ex would take with these
    buffers; decided on the host, nothing is launched."""
    path, width = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.reshard_plan_path(plan, _ptr_array(src_ptrs), _ptr_array(dst_ptrs), int(kernel),
                                  ctypes.byref(path), ctypes.byref(width)), "reshard_plan_path")
    return PATHS[int(path.value)], int(width.value)


def gather_broadcast_execute(plan: Plan, src_ptrs, dst_ptrs, full_scratch, scratch_bytes: int,
                             stream=None):
    _check(_lib.gather_broadcast_execute(plan, _ptr_array(src_ptrs), _ptr_array(dst_ptrs),
                                         _ptr(full_scratch), int(scratch_bytes), _stream(stream)),
           "gather_broadcast_execute")


def gather_broadcast_execute_static(plan: Plan, src_ptrs, dst_ptrs, stream=None):
    """gather_broadcast_execute with the library's static device scratch (no allocation;
    see include/reshard.h for the size limits and the sharing rules)."""
    _check(_lib.gather_broadcast_execute_static(plan, _ptr_array(src_ptrs), _ptr_array(dst_ptrs),
                                                _stream(stream)),
           "gather_broadcast_execute_static")


def reshard_device_status(clear: bool = False) -> int:
    """Status word of the current device's copy kernels (0 = no wait ever ran out)."""
    v = ctypes.c_uint32()
    _check(_lib.reshard_device_status(1 if clear else 0, ctypes.byref(v)), "reshard_device_status")
    return int(v.value)


def reshard_selftest_wait_timeout(polls: int = 4096, stream=None):
    _check(_lib.reshard_selftest_wait_timeout(int(polls), _stream(stream)),
           "reshard_selftest_wait_timeout")


# sizes of the static device arrays behind gather_broadcast_execute_static
STATIC_SCRATCH_BYTES = _DEFINES["RESHARD_STATIC_SCRATCH_BYTES"]
STATIC_TABLE_BYTES = _DEFINES["RESHARD_STATIC_TABLE_BYTES"]


def reshard_plan_local_shape(plan: Plan, side: int, rank: int):
    """(shape, offset) tuples of one rank's local shard (side 0 = source, 1 = destination)."""
    nd = len(plan.global_shape)
    shp = (ctypes.c_int64 * nd)()
    off = (ctypes.c_int64 * nd)()
    _check(_lib.reshard_plan_local_shape(plan, int(side), int(rank), shp, off),
           "reshard_plan_local_shape")
    return tuple(shp), tuple(off)


def reshard_plan_stats(plan: Plan) -> dict:
    s = reshard_stats_t()
    _check(_lib.reshard_plan_stats(plan, ctypes.byref(s)), "reshard_plan_stats")
    return s.as_dict()


def reshard_plan_program(plan: Plan, program: int):
    """(tiles, unit_prefix, group_offsets, group_buffers) of one program, copied to Python."""
    tp = ctypes.POINTER(reshard_tile_t)()
    nt = ctypes.c_int64()
    pp = ctypes.POINTER(ctypes.c_int64)()
    go = ctypes.POINTER(ctypes.c_uint32)()
    gb = ctypes.POINTER(ctypes.c_uint16)()
    ng = ctypes.c_int64()
    _check(_lib.reshard_plan_program(plan, int(program), ctypes.byref(tp), ctypes.byref(nt),
                                     ctypes.byref(pp), ctypes.byref(go), ctypes.byref(gb),
                                     ctypes.byref(ng)), "reshard_plan_program")
    n, g = nt.value, ng.value
    tiles = [{f: getattr(tp[i], f) for f, _ in reshard_tile_t._fields_} for i in range(n)]
    prefix = [pp[i] for i in range(n + 1)]
    goff = [go[i] for i in range(g + 1)]
    gbuf = [gb[i] for i in range(goff[-1])] if g >= 0 and goff else []
    return tiles, prefix, goff, gbuf


def reshard_plan_transposes(plan: Plan, program: int):
    """(blocks, segments) of a program's transpose blocks, copied to Python dicts."""
    bp = ctypes.POINTER(reshard_tblock_t)()
    nb = ctypes.c_int64()
    sp = ctypes.POINTER(reshard_tseg_t)()
    ns = ctypes.c_int64()
    _check(_lib.reshard_plan_transposes(plan, int(program), ctypes.byref(bp), ctypes.byref(nb),
                                        ctypes.byref(sp), ctypes.byref(ns)),
           "reshard_plan_transposes")
    blocks = [{f: getattr(bp[i], f) for f, _ in reshard_tblock_t._fields_} for i in range(nb.value)]
    segs = [{f: getattr(sp[i], f) for f, _ in reshard_tseg_t._fields_} for i in range(ns.value)]
    return blocks, segs


def reshard_tile_units(tile: dict) -> int:
    t = reshard_tile_t(**tile)
    return int(_lib.reshard_tile_units(ctypes.byref(t)))


def reshard_plan_destroy(plan: Plan):
    if not plan.handle:
        raise ReshardError(6, "reshard_plan_destroy", "plan already destroyed")
    st = _lib.reshard_plan_destroy(plan)
    plan.handle = None
    _check(st, "reshard_plan_destroy")


# ------------------------------------------------------------------ multi-GPU partition
STEP_LOCAL, STEP_PACK, STEP_FORWARD, STEP_UNPACK = 0, 1, 2, 3


class Partition:
    """Handle of one plan cut by destination ownership over several GPUs."""

    def __init__(self, handle: int, plan: Plan, ngpus: int):
        self.handle = handle
        self.plan = plan   # the partition's programs index the plan's ranks
        self.ngpus = ngpus

    @property
    def _as_parameter_(self):
        if not self.handle:
            raise ReshardError(6, "partition", "partition already destroyed")
        return ctypes.c_void_p(self.handle)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            try:
                _lib.reshard_partition_destroy(ctypes.c_void_p(h))
            except Exception:  # noqa: BLE001 - interpreter shutdown
                pass
            self.handle = None


def reshard_partition_create(plan: Plan, src_gpu, dst_gpu, gpu_domain, nchunks: int = 1):
    """Cut ``plan`` over ``len(gpu_domain)`` GPUs: src_gpu[r] / dst_gpu[r] is the GPU of
    each source / destination rank, gpu_domain[g] the NVLink domain of GPU g."""
    def arr(v):
        v = [int(x) for x in v]
        return (ctypes.c_int32 * max(1, len(v)))(*v)
    h = ctypes.c_void_p()
    _check(_lib.reshard_partition_create(plan, arr(src_gpu), arr(dst_gpu), len(gpu_domain),
                                         arr(gpu_domain), int(nchunks), ctypes.byref(h)),
           "reshard_partition_create")
    return Partition(h.value, plan, len(gpu_domain))


def reshard_partition_stats(part: Partition) -> dict:
    s = reshard_partition_stats_t()
    _check(_lib.reshard_partition_stats(part, ctypes.byref(s)), "reshard_partition_stats")
    return {n: int(getattr(s, n)) for n, _ in s._fields_}


def reshard_partition_gpu(part: Partition, gpu: int) -> dict:
    s = reshard_partition_gpu_t()
    _check(_lib.reshard_partition_gpu(part, int(gpu), ctypes.byref(s)), "reshard_partition_gpu")
    return {n: int(getattr(s, n)) for n, _ in s._fields_}


def reshard_partition_transfers(part: Partition, gpu: int) -> list:
    """One GPU's messages as dicts (chunk, stage, peer, dir, offset, bytes)."""
    xp = ctypes.POINTER(reshard_xfer_t)()
    n = ctypes.c_int64()
    _check(_lib.reshard_partition_transfers(part, int(gpu), ctypes.byref(xp), ctypes.byref(n)),
           "reshard_partition_transfers")
    return [{f: int(getattr(xp[i], f)) for f, _ in reshard_xfer_t._fields_}
            for i in range(n.value)]


def reshard_partition_program(part: Partition, gpu: int, step: int, chunk: int = 0):
    """(tiles, unit_prefix, group_offsets, group_buffers) of one step of one GPU."""
    tp = ctypes.POINTER(reshard_tile_t)()
    nt = ctypes.c_int64()
    pp = ctypes.POINTER(ctypes.c_int64)()
    go = ctypes.POINTER(ctypes.c_uint32)()
    gb = ctypes.POINTER(ctypes.c_uint16)()
    ng = ctypes.c_int64()
    _check(_lib.reshard_partition_program(part, int(gpu), int(step), int(chunk),
                                          ctypes.byref(tp), ctypes.byref(nt), ctypes.byref(pp),
                                          ctypes.byref(go), ctypes.byref(gb), ctypes.byref(ng)),
           "reshard_partition_program")
    n, g = nt.value, ng.value
    tiles = [{f: getattr(tp[i], f) for f, _ in reshard_tile_t._fields_} for i in range(n)]
    prefix = [pp[i] for i in range(n + 1)]
    goff = [go[i] for i in range(g + 1)]
    gbuf = [gb[i] for i in range(goff[-1])] if g >= 0 and goff else []
    return tiles, prefix, goff, gbuf


def reshard_partition_execute(part: Partition, gpu: int, step: int, chunk: int, src_ptrs,
                              dst_ptrs, recv_buf, send_buf, stream=None):
    _check(_lib.reshard_partition_execute(part, int(gpu), int(step), int(chunk),
                                          _ptr_array(src_ptrs), _ptr_array(dst_ptrs),
                                          _ptr(recv_buf), _ptr(send_buf), _stream(stream)),
           "reshard_partition_execute")


def reshard_partition_destroy(part: Partition):
    if not part.handle:
        raise ReshardError(6, "reshard_partition_destroy", "partition already destroyed")
    st = _lib.reshard_partition_destroy(part)
    part.handle = None
    _check(st, "reshard_partition_destroy")


def partition_schedule(nchunks: int):
    """The order in which one GPU runs a partition: a list of ("step", STEP_*, chunk) and
    ("exchange", [(chunk, stage), ...]) items.  Stage 1 of a chunk is exchanged together
    with stage 0 of the next one (the pipeline of the two stages); every GPU follows the
    same list, so grouped point-to-point calls match."""
    out = [("step", STEP_LOCAL, 0), ("step", STEP_PACK, 0), ("exchange", [(0, 0)]),
           ("step", STEP_FORWARD, 0)]
    for c in range(1, nchunks):
        out += [("step", STEP_PACK, c), ("exchange", [(c - 1, 1), (c, 0)]),
                ("step", STEP_UNPACK, c - 1), ("step", STEP_FORWARD, c)]
    out += [("exchange", [(nchunks - 1, 1)]), ("step", STEP_UNPACK, nchunks - 1)]
    return out


def partition_run(part: Partition, gpu: int, src_ptrs, dst_ptrs, recv_buf, send_buf, exchange,
                  stream=None, run_step=None):
    """Run GPU ``gpu``'s share of a partitioned reshard in ``partition_schedule`` order.

    ``exchange(gpu, sends, recvs)`` performs one round of messages: ``sends`` and
    ``recvs`` are this GPU's transfer dicts of that round (offsets into send_buf /
    recv_buf), each list in (chunk, stage, peer) order; it must order them after the
    steps already enqueued on ``stream`` and the next steps after them (NCCL on the
    same stream does; a host-side exchange synchronises the stream first).  Each step
    is ``reshard_partition_execute`` on ``stream`` (the library's kernels do every copy
    on the GPU), or ``run_step(step, chunk)`` when given.
    """
    if run_step is None:
        def run_step(step, chunk):
            reshard_partition_execute(part, gpu, step, chunk, src_ptrs, dst_ptrs, recv_buf,
                                      send_buf, stream)
    xfers = reshard_partition_transfers(part, gpu)
    for item in partition_schedule(reshard_partition_stats(part)["nchunks"]):
        if item[0] == "step":
            run_step(item[1], item[2])
        else:
            rounds = set(item[1])
            sends = [x for x in xfers if (x["chunk"], x["stage"]) in rounds and x["dir"] == 0]
            recvs = [x for x in xfers if (x["chunk"], x["stage"]) in rounds and x["dir"] == 1]
            exchange(gpu, sends, recvs)


def nccl_exchange(gpu_rank, send_buf, recv_buf):
    """An ``exchange`` for partition_run over torch.distributed point-to-point (NCCL on
    the current stream): process ``gpu_rank[g]`` runs GPU g; send_buf / recv_buf are
    uint8 device tensors.  The messages of one round go out as one batch; two messages
    between one pair of GPUs in a round are matched in list order on both sides.  NCCL
    wants the process group to have run a collective before its first batch of
    point-to-point calls (a barrier will do).  Not run on more than one GPU here."""
    import torch.distributed as dist

    def exchange(gpu, sends, recvs):
        ops = [dist.P2POp(dist.isend, send_buf[x["offset"]:x["offset"] + x["bytes"]],
                          gpu_rank[x["peer"]]) for x in sends]
        ops += [dist.P2POp(dist.irecv, recv_buf[x["offset"]:x["offset"] + x["bytes"]],
                           gpu_rank[x["peer"]]) for x in recvs]
        if ops:
            for w in dist.batch_isend_irecv(ops):
                w.wait()
    return exchange

