"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError (or OracleError)
when the oracle disagrees with:
  * the worked example printed on the pages (tests/golden/worked_example_8x8.txt);
  * torch.chunk, the library routine DTensor's Shard placement is defined by
    (1-D meshes, and nested chunking mesh dim by mesh dim for n-D meshes);
  * PyTorch DTensor's own local-shape/offset utility (CPU, no process group);
  * brute force over small tensors, meshes and placements, where the expected
    destination shards are sliced out of the global tensor with torch.chunk;
  * the invariants that destination shards reassemble the global tensor and
    that replicas are equal;
  * HybridFlow's strided-rank property: a generation shard is the concatenation
    of its micro-group's training shards.

Run as a script (``python tests/oracle_pins.py LIB``) it executes every pin
against the oracle library at LIB and prints a JSON map pin -> "ok" | error.
The planted-mistake test uses that to show each planted mistake is caught.
"""
from __future__ import annotations

import json
import math
import os
import random
import sys

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
for p in (_ROOT, _HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import torch_chunk_layout as tcl  # noqa: E402

GOLDEN = os.path.join(_HERE, "golden", "worked_example_8x8.txt")


def _bytes(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous()
    return t.view(torch.uint8).reshape(-1).numpy().copy() if t.numel() else \
        np.zeros(0, dtype=np.uint8)


def _bits_tensor(shape, elem_bytes, seed):
    g = torch.Generator().manual_seed(seed)
    n = math.prod(shape)
    raw = torch.randint(0, 256, (n * elem_bytes,), generator=g, dtype=torch.uint8)
    return raw, shape


def _raw_global(shape, elem_bytes, seed):
    """A global tensor of random bytes, as a uint8 tensor of shape [*shape, elem_bytes]."""
    raw, _ = _bits_tensor(shape, elem_bytes, seed)
    return raw.reshape(*shape, elem_bytes) if shape else raw


def parse_golden(path=GOLDEN):
    out = {"shards": {"src": {}, "dst": {}}, "blocks": [], "layout": {}}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            if line[0] == "global":
                out["global"] = tuple(int(x) for x in line[1:])
            elif line[0] == "layout":
                out["layout"][line[1]] = ((int(line[2]),), (line[3],))
            elif line[0] == "shard":
                r0, c0, nr, nc = (int(x) for x in line[3:7])
                out["shards"][line[1]][int(line[2])] = ((r0, c0), (nr, nc))
            elif line[0] == "block":
                out["blocks"].append(tuple(int(x) for x in line[1:]))
    return out


# ------------------------------------------------------------------------------------ pins
def pin_worked_example(o):
    """The 8x8 example: shard shapes and the 4x2 blocks each destination receives."""
    gd = parse_golden()
    gshape = gd["global"]
    (sm, sp), (dm, dp) = gd["layout"]["src"], gd["layout"]["dst"]
    for side, mesh, pl in (("src", sm, sp), ("dst", dm, dp)):
        for r, (off, shp) in gd["shards"][side].items():
            assert o.resolve(gshape, mesh, pl, r) == (off, shp), (side, r)
    # sources cut straight from the fixture's statement of the source shards
    glob = _raw_global(gshape, 2, seed=11)
    srcs = []
    for r in range(2):
        (r0, c0), (nr, nc) = gd["shards"]["src"][r]
        srcs.append(glob[r0:r0 + nr, c0:c0 + nc].contiguous())
    outs = o.reshard(gshape, 2, sm, sp, dm, dp, [_bytes(s) for s in srcs])
    covered = {r: np.zeros((8, 2), dtype=bool) for r in range(4)}
    nblocks = {r: 0 for r in range(4)}
    for (dr, sr, sr0, sc0, dr0, dc0, nr, nc) in gd["blocks"]:
        got = outs[dr].reshape(8, 2, 2)[dr0:dr0 + nr, dc0:dc0 + nc]
        want = srcs[sr][sr0:sr0 + nr, sc0:sc0 + nc].numpy()
        assert np.array_equal(got, want), ("block", dr, sr)
        covered[dr][dr0:dr0 + nr, dc0:dc0 + nc] = True
        nblocks[dr] += 1
    for r in range(4):
        assert covered[r].all() and nblocks[r] == 2, r


def pin_resolve_chunk_1d(o):
    """1-D meshes: local shapes/offsets equal torch.chunk's pieces (empty tail ranks)."""
    for n in range(0, 23):
        for k in range(1, 10):
            pieces = torch.chunk(torch.arange(n), k) if n else ()
            for c in range(k):
                off, shp = o.resolve((n,), (k,), ("S0",), c)
                if c < len(pieces) and pieces[c].numel():
                    assert (off, shp) == ((int(pieces[c][0]),), (pieces[c].numel(),)), (n, k, c)
                else:
                    assert shp == (0,) and off == (n,), (n, k, c, off, shp)


def _layout_space(seed, tensor_ndims=(1, 2, 3), shapes_per=2, max_ranks=4, max_dim=7):
    rng = random.Random(seed)
    for nd in tensor_ndims:
        for mesh in tcl.all_meshes(max_ranks):
            for pl in tcl.all_placements(len(mesh), nd):
                for _ in range(shapes_per):
                    yield tuple(rng.randint(0, max_dim) for _ in range(nd)), mesh, pl


def pin_resolve_nested_chunk(o):
    """n-D meshes: nested torch.chunk, mesh dim 0 outermost, over all small layouts."""
    for gshape, mesh, pl in _layout_space(seed=1):
        for r in range(math.prod(mesh)):
            assert o.resolve(gshape, mesh, pl, r) == tcl.box(gshape, mesh, pl, r), \
                (gshape, mesh, pl, r)


def pin_resolve_dtensor(o):
    """PyTorch DTensor's local shape/offset utility agrees on every small layout."""
    try:
        from torch.distributed.tensor import Replicate, Shard
        from torch.distributed.tensor._utils import _compute_local_shape_and_global_offset
    except Exception:  # pragma: no cover - older/newer torch without the helper
        return
    for gshape, mesh, pl in _layout_space(seed=2, shapes_per=1):
        tpl = [Replicate() if p == "R" else Shard(int(p[1:])) for p in pl]
        for r in range(math.prod(mesh)):
            shp, off = _compute_local_shape_and_global_offset(gshape, mesh, list(tcl.coords(mesh, r)),
                                                              tpl)
            got_off, got_shp = o.resolve(gshape, mesh, pl, r)
            assert got_shp == tuple(shp), (gshape, mesh, pl, r)
            if math.prod(got_shp):
                assert got_off == tuple(off), (gshape, mesh, pl, r, got_off, off)
            else:
                for d in range(len(gshape)):
                    if got_shp[d] == 0:
                        assert got_off[d] == off[d], (gshape, mesh, pl, r)


def _check_pair(o, gshape, elem_bytes, sm, sp, dm, dp, seed):
    glob = _raw_global(gshape, elem_bytes, seed)
    srcs = [_bytes(tcl.local_shard(glob, sm, sp, r)) for r in range(math.prod(sm))]
    outs = o.reshard(gshape, elem_bytes, sm, sp, dm, dp, srcs)
    for r in range(math.prod(dm)):
        want = _bytes(tcl.local_shard(glob, dm, dp, r))
        assert np.array_equal(outs[r], want), (gshape, sm, sp, dm, dp, r)


def pin_reshard_bruteforce(o):
    """Brute force: every destination shard equals torch.chunk slicing of the global tensor."""
    rng = random.Random(3)
    layouts = {nd: [(m, p) for m in tcl.all_meshes(4) for p in tcl.all_placements(len(m), nd)]
               for nd in (1, 2, 3)}
    # exhaustive over 1-D layouts of a ragged 1-D and 2-D tensor
    for gshape in ((7,), (5, 3)):
        nd = len(gshape)
        one_d = [(m, p) for (m, p) in layouts[nd] if len(m) == 1]
        for (sm, sp) in one_d:
            for (dm, dp) in one_d:
                _check_pair(o, gshape, 2, sm, sp, dm, dp, seed=rng.randrange(1 << 30))
    # random pairs over all layouts, tensor ndim 1..3, dims 0..7, element sizes 1/2/4/8
    for _ in range(600):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(0 if rng.random() < 0.05 else 1, 7) for _ in range(nd))
        (sm, sp), (dm, dp) = rng.choice(layouts[nd]), rng.choice(layouts[nd])
        _check_pair(o, gshape, rng.choice((1, 2, 4, 8)), sm, sp, dm, dp,
                    seed=rng.randrange(1 << 30))


def pin_reassembly_and_replicas(o):
    """Destination shards reassemble the global tensor; replicas hold identical bytes."""
    rng = random.Random(4)
    for _ in range(150):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 9) for _ in range(nd))
        sm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        dm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        sp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in sm)
        dp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in dm)
        glob = _raw_global(gshape, 4, rng.randrange(1 << 30))
        srcs = [_bytes(tcl.local_shard(glob, sm, sp, r)) for r in range(math.prod(sm))]
        outs = o.reshard(gshape, 4, sm, sp, dm, dp, srcs)
        canvas = np.zeros(tuple(gshape) + (4,), dtype=np.uint8)
        hit = np.zeros(tuple(gshape), dtype=np.int64)
        seen = {}
        for r, buf in enumerate(outs):
            off, shp = tcl.box(gshape, dm, dp, r)
            if math.prod(shp) == 0:
                continue
            sl = tuple(slice(a, a + b) for a, b in zip(off, shp))
            blk = buf.reshape(tuple(shp) + (4,))
            if (off, shp) in seen:
                assert np.array_equal(seen[(off, shp)], blk), "replicas differ"
                continue
            seen[(off, shp)] = blk
            canvas[sl] = blk
            hit[sl] += 1
        assert (hit == 1).all(), "distinct dst boxes must tile the tensor exactly once"
        assert np.array_equal(canvas, glob.numpy()), (gshape, sm, sp, dm, dp)
        total = sum(b.size for b in outs)
        assert total == sum(4 * math.prod(tcl.box(gshape, dm, dp, r)[1])
                            for r in range(math.prod(dm)))


def pin_hybridflow_concat(o):
    """Strided generation ranks: dst rank 4t+d = concat(training shards 4t..4t+3).

    The property holds when the sharded dim divides evenly by the training TP size.
    """
    for gshape in ((40, 5), (32, 3), (8, 7), (64, 1)):
        glob = _raw_global(gshape, 2, seed=5)
        sm, sp, dm, dp = (8,), ("S0",), (2, 4), ("S0", "R")
        srcs = [tcl.local_shard(glob, sm, sp, r) for r in range(8)]
        outs = o.reshard(gshape, 2, sm, sp, dm, dp, [_bytes(s) for s in srcs])
        for r in range(8):
            t = r // 4
            want = _bytes(torch.cat(srcs[4 * t:4 * t + 4], dim=0))
            assert np.array_equal(outs[r], want), (gshape, r)


def pin_gather_full(o):
    """The all-gather intermediate equals the global tensor."""
    rng = random.Random(6)
    for _ in range(80):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 8) for _ in range(nd))
        sm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 3)))
        sp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in sm)
        glob = _raw_global(gshape, 2, rng.randrange(1 << 30))
        srcs = [_bytes(tcl.local_shard(glob, sm, sp, r)) for r in range(math.prod(sm))]
        full = o.gather_full(gshape, 2, sm, sp, srcs)
        assert np.array_equal(full, _bytes(glob)), (gshape, sm, sp)


def pin_source_of(o):
    """Single-element mapping agrees with torch.chunk index lists."""
    rng = random.Random(7)
    for _ in range(300):
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 9) for _ in range(nd))
        sm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        dm = tuple(rng.randint(1, 4) for _ in range(rng.randint(1, 2)))
        sp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in sm)
        dp = tuple(rng.choice(["R"] + [f"S{d}" for d in range(nd)]) for _ in dm)
        r = rng.randrange(math.prod(dm))
        didx = tcl.index_lists(gshape, dm, dp, r)
        n = math.prod(len(ix) for ix in didx)
        if n == 0:
            continue
        e = rng.randrange(n)
        loc = np.unravel_index(e, tuple(len(ix) for ix in didx))
        g = tuple(int(didx[d][loc[d]]) for d in range(nd))
        s, j = o.source_of(gshape, sm, sp, dm, dp, r, e)
        sidx = tcl.index_lists(gshape, sm, sp, s)
        sloc = np.unravel_index(j, tuple(len(ix) for ix in sidx))
        assert tuple(int(sidx[d][sloc[d]]) for d in range(nd)) == g, (gshape, sm, sp, dm, dp)
        # first owner in flat order
        for s2 in range(s):
            ix2 = tcl.index_lists(gshape, sm, sp, s2)
            assert not all(g[d] in set(ix2[d].tolist()) for d in range(nd)), "not first owner"


def pin_reshard_elems(o):
    """A range [e_begin, e_end) of one destination rank: exactly that slice of the
    torch.chunk-sliced expected shard is written, and nothing outside it.

    Ranges start anywhere (mid-row, mid-plane, at the last element), so the
    unravel of the start index into a multi-index is exercised, not only e = 0.
    """
    rng = random.Random(8)
    layouts = {nd: [(m, p) for m in tcl.all_meshes(4) for p in tcl.all_placements(len(m), nd)]
               for nd in (1, 2, 3)}
    checked = 0
    while checked < 400:
        nd = rng.choice((1, 2, 3))
        gshape = tuple(rng.randint(1, 9) for _ in range(nd))
        (sm, sp), (dm, dp) = rng.choice(layouts[nd]), rng.choice(layouts[nd])
        eb = rng.choice((1, 2, 4, 8))
        glob = _raw_global(gshape, eb, rng.randrange(1 << 30))
        srcs = [_bytes(tcl.local_shard(glob, sm, sp, r)) for r in range(math.prod(sm))]
        r = rng.randrange(math.prod(dm))
        want = _bytes(tcl.local_shard(glob, dm, dp, r))
        n = want.size // eb
        if n < 2:
            continue
        e0 = rng.randrange(n)
        e1 = rng.randrange(e0, n + 1)
        sentinel = np.full(want.size, 0xA5, dtype=np.uint8)
        out = sentinel.copy()
        ptrs = [b.ctypes.data if b.size else None for b in srcs]
        o.reshard_elems(gshape, eb, sm, sp, dm, dp, ptrs, out.ctypes.data, r, e0, e1)
        assert np.array_equal(out[e0 * eb:e1 * eb], want[e0 * eb:e1 * eb]), \
            (gshape, sm, sp, dm, dp, r, e0, e1)
        assert np.array_equal(out[:e0 * eb], sentinel[:e0 * eb]), "wrote before e_begin"
        assert np.array_equal(out[e1 * eb:], sentinel[e1 * eb:]), "wrote past e_end"
        checked += 1
    # splitting a rank into consecutive ranges reproduces the whole shard
    for gshape, sm, sp, dm, dp in (((9, 7, 5), (2, 2), ("S0", "S2"), (3,), ("S1",)),
                                   ((7, 8), (4,), ("S1",), (2, 2), ("S0", "R"))):
        glob = _raw_global(gshape, 2, seed=81)
        srcs = [_bytes(tcl.local_shard(glob, sm, sp, r)) for r in range(math.prod(sm))]
        ptrs = [b.ctypes.data if b.size else None for b in srcs]
        for r in range(math.prod(dm)):
            want = _bytes(tcl.local_shard(glob, dm, dp, r))
            out = np.zeros_like(want)
            n = want.size // 2
            cuts = sorted({0, n, *(rng.randrange(n + 1) for _ in range(4))})
            for a, b in zip(cuts, cuts[1:]):
                o.reshard_elems(gshape, 2, sm, sp, dm, dp, ptrs, out.ctypes.data, r, a, b)
            assert np.array_equal(out, want), (gshape, r, cuts)


PINS = {
    "worked_example": pin_worked_example,
    "resolve_chunk_1d": pin_resolve_chunk_1d,
    "resolve_nested_chunk": pin_resolve_nested_chunk,
    "resolve_dtensor": pin_resolve_dtensor,
    "reshard_bruteforce": pin_reshard_bruteforce,
    "reassembly_and_replicas": pin_reassembly_and_replicas,
    "hybridflow_concat": pin_hybridflow_concat,
    "gather_full": pin_gather_full,
    "source_of": pin_source_of,
    "reshard_elems": pin_reshard_elems,
}


def run_all(lib_path):
    import oracle as oracle_mod
    o = oracle_mod.Oracle(lib_path)
    res = {}
    for name, fn in PINS.items():
        try:
            fn(o)
            res[name] = "ok"
        except Exception as e:  # noqa: BLE001 - report every failure kind
            res[name] = f"{type(e).__name__}: {str(e)[:200]}"
    return res


if __name__ == "__main__":
    print(json.dumps(run_all(sys.argv[1])))
