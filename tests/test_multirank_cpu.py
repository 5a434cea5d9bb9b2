"""The benchmark's multi-rank path (barrier, max/sum over ranks, weak-scaling value) on
two gloo ranks on the CPU, plus planning done independently on every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import dtensor_reshard_gb300 as rs
    from inputs import moe_refit
    ctx = bench.DistCtx(world)
    ctx.barrier()
    # every rank plans its own layer (independent problems); bytes are identical
    w = moe_refit()
    eff = 0
    for spec in w.tensors:
        p = rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                   spec.src_placements, spec.dst_mesh, spec.dst_placements)
        st = rs.reshard_plan_stats(p)
        eff += st["global_bytes"] + st["dst_bytes"]
    my_ms = 10.0 + rank  # rank 1 is the slowest
    ms = ctx.max(my_ms)
    total = ctx.sum(float(eff))
    q.put((rank, ms, total, eff))
    ctx.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    eff = res[0][3]
    assert res[0][3] == res[1][3]
    for _, ms, total, _ in res:
        assert ms == 11.0                     # max over ranks
        assert total == pytest.approx(2 * eff)  # sum over ranks
    value = res[0][2] / (res[0][1] * 1e-3) / 1e9
    assert value == pytest.approx(2 * eff / 11e-3 / 1e9)


def test_reference_arm_other_ranks_exit_quietly(capsys):
    import bench
    args = bench.parse_args(["--impl", "reference"])
    assert bench.reference_arm(args, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
