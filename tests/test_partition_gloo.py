"""The multi-GPU partition across processes: 2 and 4 gloo ranks on the CPU.

Each process stands for one GPU.  It builds the same plan and partition as the
others, runs only its own share (the test CPU tile executor on host buffers that
hold only its own source and destination ranks), exchanges the messages with
the other processes through torch.distributed point-to-point calls, and
compares every byte of its destination ranks with the oracle.
"""
import os
import random
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cases(world):
    """(spec, src_gpu, dst_gpu, gpu_domain, nchunks) built the same way on every rank."""
    from inputs import TensorSpec, workload

    import dtensor_reshard_gb300 as rs

    rng = random.Random(1000 + world)
    dom = [g // 2 for g in range(world)] if world > 2 else list(range(world))
    specs = [TensorSpec("w8x8", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",), init=("bits",),
                        seed=1)]
    for cfg in (2, 3, 5):
        specs += list(workload(cfg, reduced=True).tensors[:2])
    specs += list(workload(4, reduced=True).tensors[:6])
    out = []
    for k, spec in enumerate(specs):
        plan = rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                      spec.src_placements, spec.dst_mesh, spec.dst_placements)
        M, N = plan.n_src, plan.n_dst
        if k % 3 == 0:      # colocated: rank r of both layouts on GPU r mod world
            src_gpu, dst_gpu = [r % world for r in range(M)], [r % world for r in range(N)]
        elif k % 3 == 1:    # disaggregated: sources on the first domain, destinations after
            h = max(1, world // 2)
            src_gpu = [r % h for r in range(M)]
            dst_gpu = [h + r % (world - h) for r in range(N)]
        else:
            src_gpu = [rng.randrange(world) for _ in range(M)]
            dst_gpu = [rng.randrange(world) for _ in range(N)]
        out.append((spec, src_gpu, dst_gpu, dom, 1 + k % 3))
    return out


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import numpy as np
    import torch
    import torch.distributed as dist

    import dtensor_reshard_gb300 as rs
    import oracle as oracle_mod
    from inputs import global_tensor
    from tests import helpers

    dist.init_process_group("gloo", rank=rank, world_size=world)
    o = oracle_mod.load()
    report = []
    try:
        for spec, src_gpu, dst_gpu, dom, nchunks in _cases(world):
            glob = global_tensor(spec)
            src_bytes = [helpers.to_bytes(s) for s in helpers.scatter_with_oracle(
                o, glob, spec.src_mesh, spec.src_placements)]
            mine = [r for r, g in enumerate(dst_gpu) if g == rank]
            want = dict(zip(mine, o.reshard(spec.global_shape, spec.elem_bytes, spec.src_mesh,
                                            spec.src_placements, spec.dst_mesh,
                                            spec.dst_placements, src_bytes, dst_ranks=mine)))
            plan = helpers.spec_plan(spec)
            part = rs.reshard_partition_create(plan, src_gpu, dst_gpu, dom, nchunks)
            sizes = [0] * plan.n_dst
            for r in range(plan.n_dst):
                shp, _ = rs.reshard_plan_local_shape(plan, 1, r)
                sizes[r] = int(np.prod(shp)) * spec.elem_bytes
            # sources of other GPUs are never given to this process
            local_src = [b if src_gpu[r] == rank else np.zeros(0, np.uint8)
                         for r, b in enumerate(src_bytes)]
            bufs, writes = helpers.partition_gpu_buffers(part, rank, local_src, sizes, src_gpu,
                                                         dst_gpu)

            def exchange(gpu, sends, recvs, bufs=bufs):
                reqs = []
                for x in sends:
                    t = torch.from_numpy(bufs[-1][x["offset"]:x["offset"] + x["bytes"]])
                    reqs.append(dist.isend(t, dst=x["peer"], tag=2 * x["chunk"] + x["stage"]))
                for x in recvs:
                    t = torch.from_numpy(bufs[-2][x["offset"]:x["offset"] + x["bytes"]])
                    reqs.append(dist.irecv(t, src=x["peer"], tag=2 * x["chunk"] + x["stage"]))
                for r in reqs:
                    r.wait()

            # the library's executor, with the CPU tile executor for its steps
            rs.partition_run(part, rank, None, None, None, None, exchange,
                             run_step=lambda step, chunk, bufs=bufs, writes=writes, part=part:
                             helpers.run_partition_step_cpu(part, rank, step, chunk, bufs,
                                                            writes))
            M = plan.n_src
            bad = [r for r in mine if not np.array_equal(bufs[M + r], want[r]) or
                   not (writes[M + r] == 1).all()]
            st = rs.reshard_partition_gpu(part, rank)
            report.append((spec.name, nchunks, bad, st["recv_inter_bytes"] + st["recv_intra_bytes"]))
            dist.barrier()
        q.put((rank, "ok", report))
    except Exception as e:  # noqa: BLE001 - report to the parent
        import traceback
        q.put((rank, "error", traceback.format_exc()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_partition_over_gloo_ranks(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=600) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
    for rank, status, rep in res:
        assert status == "ok", f"rank {rank}:\n{rep}"
        for name, nchunks, bad, _ in rep:
            assert not bad, f"rank {rank}: {name} (chunks {nchunks}): destination ranks {bad}"
    # some bytes really crossed between the processes
    assert sum(sum(r[3] for r in rep) for _, _, rep in res) > 0
    for p in procs:
        assert p.exitcode == 0
