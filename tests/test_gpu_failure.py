"""Failure path of the copy kernels on the GPU, made without a fault: a barrier wait
that nothing answers runs out of its poll budget, the kernel records a status code
and returns, and the device stays usable (needs a GB300)."""
import pytest
import torch

import dtensor_reshard_gb300 as rs
from inputs import workload

pytestmark = pytest.mark.gpu


def test_unanswered_wait_reports_status_and_device_stays_usable():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    rs.reshard_device_status(clear=True)
    rs.reshard_selftest_wait_timeout(polls=2048)
    torch.cuda.synchronize()
    assert rs.reshard_device_status(clear=True) == 3
    assert rs.reshard_device_status() == 0
    # the context is intact: a reshard still runs and is exact
    spec = workload(1).tensors[0]
    g = torch.arange(64, dtype=torch.float32).reshape(8, 8).to(torch.bfloat16).cuda()
    plan = rs.reshard_plan_create(spec.global_shape, spec.dtype, spec.src_mesh,
                                  spec.src_placements, spec.dst_mesh, spec.dst_placements)
    srcs = [g[:4].contiguous(), g[4:].contiguous()]
    dsts = [torch.empty(8, 2, dtype=g.dtype, device="cuda") for _ in range(4)]
    rs.reshard_execute(plan, srcs, dsts)
    torch.cuda.synchronize()
    for j in range(4):
        assert torch.equal(dsts[j], g[:, 2 * j:2 * j + 2])
    assert rs.reshard_device_status() == 0


def test_selftest_rejects_unbounded_budget():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    with pytest.raises(rs.ReshardError):
        rs.reshard_selftest_wait_timeout(polls=0)
    with pytest.raises(rs.ReshardError):
        rs.reshard_selftest_wait_timeout(polls=(1 << 20) + 1)
