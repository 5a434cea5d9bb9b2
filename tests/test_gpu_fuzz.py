"""Seeded fuzzing of the whole copy path on the GPU: random non-divisible tensors and
meshes (the uneven-stress generator at smaller sizes), random source and destination
misalignment, every destination byte and guard band checked against the oracle; the
cases together must reach every copy path and the transpose blocks."""
import random

import pytest

import dtensor_reshard_gb300 as rs
from inputs import uneven_stress
from tests import helpers
from tests.test_gpu_parity import run_and_compare

pytestmark = pytest.mark.gpu

N_CASES = 72
CASES = uneven_stress(n=N_CASES, seed=7331, max_dim=3000, max_numel=1 << 21,
                      max_bytes=256 << 20, name="fuzz").tensors
_rng = random.Random(7331)
# (source misalignment, destination misalignment rule) per case
MIS = [(_rng.choice([0, 0, 1, 2, 3, 4, 6, 8, 12]), _rng.choice(["same", "mixed", "zero"]))
       for _ in range(N_CASES)]
SEEN_PATHS = set()
SEEN_TRANSPOSES = []


def _dst_rule(rule, smis):
    if rule == "same":
        return lambda r: smis
    if rule == "zero":
        return lambda r: 0
    return lambda r: (3 * r + smis) % 16


def _fake(plan, side, n, mis):
    out = []
    for r in range(n):
        shp, _ = rs.reshard_plan_local_shape(plan, side, r)
        out.append(0 if 0 in shp else ((r + 1 + 4096 * side) << 24) + 512 + mis(r))
    return out


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_case(oracle, i):
    spec = CASES[i]
    smis, rule = MIS[i]
    dmis = _dst_rule(rule, smis)
    plan = helpers.spec_plan(spec)
    path = rs.reshard_plan_path(plan, _fake(plan, 0, plan.n_src, lambda r: smis),
                                _fake(plan, 1, plan.n_dst, dmis))[0]
    SEEN_PATHS.add(path)
    blocks, _ = rs.reshard_plan_transposes(plan, rs.PROGRAM_FANOUT)
    SEEN_TRANSPOSES.append(len(blocks) > 0)
    run_and_compare(oracle, spec, misalign=smis, dst_misalign=dmis, expect_path=path)
    if i % 3 == 0:
        run_and_compare(oracle, spec, kernel=rs.KERNEL_BOXCOPY, misalign=smis, dst_misalign=dmis)
    if i % 5 == 0:
        run_and_compare(oracle, spec, misalign=smis, path="gather_broadcast")


def test_zz_fuzz_reached_every_path():
    if len(SEEN_TRANSPOSES) < N_CASES:
        pytest.skip("run together with the fuzz cases")
    assert {"vector", "tma_fanout", "realign", "staged"} <= SEEN_PATHS, SEEN_PATHS
    assert any(SEEN_TRANSPOSES)
