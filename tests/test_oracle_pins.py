"""The CPU oracle against facts it does not produce itself (runs without a GPU)."""
import json
import os
import subprocess
import sys

import pytest

import oracle as oracle_mod
from tests import oracle_pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("name", list(oracle_pins.PINS))
def test_oracle_pin(name, oracle):
    oracle_pins.PINS[name](oracle)


# Each planted mistake is a plausible slip in the oracle (see ORACLE_PLANT in
# oracle.c).  The pins above must catch every one of them; they run in a child
# process because a wrong index can make the planted oracle read out of bounds.
PLANTS = {
    1: "chunk size floor(n/k) instead of ceil(n/k)",
    2: "column-major local layout",
    4: "closed upper bound in the box containment test",
    5: "mesh dims applied innermost first",
    6: "empty-shard offset convention skipped",
    7: "outer split offset dropped in nested sharding",
    8: "range start index unravelled with the first dim fastest",
    9: "range start index unravel drops the carry into outer dims",
}


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_planted_mistake_is_caught(plant, tmp_path):
    lib = oracle_mod.build(plant=plant, out=str(tmp_path / f"liboracle_plant{plant}.so"))
    proc = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), lib],
                          capture_output=True, text=True, timeout=600)
    if proc.returncode != 0:
        return  # the planted oracle crashed outright: caught
    res = json.loads(proc.stdout.strip().splitlines()[-1])
    failed = [k for k, v in res.items() if v != "ok"]
    assert failed, f"planted mistake {plant} ({PLANTS[plant]}) passed every pin"
