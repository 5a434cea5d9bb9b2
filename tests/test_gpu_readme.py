"""The README's Python example, run as written: the fan-out and the gather-and-broadcast
baseline both give every destination rank its column band of the global matrix."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def _python_example():
    text = open(README).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README has no python example"
    return blocks[0]


def test_readme_python_example_runs_and_is_exact():
    ns = {}
    exec(compile(_python_example(), "README.md", "exec"), ns)
    torch.cuda.synchronize()
    g, dsts = ns["g"], ns["dsts"]
    assert len(dsts) == 4
    for r, d in enumerate(dsts):
        # Shard(1) over 4 ranks of 8 columns: rank r holds columns 2r, 2r + 1
        assert torch.equal(d, g[:, 2 * r:2 * r + 2]), r
