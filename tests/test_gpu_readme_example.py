"""The Python example in the top-level readme runs as written (a delayed-scaling step)."""
import os
import re

import pytest

from conftest import ROOT


@pytest.mark.gpu
def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "no python example in the readme"
    ns = {}
    exec(compile(blocks[0], "readme example", "exec"), ns)
    import torch
    torch.cuda.synchronize()
    # the update moved each slot's amax into the history and set scale = amax / 448
    assert float(ns["history"][0, 0]) > 0 and float(ns["history"][0, 1]) > 0
    assert torch.all(ns["scale"] != 1.0)
    assert float(ns["amax"].abs().sum()) == 0.0
