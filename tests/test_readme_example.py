"""The Python example in README.md runs as written (GPU), so the documented calls stay in
step with the binding."""
import re
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def test_readme_python_example_runs():
    import __graft_entry__ as g
    g.build()
    text = (ROOT / "README.md").read_text()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README.md has no python example"
    ns = {}
    exec(compile(blocks[0], "README.md", "exec"), ns)
    import torch
    torch.cuda.synchronize()
    # the example's zero inputs give an exactly zero update and zero outputs
    assert torch.count_nonzero(ns["master"]) == 0 and torch.count_nonzero(ns["param"].float()) == 0
    assert torch.count_nonzero(ns["Y"]) == 0
