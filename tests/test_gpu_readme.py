"""The README's Python example runs as written (one fused decode step)."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in the README"
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    o, status = scope["o"], scope["status"]
    assert int(status.item()) == 0
    assert bool(o.float().isfinite().all())
    assert float(o.float().abs().max()) > 0.0
