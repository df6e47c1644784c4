"""The README's Python example runs as written (GPU)."""

import os
import re

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs(pa, capsys):
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README has no python example"
    exec(compile(blocks[0], "README.md", "exec"), {})
    out = capsys.readouterr().out
    assert "frames_in_use" in out
    assert pa.pa_get_device_status() == 0
