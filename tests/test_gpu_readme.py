"""The Python usage example of the repository's readme runs as written on the GPU."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(__file__)), "README.md")


def test_readme_example_runs():
    text = open(README).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README has no python example"
    scope = {}
    exec(compile(blocks[0], "readme example", "exec"), scope)
    out, B = scope["out"], scope["B"]
    assert tuple(out.shape) == (B, 32, 128)
    assert bool(out.float().isfinite().all())
