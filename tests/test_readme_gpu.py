"""The Python example in README.md runs as written (its asserts included)."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example():
    from paged_kv_prep_gb300 import build as pbuild

    pbuild.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README.md has no python example"
    for code in blocks:
        exec(compile(code, "README.md", "exec"), {})
