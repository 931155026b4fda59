"""The README's Python example runs as written (on the GPU)."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in README.md"
    for code in blocks:
        scope = {}
        exec(compile(code, "README.md", "exec"), scope)
        if "ctx" in scope:
            import server_side_fedavg_gb300 as fa
            fa.fa_close(scope["ctx"])
