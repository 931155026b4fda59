"""The README's Python example (tests/example_round.py, quoted there) runs as written
on the GPU."""
import os
import runpy

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_example_round_runs():
    runpy.run_path(os.path.join(HERE, "example_round.py"), run_name="__example__")
