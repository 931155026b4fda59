"""The C ABI driven from a plain C program (tests/native/abi_example.c) on the GPU."""
import subprocess

import pytest

from tests.test_abi import build_c_example

pytestmark = pytest.mark.gpu


def test_c_program_runs_a_round():
    r = subprocess.run([build_c_example()], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi example ok" in r.stdout
