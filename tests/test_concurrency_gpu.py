"""The library's one-time set-up under concurrent first calls: a fresh process
(tests/concurrent_first_calls.py) starts eight host threads that make their
first attention, decode and GEMM calls at once on separate streams, and
checks every result against the same call made from one thread."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_concurrent_first_calls(cuda_lib):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "concurrent_first_calls.py")],
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "concurrent first calls ok" in res.stdout
