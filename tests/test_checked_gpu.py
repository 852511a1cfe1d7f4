"""The self-checking build (libgb300attn_checked.so): every TMA copy and TMEM
access of a battery of calls over all entry points passes its precondition
checks (no ATTN_ERR_SELF_CHECK), and the results are bit-identical to the
normal build's."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_agrees_and_reports_nothing(cuda_lib, tmp_path):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_gb300attn_build", os.path.join(ROOT, "transformer_scaled_dot_sdpa_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(checked=True)
    path = str(tmp_path / "checked.npz")
    env = dict(os.environ, GB300ATTN_CHECKED="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_battery.py"), path],
                         env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    checked = np.load(path)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import checked_battery
    assert not cuda_lib.is_checked_build()
    normal = checked_battery.run(cuda_lib)
    assert sorted(checked.files) == sorted(normal)
    for k in normal:
        assert np.array_equal(checked[k], normal[k]), k
