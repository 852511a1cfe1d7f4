"""The self-check predicates of the checked build (ptx.cuh), evaluated on the
host: the 16-byte rule for the innermost TMA coordinate, the 1024-byte
alignment of 128B-swizzled tiles, and the TMEM lane quarter and column range
of a warp's access.  Compiled with nvcc (host code only runs; no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

EXPECTED = {
    "coord_bf16_0": 1, "coord_bf16_64": 1, "coord_bf16_8": 1, "coord_bf16_4": 0,
    "coord_bf16_neg8": 1, "coord_bf16_neg3": 0, "coord_f32_4": 1, "coord_f32_2": 0,
    "coord_u8_16": 1, "coord_u8_8": 0,
    "tile_0": 1, "tile_16384": 1, "tile_512": 0, "tile_1040": 0,
    "tmem_w2_col0": 1, "tmem_w6_col480": 1, "tmem_w6_col481": 0, "tmem_w1_lane64": 0,
    "tmem_w0_lane0_col256": 1,
}


def test_selfcheck_predicates(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "selfcheck_predicates")
    src = os.path.join(ROOT, "tests", "selfcheck_predicates.cu")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-o", exe,
                    src], check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}
    assert got == EXPECTED
