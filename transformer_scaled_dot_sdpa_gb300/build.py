"""Build libgb300attn.so in-tree with nvcc (sm_103a only).

    python transformer_scaled_dot_sdpa_gb300/build.py [--verbose]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libgb300attn.so")
LIB_CHECKED = os.path.join(HERE, "libgb300attn_checked.so")  # self-checking build
SOURCES = [os.path.join(CSRC, "capi.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(os.path.dirname(HERE), "include", "gb300attn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Build libgb300attn.so, or with ``checked`` the self-checking build
    libgb300attn_checked.so (GB300_CHECKED: TMA and TMEM preconditions tested
    before every access)."""
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-o", tmp, *SOURCES]
    if checked:
        cmd.append("-DGB300_CHECKED")
    if verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """Both builds, compiled in parallel."""
    import concurrent.futures
    with concurrent.futures.ThreadPoolExecutor(2) as ex:
        for f in [ex.submit(build, force, False, c) for c in (False, True)]:
            f.result()


if __name__ == "__main__":
    checked = "--checked" in sys.argv
    print(build(force=True, verbose="--verbose" in sys.argv, checked=checked))
