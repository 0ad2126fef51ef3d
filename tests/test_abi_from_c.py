"""The boundary is usable from plain C: tests/c_abi/abi_from_c.c includes only include/sdv2.h,
links the built libsdv2.so with gcc and checks the host-side contract (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_against_the_abi():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    import __graft_entry__
    __graft_entry__.build_library()
    pkg = os.path.join(ROOT, "streaming_causal_video_gb300")
    out = os.path.join(pkg, "_build")             # in-tree build folder (not committed)
    os.makedirs(out, exist_ok=True)
    exe = os.path.join(out, "abi_from_c")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_from_c.c"), "-o", exe, os.path.join(pkg, "libsdv2.so"),
           "-Wl,-rpath," + pkg]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all host-side checks passed" in r.stdout
