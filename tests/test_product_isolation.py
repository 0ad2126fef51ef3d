"""The product path never reaches the oracle: the package's Python modules do not import it,
its C/CUDA sources include nothing from oracle/, the built library does not link it, and
importing the package (and its timing tools) leaves `oracle` out of sys.modules.  The oracle
is test infrastructure; a product path through it would be a CPU fallback."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "streaming_causal_video_gb300")


def test_package_sources_do_not_reference_the_oracle_module():
    for dirpath, _, files in os.walk(PKG):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h")):
                continue
            text = open(os.path.join(dirpath, f), encoding="utf-8").read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
            assert "liboracle" not in text and '#include "../../oracle' not in text, f


def test_importing_the_package_does_not_load_the_oracle():
    code = ("import sys; import streaming_causal_video_gb300, streaming_causal_video_gb300.layer, "
            "streaming_causal_video_gb300.kernel_timings, streaming_causal_video_gb300.stream_run; "
            "assert 'oracle' not in sys.modules, sorted(m for m in sys.modules if 'oracle' in m)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]


def test_library_does_not_link_the_oracle():
    import __graft_entry__
    path = __graft_entry__.build_library()
    path = path if isinstance(path, str) and os.path.exists(path) else os.path.join(PKG, "libsdv2.so")
    out = subprocess.run(["ldd", path], capture_output=True, text=True).stdout
    assert "oracle" not in out, out
