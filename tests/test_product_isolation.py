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


def test_missing_library_fails_loudly():
    """Without libsdv2.so every entry point raises; nothing falls back to another path."""
    code = ("import streaming_causal_video_gb300._binding as b, streaming_causal_video_gb300 as sd\n"
            "b._LIB = None; b._LIB_PATH = '/nonexistent/libsdv2.so'\n"
            "cfg = sd.StreamConfig.make(batch=1, heads=1, head_dim=128, rope_t=44, rope_h=42, rope_w=42,\n"
            "    rope_base=1e4, grid_h=2, grid_w=2, chunk_frames=1, sink_frames=1, window_frames=1)\n"
            "for call in (lambda: sd.workspace_bytes(cfg), lambda: sd.visible_tokens(cfg, 0),\n"
            "             lambda: sd.chunk_attention(cfg, [0], 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, stream=0)):\n"
            "    try:\n"
            "        call()\n"
            "    except RuntimeError as e:\n"
            "        assert 'not built' in str(e), e\n"
            "    else:\n"
            "        raise SystemExit('an entry point ran without the library')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
