"""CPU tests of bench.py's host-side helpers: the source hash that keys the committed ncu
traffic record, the peak lookup, and the parsing of the clock samples taken during the timed
region (fed synthetic nvidia-smi lines; no GPU, no nvidia-smi)."""
import json
import os
import threading

import bench

CSRC = os.path.join(bench.ROOT, "streaming_causal_video_gb300", "csrc")


def _read(f):
    with open(os.path.join(CSRC, f)) as fh:
        return fh.read()


def test_source_hash_ignores_comments_and_sees_code():
    base = bench.attention_source_hash(_read)
    assert base == bench.attention_source_hash()
    commented = lambda f: _read(f) + ("\n// a new comment\n/* and a block\n comment */\n" if f == "attention.cu" else "")
    assert bench.attention_source_hash(commented) == base
    edited = lambda f: _read(f).replace("kRescaleThreshold", "kRescaleThreshold2", 1) if f == "attention.cu" else _read(f)
    assert bench.attention_source_hash(edited) != base
    assert bench.code_only("a /* x */ b // y\n  c") == "a b c"


def test_traffic_record_is_used_only_for_the_source_it_was_taken_on(monkeypatch):
    path = os.path.join(bench.ROOT, "profiles", "chunk_attention_wan13b_480p.json")
    with open(path) as fh:
        rec = json.load(fh)
    got = bench.profiled_traffic("wan13b_480p")
    if rec["source_hash"] == bench.attention_source_hash():
        assert got == rec["dram_bytes_per_launch"]
    else:
        assert got is None
    monkeypatch.setattr(bench, "attention_source_hash", lambda read=None: "0" * 16)
    assert bench.profiled_traffic("wan13b_480p") is None
    assert bench.profiled_traffic("no_such_workload") is None


def test_peak_lookup_at_any_nesting():
    assert bench.peak_value({"hbm_gbs": 7000}, "hbm_gbs") == 7000.0
    assert bench.peak_value({"gemm": {"bf16": {"bf16_tflops_sustained": 1690.3}}}, "bf16_tflops_sustained") == 1690.3
    assert bench.peak_value({"hbm": {"gbs": "n/a"}}, "hbm_gbs") is None
    d, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    if src == "fallback":
        assert d == bench.PEAK_FALLBACK


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _summary(lines):
    s = bench.ClockSampler(0)
    s.proc = _FakeProc()
    s.thread = threading.Thread(target=lambda: None)
    s.thread.start()
    s.lines = list(lines)
    return s.stop()


def test_clock_samples_give_median_max_and_active_reasons():
    lines = ["1905, 2070, 1350.2, 0x4, Not Active, Not Active, Not Active, Active",
             "1860, 2070, 1371.0, 0x4, Not Active, Not Active, Not Active, Active",
             "1920, 2070, 1302.5, 0x0, Not Active, Not Active, Not Active, Not Active",
             "[N/A], 2070, 1300, 0x0, Not Active, Not Active, Not Active, Not Active",   # skipped
             "garbage"]                                                                   # skipped
    r = _summary(lines)
    assert r["sm_mhz"] == 1905.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["power_w"] == 1350.2
    assert r["reasons"] == ["sw_power_cap"]
    r = _summary(["1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active"])
    assert r["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]


# The text of get_encode_tiled in the build the ncu traffic record was captured on.
def test_cpu_baseline_entry_times_attention_rope_append_and_motion():
    """The bench's CPU-baseline leg on the tiny workload with short samples: all three parts of
    the path are timed on all cores and on one thread, with their units and core counts."""
    from synth_inputs import WORKLOADS, motion_frames_host
    w = WORKLOADS["tiny"]
    frames = motion_frames_host(1, 5, 16, 32, 3, seed=2).numpy()
    out = bench.cpu_baseline_entry(w, frames, seconds=0.2, single_seconds=0.1, rope_seconds=0.1,
                                   motion_seconds=0.05)
    assert out["kind"] == "oracle" and out["value"] > 0 and out["single_thread_value"] > 0
    for part in ("rope_append", "motion"):
        d = out[part]
        assert d["unit"] == "GB/s" and d["value"] > 0 and d["single_thread_value"] > 0
        assert d["cores"] >= 1 and d["kind"] == "oracle"
    t = out["tiny_run"]
    assert t["unit"] == "s per run" and t["value"] > 0 and t["single_thread_value"] > 0 and t["tflops"] > 0
    assert "motion" not in bench.cpu_baseline_entry(w, None, seconds=0.1, single_seconds=0.05,
                                                    rope_seconds=0.05)
