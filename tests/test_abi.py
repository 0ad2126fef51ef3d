"""CPU tests of the C ABI: the library loads, exports what the header declares, and its host
logic (sizes, visible prefix, argument validation) agrees with the oracle's list model.
No kernel is launched here."""
import ctypes
import os
import re

import pytest

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS, stream_config_dict

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "sdv2.h")).read()
    return sorted(set(re.findall(r"\b(sdv2_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    declared = header_functions()
    assert len(declared) == 23, declared
    L = sd.lib()
    missing = [n for n in declared if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(sd.exported_symbols()) == declared


def test_config_struct_layout():
    assert ctypes.sizeof(sd.StreamConfig) == 64
    assert sd.StreamConfig.rope_base.offset == 24
    assert sd.StreamConfig.qkv_token_stride.offset == 56


def _cfg(name="tiny", **over):
    d = stream_config_dict(WORKLOADS[name])
    d.update(over)
    return sd.StreamConfig.make(**d)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_sizes(name):
    w = WORKLOADS[name]
    c = _cfg(name)
    assert sd.cache_bytes(c) == w.batch * w.heads * w.slots * w.hw * w.head_dim * 2
    assert sd.meta_bytes(c) == w.batch * w.slots * 16
    assert sd.workspace_bytes(c) >= 256 + (w.grid_h * 21 + w.grid_w * 21) * 8


@pytest.mark.parametrize("F,Fs,W", [(3, 3, 4), (3, 3, 18), (3, 2, 3), (3, 0, 6), (2, 5, 2), (1, 1, 1)])
def test_visible_tokens_equals_list_model(F, Fs, W):
    c = _cfg(chunk_frames=F, sink_frames=Fs, window_frames=W)
    cache = oracle.FrameListCache(Fs, W)
    hw = c.grid_h * c.grid_w
    for ch in range(40):
        for i in range(F):
            cache.append(ch * F + i, 0, None, None)
        assert sd.visible_tokens(c, ch) == len(cache.frames()) * hw
    assert sd.visible_tokens(c, -1) == -1


def _status(fn, *args):
    with pytest.raises(sd.SDV2Error) as e:
        fn(*args)
    return e.value.status


FAKE = 1 << 20          # an aligned non-null address; every call below is rejected before use


@pytest.mark.parametrize("over,status", [
    (dict(rope_t=46), 1),                       # split does not sum to head_dim
    (dict(rope_t=43, rope_h=43), 1),            # odd split
    (dict(head_dim=64, rope_t=22, rope_h=22, rope_w=20), 2),   # not built
    (dict(window_frames=2), 1),                 # window smaller than a chunk
    (dict(sink_frames=-1), 1),
    (dict(refresh_chunks=-2), 1),
    (dict(rope_base=1.0), 1),
    (dict(qkv_token_stride=12), 1),             # smaller than H*D
    (dict(grid_h=0), 1),
])
def test_invalid_configs_are_rejected(over, status):
    c = _cfg(**over)
    assert sd.cache_bytes(c) == 0
    assert _status(sd.rope_append_kv, c, [0], [0], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == status
    assert _status(sd.chunk_attention, c, [0], FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.0, 0) == status


def test_invalid_pointers_and_indices_are_rejected():
    c = _cfg()
    assert _status(sd.rope_append_kv, c, [0], [0], FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert _status(sd.rope_append_kv, c, [0], [-1], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert _status(sd.rope_append_kv, c, [-5], [0], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == 1
    assert _status(sd.chunk_attention, c, [-1], FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.0, 0) == 1
    assert _status(sd.chunk_attention, c, [0], 0, FAKE, FAKE, FAKE, FAKE, None, 0.0, 0) == 1
    big = _cfg(batch=17)
    assert _status(sd.chunk_attention, big, [0] * 17, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.0, 0) == 2
    wide = _cfg(batch=30)     # 30 streams x 3 frames > 64 frames per append call
    assert _status(sd.rope_append_kv, wide, [0] * 30, [0] * 30, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                   FAKE, 0) == 2


def test_motion_argument_checks():
    L = sd.lib()
    assert L.sdv2_motion_l2(FAKE, 1, 1, 3, 5, 1, FAKE, None, None) == 1        # 15 bytes per frame
    assert b"multiple of 16" in L.sdv2_last_error()
    assert L.sdv2_motion_l2(FAKE, 1, 0, 4, 4, 1, FAKE, None, None) == 1        # T = 0
    assert L.sdv2_motion_l2(FAKE + 4, 1, 1, 4, 4, 1, FAKE, None, None) == 1    # misaligned
    assert L.sdv2_motion_l2(None, 1, 1, 4, 4, 1, FAKE, None, None) == 1
    assert L.sdv2_motion_l2(FAKE, 1 << 10, 64, 4, 4, 1, FAKE, None, None) == 2  # B*T > 65535


def test_status_strings():
    L = sd.lib()
    assert L.sdv2_status_string(0) == b"ok"
    assert L.sdv2_status_string(4) == b"device wait timed out"


def test_binding_checks_tensor_device_and_extent_before_the_call():
    """The binding turns a host tensor, or one whose storage ends before the bytes an entry point
    touches, into ValueError on the host, before any C call (raw integer pointers are not
    checked: the C ABI cannot see buffer sizes)."""
    import torch
    from streaming_causal_video_gb300 import _binding as b
    assert b._row_span(0, 7, 5, 2) == 0
    assert b._row_span(3, 10, 4, 2) == (2 * 10 + 4) * 2          # last row starts 20 elements in
    with pytest.raises(ValueError, match="CUDA tensor"):
        b._dev(torch.zeros(4), "x", 16)
    assert b._dev(FAKE, "x", 1 << 40) == FAKE and b._dev(None, "x", 1) is None
    cfg = sd.StreamConfig.make(**stream_config_dict(WORKLOADS["tiny"]))
    host = torch.zeros(16)
    with pytest.raises(ValueError, match="q_rot must be a CUDA tensor"):
        sd.chunk_attention(cfg, [0], host, FAKE, FAKE, FAKE, FAKE, stream=0)
    with pytest.raises(ValueError, match="k_cache must be a CUDA tensor"):
        sd.sink_update(cfg, [0], [1], host, FAKE, FAKE, stream=0)


def test_binding_buffer_sizes_match_the_header():
    """Bytes the binding requires of each buffer, against the layouts include/sdv2.h states:
    q_rot/out [B][H][Nq][128] bf16, lse [B][H][Nq] fp32, caches and metadata per the size queries."""
    from streaming_causal_video_gb300 import _binding as b
    w = WORKLOADS["wan13b_480p"]
    cfg = sd.StreamConfig.make(**stream_config_dict(w))
    qo, cb, mb, wb, lb = b._sizes(cfg)
    assert qo == w.batch * w.heads * w.nq * 128 * 2
    assert lb == w.batch * w.heads * w.nq * 4
    assert cb == sd.cache_bytes(cfg) and mb == sd.meta_bytes(cfg) and wb == sd.workspace_bytes(cfg)


def test_next_row_entry_points_validate_on_the_host():
    """The fused projection, the re-rotation, the sink update and the noise controller reject
    bad arguments with a status and a message before touching the device."""
    c = _cfg()
    C = c.heads * 128
    args = lambda **o: dict(dict(x=FAKE, stride=0, w=FAKE, bias=None, start=[0], chunk=[0]), **o)

    def qkv(a):
        return _status(sd.qkv_rope_append, c, a["start"], a["chunk"], a["x"], a["w"], FAKE, FAKE, FAKE, FAKE, FAKE,
                       a["bias"], a["stride"], 0)
    assert qkv(args(x=FAKE + 8)) == 1                       # misaligned x
    assert qkv(args(w=None)) == 1
    assert qkv(args(stride=C - 8)) == 1                     # token stride below H*D
    assert qkv(args(stride=C + 4)) == 1                     # not a multiple of 8
    assert b"x_token_stride" in sd.lib().sdv2_last_error()
    assert qkv(args(bias=FAKE + 4)) == 1                    # bias not 16-byte aligned
    assert qkv(args(chunk=[-1])) == 1 and qkv(args(start=[-5])) == 1
    rr = _cfg(refresh_chunks=3)
    assert _status(sd.rope_refresh_rerotate, rr, [3], None, FAKE, 0) == 1
    assert _status(sd.rope_refresh_rerotate, rr, [3], FAKE, FAKE + 8, 0) == 1
    assert _status(sd.rope_refresh_rerotate, rr, [-1], FAKE, FAKE, 0) == 1
    assert b"chunk_index" in sd.lib().sdv2_last_error()
    assert _status(sd.rope_refresh_rerotate, _cfg(batch=65), [3] * 65, FAKE, FAKE, 0) == 2
    s = _cfg(sink_frames=3, window_frames=4, chunk_frames=3)
    assert _status(sd.sink_update, s, [0], [1], FAKE, FAKE, FAKE, 0) == 1      # 3 frames < 2 * sink
    assert b"2*sink_frames" in sd.lib().sdv2_last_error()
    assert _status(sd.sink_update, s, [-1], [1], FAKE, FAKE, FAKE, 0) == 1
    assert _status(sd.sink_update, s, [5], [1], None, FAKE, FAKE, 0) == 1
    sd.sink_update(s, [5], [0], FAKE, FAKE, FAKE, 0)                             # nothing to do: ok
    sd.sink_update(_cfg(sink_frames=0), [5], [1], FAKE, FAKE, FAKE, 0)          # no sink: ok
    L = sd.lib()

    def noise(ctl, B=2, T=5, m=FAKE, rate=FAKE):
        return L.sdv2_noise_from_motion(ctypes.byref(ctl), m, B, T, None, rate, None)
    good = dict(motion_lo=2.0, motion_hi=12.0, rate_lo=0.1, rate_hi=0.9, ema=0.5, more_noise_when_fast=1)
    mk = lambda **o: sd.NoiseCtl(**dict(good, **o))
    assert noise(mk(), B=0) == 1 and noise(mk(), T=0) == 1
    assert noise(mk(motion_hi=2.0)) == 1 and noise(mk(motion_lo=float("nan"))) == 1
    assert noise(mk(rate_lo=-0.1)) == 1 and noise(mk(rate_hi=float("inf"))) == 1
    assert noise(mk(ema=1.0)) == 1 and noise(mk(ema=-0.1)) == 1
    assert noise(mk(), m=FAKE + 2) == 1 and noise(mk(), rate=None) == 1
    assert noise(mk()) not in (0, 1)          # valid arguments reach the device check (no GPU here)


@pytest.mark.parametrize("items,tiles,sms,expect", [
    (228, 256, 152, (152, 2)),     # 1.3B-480p: one wave of whole items, the other 76 items in halves
    (516, 591, 152, (456, 2)),     # 1.3B-720p: three whole waves, 60 items in halves
    (760, 256, 152, (760, 1)),     # 14B-480p: exactly five waves, nothing split
    (912, 256, 152, (912, 1)),     # stream batch: six waves
    (48, 53, 152, (0, 3)),         # fewer items than SMs: every item in three key ranges (one wave)
    (2, 2, 152, (0, 2)),           # tiny: capped by the number of key tiles
    (2, 1, 152, (2, 1)),           # one key tile: nothing to split
    (153, 256, 152, (152, 4)),     # one item left over: cut four ways
])
def test_attention_schedule(items, tiles, sms, expect):
    assert sd.debug_kv_schedule(items, tiles, sms) == expect


def test_attention_schedule_never_worse_than_uniform_splits():
    """The chosen schedule's estimated makespan is at most that of the best uniform split count
    (the cost model: whole waves plus ceil(units / SMs) waves of 1/s, 2 % per split phase)."""
    import math
    for items in list(range(1, 700, 7)) + [1520, 3000]:
        for tiles in (1, 2, 3, 8, 256):
            full, s = sd.debug_kv_schedule(items, tiles, 152)
            assert 0 <= full <= items and 1 <= s <= min(4, tiles)
            assert (s == 1) == (full == items)
            cost = full / 152 + math.ceil((items - full) * s / 152) / s * (1.02 if s > 1 else 1.0)
            uni = min(math.ceil(items * u / 152) / u * (1.02 if u > 1 else 1.0) for u in range(1, min(4, tiles) + 1))
            assert cost <= uni + 1e-9, (items, tiles, full, s, cost, uni)
