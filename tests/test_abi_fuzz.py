"""Seeded fuzz of the C ABI's host logic on CPU (no kernel launches).

* Random valid configurations: the size queries equal their closed forms and the visible-token
  count equals the oracle's list model at every chunk.
* Random invalid configurations (one field broken at a time): every size query returns 0 and
  every entry point returns INVALID_ARG or UNSUPPORTED with a message, before touching memory.
"""
import numpy as np
import pytest

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS, stream_config_dict


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build_library()


FAKE = 1 << 20          # aligned, non-null; never dereferenced because validation fails first


def _random_valid(rng):
    F = int(rng.integers(1, 8))
    Fs = int(rng.integers(0, 8))
    W = int(rng.integers(F, F + 12))
    rt = 2 * int(rng.integers(0, 65))
    rh = 2 * int(rng.integers(0, (128 - rt) // 2 + 1))
    d = dict(stream_config_dict(WORKLOADS["tiny"]))
    d.update(batch=int(rng.integers(1, 17)), heads=int(rng.integers(1, 41)), rope_t=rt, rope_h=rh,
             rope_w=128 - rt - rh, grid_h=int(rng.integers(1, 60)), grid_w=int(rng.integers(1, 90)),
             chunk_frames=F, sink_frames=Fs, window_frames=W, refresh_chunks=int(rng.integers(0, 70)))
    return d


def test_random_valid_configs_sizes_and_visible_prefix():
    rng = np.random.default_rng(11)
    for _ in range(300):
        d = _random_valid(rng)
        c = sd.StreamConfig.make(**d)
        slots = d["sink_frames"] + d["window_frames"]
        hw = d["grid_h"] * d["grid_w"]
        assert sd.cache_bytes(c) == d["batch"] * d["heads"] * slots * hw * 128 * 2
        assert sd.meta_bytes(c) == d["batch"] * slots * 16
        assert sd.workspace_bytes(c) > 0
        cache = oracle.FrameListCache(d["sink_frames"], d["window_frames"])
        F = d["chunk_frames"]
        for ch in range(int(rng.integers(1, 25))):
            for i in range(F):
                cache.append(ch * F + i, 0, None, None)
            assert sd.visible_tokens(c, ch) == len(cache.frames()) * hw


BREAKS = [
    ("batch", 0), ("batch", -3), ("heads", 0), ("head_dim", 64), ("rope_t", 3), ("rope_t", -2),
    ("rope_h", 130), ("grid_h", 0), ("grid_w", -1), ("chunk_frames", 0), ("sink_frames", -1),
    ("window_frames", 0), ("refresh_chunks", -1), ("rope_base", 0.0), ("rope_base", -10.0),
    ("qkv_token_stride", 5),
]


@pytest.mark.parametrize("field,value", BREAKS)
def test_random_configs_with_one_broken_field_are_rejected(field, value):
    rng = np.random.default_rng(hash((field, str(value))) % (2 ** 32))
    for _ in range(20):
        d = _random_valid(rng)
        d[field] = value
        if field == "rope_t":                  # keep the sum at 128 so that only the broken property fails
            d["rope_h"] = 128 - value - d["rope_w"] if 128 - value - d["rope_w"] >= 0 else d["rope_h"]
        c = sd.StreamConfig.make(**d)
        assert sd.cache_bytes(c) == 0
        assert sd.meta_bytes(c) == 0
        assert sd.workspace_bytes(c) == 0
        n = max(d["batch"], 0)
        for fn, args in ((sd.rope_append_kv, ([0] * n, [0] * n) + (FAKE,) * 8 + (0,)),
                         (sd.chunk_attention, ([0] * n, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.0, 0))):
            if d["batch"] < 0:
                # the binding cannot size the per-stream arrays: it refuses before the C call
                with pytest.raises(ValueError):
                    fn(c, *args)
                continue
            with pytest.raises(sd.SDV2Error) as e:
                fn(c, *args)
            assert e.value.status in (1, 2), (field, value, e.value.status)
            assert sd.lib().sdv2_last_error(), (field, value)


@pytest.mark.parametrize("chunk", [-1, (1 << 40) + 1, (1 << 62)])
@pytest.mark.parametrize("name,batch", [("tiny", 1), ("tiny", 3), ("stream_batch", 4)])
def test_chunk_index_outside_zero_to_two_pow_40_is_rejected_everywhere(chunk, name, batch):
    """Every entry point that takes chunk indices refuses one outside [0, 2^40] before anything
    is enqueued (frame numbers c*F and the visible-prefix arithmetic stay far inside int64)."""
    import ctypes
    c = sd.StreamConfig.make(**stream_config_dict(WORKLOADS[name], batch=batch))
    L = sd.lib()
    for bad in range(batch):
        idx = [5] * batch
        idx[bad] = chunk
        arr = (ctypes.c_int64 * batch)(*idx)
        zeros = (ctypes.c_int64 * batch)(*([0] * batch))
        upd = (ctypes.c_int32 * batch)(*([1] * batch))
        calls = [
            lambda: L.sdv2_rope_append_kv(ctypes.byref(c), zeros, arr, *([FAKE] * 8), None),
            lambda: L.sdv2_chunk_attention(ctypes.byref(c), arr, FAKE, FAKE, FAKE, 0.0, FAKE, None, FAKE, None),
            lambda: L.sdv2_chunk_attention_noalloc(ctypes.byref(c), arr, FAKE, FAKE, FAKE, 0.0, FAKE, None, None),
            lambda: L.sdv2_rope_refresh_rerotate(ctypes.byref(c), arr, FAKE, FAKE, None),
            lambda: L.sdv2_sink_update(ctypes.byref(c), arr, upd, FAKE, FAKE, FAKE, None),
        ]
        for k, call in enumerate(calls):
            assert call() == 1, k
            assert b"chunk_index" in L.sdv2_last_error(), (k, L.sdv2_last_error())
