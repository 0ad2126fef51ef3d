"""Seeded sweep of the cache-maintenance rows against the oracle: random RoPE splits (time axes
from 0 to all 128 dims), grids, chunk sizes, sink and window lengths, refresh periods and start
offsets.  Every chunk: re-rotation at refresh chunks, append, a sink update on random streams at
some refresh chunks, attention; then bit-exact q_rot, cache rows and metadata (sink copies
included) and attention within tolerance.  SDV2_SWEEP_NEXT_CONFIGS sets the number of
configurations (default 8)."""
import os

import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS
from gpu_common import LockStep, small_workload
from test_gpu_next_rows import _append, _attend

pytestmark = pytest.mark.gpu

N_CONFIGS = int(os.environ.get("SDV2_SWEEP_NEXT_CONFIGS", "8"))


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def _random_workload(seed):
    rng = np.random.default_rng(3000 + seed)
    F = int(rng.integers(1, 4))
    Fs = int(rng.integers(0, 4))
    W = int(rng.integers(max(F, Fs), max(F, Fs) + 6))
    B = int(rng.choice([1, 2, 3]))
    rt = int(rng.choice([0, 8, 20, 44, 72, 100, 128]))
    rh = 2 * int(rng.integers(0, (128 - rt) // 2 + 1))
    rw = 128 - rt - rh
    big = seed % 4 == 3
    gh = int(rng.integers(6, 20)) if big else int(rng.integers(1, 9))
    gw = int(rng.integers(8, 24)) if big else int(rng.integers(1, 11))
    return small_workload(WORKLOADS["tiny"], batch=B, heads=int(rng.choice([1, 2, 3])), grid_h=gh, grid_w=gw,
                          chunk_frames=F, sink_frames=Fs, window_frames=W, refresh_chunks=int(rng.choice([2, 3, 5])),
                          rope_t=rt, rope_h=rh, rope_w=rw,
                          start_frames=[int(x) for x in rng.integers(0, 120000, B)], seed=70 + seed)


@pytest.mark.parametrize("seed", range(N_CONFIGS))
def test_random_refresh_and_sink_configs(seed):
    w = _random_workload(seed)
    rng = np.random.default_rng(4000 + seed)
    ls = LockStep(w)
    L = ls.sess.layers[0]
    R = w.refresh_chunks
    n_chunks = (w.sink_frames + w.window_frames) // w.chunk_frames + 2 * R + 2
    rows = None if w.nq <= 300 else np.unique(np.linspace(0, w.nq - 1, 48).astype(np.int64))
    for c in range(n_chunks):
        chunks = [c] * w.batch
        sd.rope_refresh_rerotate(ls.cfg, chunks, L.k, L.meta)
        refresh = c > 0 and c % R == 0
        for so in ls.oracles:
            assert so.refresh_rerotate(c) == refresh
        q_rot_o = _append(ls, chunks, 0)
        if (refresh and w.sink_frames > 0 and (c + 1) * w.chunk_frames >= 2 * w.sink_frames
                and rng.random() < 0.6):
            flags = [int(x) for x in rng.integers(0, 2, w.batch)]
            sd.sink_update(ls.cfg, chunks, flags, L.k, L.v, L.meta)
            for b, f in enumerate(flags):
                if f:
                    ls.oracles[b].sink_update()
        _attend(ls, chunks)
        ls.check_q_rot(q_rot_o)
        ls.check_cache_entries_in_slots()
        ls.check_attention(q_rot_o, rows=rows)
    sd.check_device_error(ls.sess.ws)
