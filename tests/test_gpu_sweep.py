"""Seeded sweep of stream configurations through the whole path (append + attention) against the
oracle: random head counts, stream counts, grids, chunk sizes, sink and window lengths, refresh
periods and start offsets, streamed far enough to wrap the window.  Catches edge cases the
hand-picked tests miss (ragged query and key tiles, 1-4 key splits, one-frame windows).  After
the stream, the last chunk's attention is computed again with a randomly forced split count.
SDV2_SWEEP_CONFIGS sets the number of configurations (default 12)."""
import os

import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS
from gpu_common import LockStep, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def _random_workload(seed):
    rng = np.random.default_rng(1000 + seed)
    F = int(rng.integers(1, 4))
    Fs = int(rng.integers(0, 4))
    W = int(rng.integers(F, F + 6))
    B = int(rng.choice([1, 2, 3, 5]))
    big = seed % 3 == 2          # every third configuration: several query tiles and key tiles
    gh = int(rng.integers(8, 24)) if big else int(rng.integers(1, 12))
    gw = int(rng.integers(10, 30)) if big else int(rng.integers(1, 14))
    return small_workload(WORKLOADS["tiny"], batch=B, heads=int(rng.choice([1, 2, 3, 4])),
                          grid_h=gh, grid_w=gw, chunk_frames=F,
                          sink_frames=Fs, window_frames=W, refresh_chunks=int(rng.choice([0, 2, 5])),
                          start_frames=[int(x) for x in rng.integers(0, 120000, B)], seed=50 + seed)


N_CONFIGS = int(os.environ.get("SDV2_SWEEP_CONFIGS", "12"))


@pytest.mark.parametrize("seed", range(N_CONFIGS))
def test_random_stream_configs(seed):
    w = _random_workload(seed)
    ls = LockStep(w)
    n_chunks = (w.sink_frames + w.window_frames) // w.chunk_frames + 3
    rows = None if w.nq <= 300 else np.unique(np.linspace(0, w.nq - 1, 64).astype(np.int64))
    for c in range(n_chunks):
        q_rot_o = ls.step([c] * w.batch)
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o, rows=rows)
    splits = int(np.random.default_rng(2000 + seed).integers(1, 5))
    try:
        sd.debug_set_kv_splits(splits)
        L = ls.sess.layers[0]
        sd.chunk_attention(ls.cfg, [n_chunks - 1] * w.batch, ls.sess.q_rot, L.k, L.v, ls.sess.out, ls.sess.ws,
                           lse=ls.lse)
        torch.cuda.synchronize()
        ls.check_attention(q_rot_o, rows=rows)
        sd.check_device_error(ls.sess.ws)
    finally:
        sd.debug_set_kv_splits(0)
