"""Seeded sweep of stream configurations through the whole path (append + attention) against the
oracle: random head counts, stream counts, grids, chunk sizes, sink and window lengths, refresh
periods and start offsets, streamed far enough to wrap the window.  Catches edge cases the
hand-picked tests miss (ragged query and key tiles, 1-4 key splits, one-frame windows)."""
import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("seed", range(12))
def test_random_stream_configs(seed):
    w = _random_workload(seed)
    ls = LockStep(w)
    n_chunks = (w.sink_frames + w.window_frames) // w.chunk_frames + 3
    for c in range(n_chunks):
        q_rot_o = ls.step([c] * w.batch)
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        rows = None if w.nq <= 300 else np.unique(np.linspace(0, w.nq - 1, 64).astype(np.int64))
        ls.check_attention(q_rot_o, rows=rows)
