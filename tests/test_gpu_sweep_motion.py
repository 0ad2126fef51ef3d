"""Seeded sweep of the motion reduction against the oracle: random stream counts, frame counts
(runs of frame pairs with ragged ends), frame shapes and channel counts; half the cases use
uniform random pixels (large differences, near the top of the 32-bit partial sums), half the
moving-texture frames of the workloads.  SSD exact, RMS bit-exact.  SDV2_SWEEP_MOTION_CONFIGS
sets the number of configurations (default 6)."""
import os

import numpy as np
import pytest
import torch

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import motion_frames_host

pytestmark = pytest.mark.gpu

N_CONFIGS = int(os.environ.get("SDV2_SWEEP_MOTION_CONFIGS", "6"))


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


@pytest.mark.parametrize("seed", range(N_CONFIGS))
def test_random_motion_configs(seed):
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 5))
    T = int(rng.integers(1, 80))
    ch = int(rng.choice([1, 3, 4]))
    hp = int(rng.integers(1, 65))
    wp = 16 * int(rng.integers(1, 41))           # whole 16-byte vectors per frame
    if seed % 2:
        frames = torch.from_numpy(rng.integers(0, 256, (B, T + 1, hp, wp, ch), dtype=np.uint8))
    else:
        frames = motion_frames_host(B, T + 1, hp, wp, ch, seed=8000 + seed)
    ssd_ref = oracle.motion_ssd(frames.numpy())
    ssd = torch.empty((B, T), dtype=torch.int64, device="cuda")
    m = torch.empty((B, T), dtype=torch.float32, device="cuda")
    sd.motion_l2(frames.cuda(), ssd, m)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ssd.cpu().numpy().view(np.uint64), ssd_ref)
    np.testing.assert_array_equal(m.cpu().numpy(), oracle.motion_rms(ssd_ref, hp * wp * ch).astype(np.float32))
