"""Seeded sweep of the motion-to-noise controller against the oracle, bit for bit: random stream
counts, series lengths (longer than the kernel's 4096-value shared-memory tile), controller
parameters, both directions, smoothing on and off, and the smoothing state carried across a
random split of the series into two calls.  SDV2_SWEEP_NOISE_CONFIGS sets the number of
configurations (default 6)."""
import os

import numpy as np
import pytest
import torch

import oracle
import streaming_causal_video_gb300 as sd

pytestmark = pytest.mark.gpu

N_CONFIGS = int(os.environ.get("SDV2_SWEEP_NOISE_CONFIGS", "6"))


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


@pytest.mark.parametrize("seed", range(N_CONFIGS))
def test_random_noise_configs(seed):
    rng = np.random.default_rng(9000 + seed)
    B = int(rng.integers(1, 9))
    T = int(rng.integers(2, 10000))
    f32 = lambda x: float(np.float32(x))
    m_lo = f32(rng.uniform(0, 10))
    m_hi = f32(m_lo + rng.uniform(0.5, 30))
    r_lo, r_hi = (f32(x) for x in np.sort(rng.uniform(0, 1, 2)))
    ema = f32(0.0 if rng.random() < 0.3 else rng.uniform(0, 0.99))
    fast_more = int(rng.integers(0, 2))
    m = (rng.standard_normal((B, T)) * 10 + 8).astype(np.float32)
    ctl = sd.NoiseCtl(motion_lo=m_lo, motion_hi=m_hi, rate_lo=r_lo, rate_hi=r_hi, ema=ema,
                      more_noise_when_fast=fast_more)
    split = int(rng.integers(1, T))
    md = torch.from_numpy(m).cuda()
    state = torch.full((B,), -1.0, device="cuda")
    st_o = np.full(B, -1.0, np.float32)
    for part in (slice(0, split), slice(split, T)):
        mp = md[:, part].contiguous()
        rp = torch.empty_like(mp)
        sd.noise_from_motion(ctl, mp, rp, state)
        torch.cuda.synchronize()
        ref = oracle.noise(m[:, part], m_lo, m_hi, r_lo, r_hi, ema, fast_more, state=st_o)
        np.testing.assert_array_equal(rp.cpu().numpy(), ref)
    np.testing.assert_array_equal(state.cpu().numpy(), st_o)
