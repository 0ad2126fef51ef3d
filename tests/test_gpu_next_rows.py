"""GPU parity of the rows built after the hot path: refresh re-rotation of the window keys,
sink update, and the motion-to-noise controller.  Cache contents and metadata bit-exact,
attention within the parity tolerance, noise rates bit-exact (fp32 with the same roundings)."""
import numpy as np
import pytest
import torch

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS, qkv_chunk_host
from gpu_common import LockStep, bits, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def _append(ls, chunks, step):
    w = ls.w
    q, k, v = qkv_chunk_host(w, w.batch, chunks[0], step=step)
    L = ls.sess.layers[0]
    sd.rope_append_kv(ls.cfg, ls.starts, chunks, q.cuda(), k.cuda(), v.cuda(), ls.sess.q_rot, L.k, L.v, L.meta,
                      ls.sess.ws)
    return [ls.oracles[b].append_chunk(chunks[b], bits(q[b]), bits(k[b]), bits(v[b])) for b in range(w.batch)]


def _attend(ls, chunks):
    L = ls.sess.layers[0]
    sd.chunk_attention(ls.cfg, chunks, ls.sess.q_rot, L.k, L.v, ls.sess.out, ls.sess.ws, lse=ls.lse)
    torch.cuda.synchronize()


@pytest.mark.parametrize("window,sink_updates", [(9, False), (9, True), (4, True)])
def test_refresh_rerotation_and_sink_update_stream(window, sink_updates):
    w = small_workload(WORKLOADS["tiny"], batch=2, heads=2, window_frames=window, refresh_chunks=3,
                       start_frames=[0, 777])
    ls = LockStep(w)
    for c in range(11):
        chunks = [c, c]
        refresh = c > 0 and c % 3 == 0
        L = ls.sess.layers[0]
        sd.rope_refresh_rerotate(ls.cfg, chunks, L.k, L.meta)
        for b in range(w.batch):
            assert ls.oracles[b].refresh_rerotate(c) == refresh
        for step in range(2 if refresh else 1):            # a second denoise step at refresh chunks
            q_rot_o = _append(ls, chunks, step)
            if refresh and sink_updates:
                sd.sink_update(ls.cfg, chunks, [1, 1], L.k, L.v, L.meta)
                for so in ls.oracles:
                    so.sink_update()
            _attend(ls, chunks)
            ls.check_q_rot(q_rot_o)
            ls.check_cache_entries_in_slots()
            ls.check_attention(q_rot_o)


def test_rerotation_leaves_other_chunks_alone():
    """Not a refresh chunk (or R = 0): the call changes nothing."""
    w = small_workload(WORKLOADS["tiny"], refresh_chunks=0)
    ls = LockStep(w)
    for c in range(4):
        ls.step([c])
    L = ls.sess.layers[0]
    before = (bits(L.k).copy(), L.meta.cpu().numpy().copy())
    for c in (3, 4, 6):
        sd.rope_refresh_rerotate(ls.cfg, [c], L.k, L.meta)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(L.k), before[0])
    np.testing.assert_array_equal(L.meta.cpu().numpy(), before[1])


@pytest.mark.parametrize("fast_more,ema", [(1, 0.0), (0, 0.0), (1, 0.6), (0, 0.9)])
def test_noise_controller_bit_exact(fast_more, ema):
    rng = np.random.default_rng(7)
    m = (rng.random((3, 50)) * 20).astype(np.float32)
    ctl = sd.NoiseCtl(motion_lo=2.0, motion_hi=12.0, rate_lo=0.1, rate_hi=0.9, ema=ema, more_noise_when_fast=fast_more)
    md = torch.from_numpy(m).cuda()
    rate = torch.empty_like(md)
    state = torch.full((3,), -1.0, device="cuda")
    st_o = np.full(3, -1.0, np.float32)
    for part in (slice(0, 20), slice(20, 50)):       # state carried across two calls
        mp = md[:, part].contiguous()
        rp = torch.empty_like(mp)
        sd.noise_from_motion(ctl, mp, rp, state)
        torch.cuda.synchronize()
        ref = oracle.noise(m[:, part], 2.0, 12.0, 0.1, 0.9, ema, fast_more, state=st_o)
        np.testing.assert_array_equal(rp.cpu().numpy(), ref)
    np.testing.assert_array_equal(state.cpu().numpy(), st_o)
