"""GPU parity: the CUDA path through the C ABI against the oracle, on seeded inputs.

Bit-exact: q_rot, the cache rows of every retained frame, the slot metadata (frame id and
RoPE time index), the untouched state of empty slots, motion SSD and RMS.
Tolerance (bf16 inputs, fp32 accumulation): attention max-abs <= 2e-2 and mean-abs <= 2e-3
against the fp64 oracle; log-sum-exp within 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS, motion_frames_host, qkv_chunk_host
from gpu_common import (LockStep, bits, config, sample_rows, small_workload, to_f64, MAX_ABS, MEAN_ABS)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    torch.cuda.init()


# ------------------------------------------------------------------------------------------
# RoPE + append alone (no tensor cores involved)
# ------------------------------------------------------------------------------------------

def test_rope_append_tiny_every_chunk_bit_exact():
    w = WORKLOADS["tiny"]
    ls = LockStep(w)
    for c in range(w.chunks):
        q_rot_o = ls.step([c])
        ls.check_q_rot(q_rot_o)
        ls.check_cache()


# ------------------------------------------------------------------------------------------
# closed forms through the whole path (one 128-key tile, one 128-row query tile)
# ------------------------------------------------------------------------------------------

PROBE = small_workload(WORKLOADS["tiny"], heads=1, grid_h=8, grid_w=16, chunk_frames=1, sink_frames=0,
                       window_frames=2, chunks=2)


def _probe_run(q, k, v, chunk=0):
    ls = LockStep(PROBE)
    for c in range(chunk + 1):
        q_rot_o = ls.step([c], qkv=(q, k, v))
    return ls, q_rot_o


def test_probe_zero_query_gives_mean_of_values():
    g = torch.Generator().manual_seed(3)
    shape = (1, PROBE.nq, 1, 128)
    q = torch.zeros(shape, dtype=torch.bfloat16)
    k = torch.randn(shape, generator=g).to(torch.bfloat16)
    v = torch.randn(shape, generator=g).to(torch.bfloat16)
    ls, q_rot_o = _probe_run(q, k, v)
    out = to_f64(ls.sess.out)[0, :, 0, :]
    mean_v = v[0, :, 0, :].double().mean(0).numpy()
    err = np.abs(out - mean_v[None, :])
    assert err.max() <= 8e-3, "uniform weights: max err %.3g (row 0: %s vs %s)" % (
        err.max(), out[0, :4], mean_v[:4])
    lse = ls.lse.cpu().numpy()[0, 0]
    np.testing.assert_allclose(lse, math.log(PROBE.hw), atol=1e-4)


def test_probe_constant_values_pass_through():
    g = torch.Generator().manual_seed(4)
    shape = (1, PROBE.nq, 1, 128)
    q = torch.randn(shape, generator=g).to(torch.bfloat16)
    k = torch.randn(shape, generator=g).to(torch.bfloat16)
    row = torch.randn((128,), generator=g).to(torch.bfloat16)
    v = row.expand(shape).contiguous()
    ls, _ = _probe_run(q, k, v)
    out = to_f64(ls.sess.out)[0, :, 0, :]
    err = np.abs(out - row.double().numpy()[None, :])
    assert err.max() <= 2e-2, "constant V: max err %.3g" % err.max()


def test_probe_one_hot_values_expose_probabilities():
    """With v_j = e_j (128 keys, 128 dims) the output row is the softmax row itself."""
    g = torch.Generator().manual_seed(5)
    shape = (1, PROBE.nq, 1, 128)
    q = torch.randn(shape, generator=g).to(torch.bfloat16)
    k = torch.randn(shape, generator=g).to(torch.bfloat16)
    v = torch.eye(128).reshape(1, 128, 1, 128).to(torch.bfloat16)
    ls, q_rot_o = _probe_run(q, k, v)
    out = to_f64(ls.sess.out)[0, :, 0, :]
    ref, _ = ls.oracles[0].attend(q_rot_o[0], 0)
    err = np.abs(out - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, "P rows: max %.3g mean %.3g" % (err.max(), err.mean())


def test_probe_two_kv_tiles():
    g = torch.Generator().manual_seed(6)
    shape = (1, PROBE.nq, 1, 128)
    ls = LockStep(PROBE)
    for c in range(2):
        q, k, v = (torch.randn(shape, generator=g).to(torch.bfloat16) for _ in range(3))
        q_rot_o = ls.step([c], qkv=(q, k, v))
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o)


# ------------------------------------------------------------------------------------------
# whole streams
# ------------------------------------------------------------------------------------------

def test_tiny_stream_full_parity():
    w = WORKLOADS["tiny"]
    ls = LockStep(w)
    for c in range(w.chunks):
        q_rot_o = ls.step([c])
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o)


def test_two_streams_refresh_reappend_and_ragged_tiles():
    """Ragged sizes (35 tokens per frame, 105 queries, 175 keys in the window) with a sink of two
    frames, a refresh every 3 chunks, distinct start offsets, stream 0 re-appending a chunk (a
    second denoise step) while stream 1 moves on."""
    w = small_workload(WORKLOADS["tiny"], batch=2, heads=3, grid_h=5, grid_w=7, chunk_frames=3,
                       sink_frames=2, window_frames=5, refresh_chunks=3, start_frames=[0, 1000])
    ls = LockStep(w)
    schedule = [[0, 0], [1, 1], [1, 2], [2, 3], [3, 3], [4, 4], [5, 5], [6, 6], [7, 7]]
    for chunks in schedule:
        q_rot_o = ls.step(chunks)
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o)


@pytest.mark.parametrize("over", [
    dict(sink_frames=0, window_frames=3),                      # no sink, window = one chunk
    dict(grid_h=1, grid_w=1, chunk_frames=2, window_frames=2, sink_frames=1),  # one token per frame
    dict(chunk_frames=1, sink_frames=0, window_frames=1),      # each chunk attends to itself only
    dict(grid_h=16, grid_w=16, chunk_frames=1, sink_frames=1, window_frames=2),   # exact 256-row tiles
])
def test_degenerate_configs(over):
    w = small_workload(WORKLOADS["tiny"], chunks=5, **over)
    ls = LockStep(w)
    for c in range(w.chunks):
        q_rot_o = ls.step([c])
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o)


def test_sixteen_streams_maximum_batch():
    w = small_workload(WORKLOADS["tiny"], batch=16, heads=1, start_frames=[i * 37 for i in range(16)],
                       refresh_chunks=2)
    ls = LockStep(w)
    for c in range(4):
        q_rot_o = ls.step([c] * 16)
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o)


def test_stream_batch_shape_reduced_grid_across_refreshes():
    """The stream-batch workload's cache and refresh settings (F=3, sink 3, window 18, R=64,
    offsets 0, 1e3, 1e4, 1e5) on a small grid, streamed for 130 chunks; checked around the start,
    the first window wrap and both refreshes."""
    base = WORKLOADS["stream_batch"]
    w = small_workload(base, heads=2, grid_h=6, grid_w=8, chunks=130)
    ls = LockStep(w)
    check = set(range(0, 9)) | set(range(62, 67)) | set(range(126, 130))
    for c in range(w.chunks):
        q_rot_o = ls.step([c] * w.batch)
        if c in check:
            ls.check_q_rot(q_rot_o)
            ls.check_cache()
            ls.check_attention(q_rot_o, rows=sample_rows(w.nq, 40, c))


def test_packed_qkv_token_stride_matches_separate_tensors():
    w = small_workload(WORKLOADS["tiny"], heads=3)
    q, k, v = qkv_chunk_host(w, 1, 0)
    packed = torch.stack([q, k, v], dim=2).cuda()             # [B][Nq][3][H][D]
    cfg_p = config(w, qkv_token_stride=3 * w.heads * 128)
    cfg_s = config(w)
    outs = []
    for cfg, (qa, ka, va) in ((cfg_s, (q.cuda(), k.cuda(), v.cuda())),
                              (cfg_p, (packed[:, :, 0], packed[:, :, 1], packed[:, :, 2]))):
        sess = sd.StreamSession(cfg, 1, [5], "cuda")
        sess.layer_step(0, [0], qa, ka, va)
        torch.cuda.synchronize()
        outs.append((bits(sess.q_rot), bits(sess.layers[0].k), bits(sess.out)))
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


def test_repeated_call_is_deterministic():
    w = WORKLOADS["tiny"]
    cfg = config(w)
    sess = sd.StreamSession(cfg, 1, [0], "cuda")
    q, k, v = (t.cuda() for t in qkv_chunk_host(w, 1, 3))
    for c in range(4):
        sess.layer_step(0, [c], q, k, v)
    torch.cuda.synchronize()
    a = bits(sess.out).copy()
    sess.layer_step(0, [3], q, k, v)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(sess.out), a)
    sd.check_device_error(sess.ws)


@pytest.mark.parametrize("chunk_stop", [3, 8])
def test_forced_kv_splits_all_match_oracle(chunk_stop):
    """The same cached state attended with 1, 2, 3 and 4 key splits (the split that finishes
    last merges the others' partial rows): every result matches the oracle."""
    w = small_workload(WORKLOADS["wan13b_480p"], heads=2, grid_h=10, grid_w=16, chunks=chunk_stop)
    ls = LockStep(w)
    for c in range(chunk_stop):
        q_rot_o = ls.step([c])
    rows = sample_rows(w.nq, 48, 11)
    try:
        for splits in (1, 2, 3, 4):
            sd.debug_set_kv_splits(splits)
            L = ls.sess.layers[0]
            sd.chunk_attention(ls.cfg, [chunk_stop - 1], ls.sess.q_rot, L.k, L.v, ls.sess.out, ls.sess.ws,
                               lse=ls.lse)
            torch.cuda.synchronize()
            assert sd.last_kv_splits() == splits
            ls.check_attention(q_rot_o, rows=rows)
        sd.check_device_error(ls.sess.ws)
    finally:
        sd.debug_set_kv_splits(0)


GROW = small_workload(WORKLOADS["tiny"], heads=2, grid_h=8, grid_w=16, chunk_frames=1, sink_frames=1,
                      window_frames=3, chunks=4)


def test_scores_growing_across_key_tiles():
    """Each later frame's keys are scaled up (x0.05, x1, x4, x16), so the running row max jumps
    by far more than the lazy-rescale threshold from one 128-key tile to the next; a third of the
    query rows are scaled down so that only some rows of a warp jump.  Every result matches the
    oracle with 1, 2 and 3 key splits."""
    w = GROW
    g = torch.Generator().manual_seed(21)
    shape = (1, w.nq, w.heads, 128)
    row_scale = torch.where(torch.arange(w.nq) % 3 == 0, 0.02, 1.0).reshape(1, w.nq, 1, 1)
    ls = LockStep(w)
    for c, ks in enumerate((0.05, 1.0, 4.0, 16.0)):
        q = (torch.randn(shape, generator=g) * row_scale).to(torch.bfloat16)
        k = (torch.randn(shape, generator=g) * ks).to(torch.bfloat16)
        v = torch.randn(shape, generator=g).to(torch.bfloat16)
        q_rot_o = ls.step([c], qkv=(q, k, v))
        ls.check_attention(q_rot_o)
    try:
        for splits in (1, 2, 3):
            sd.debug_set_kv_splits(splits)
            L = ls.sess.layers[0]
            sd.chunk_attention(ls.cfg, [w.chunks - 1], ls.sess.q_rot, L.k, L.v, ls.sess.out, ls.sess.ws,
                               lse=ls.lse)
            torch.cuda.synchronize()
            assert sd.last_kv_splits() == splits
            ls.check_attention(q_rot_o)
        sd.check_device_error(ls.sess.ws)
    finally:
        sd.debug_set_kv_splits(0)


# ------------------------------------------------------------------------------------------
# full workload shapes, in the launch configuration the bench times (sampled rows)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name,chunks,rows_per_head,heads", [
    ("wan13b_480p", 8, 24, None),
    ("wan13b_720p", 8, 10, [0, 5, 11]),
    ("wan14b_480p", 8, 8, [0, 13, 39]),
])
def test_full_shape_streams_sampled(name, chunks, rows_per_head, heads):
    w = WORKLOADS[name]
    ls = LockStep(w)
    for c in range(chunks):
        q_rot_o = ls.step([c])
        ls.check_q_rot(q_rot_o)
        hw_frames = set(range(c * w.chunk_frames, (c + 1) * w.chunk_frames))
        ls.check_cache(only_frames=hw_frames)
        if c in (0, 1, 6, 7):
            ls.check_attention(q_rot_o, rows=sample_rows(w.nq, rows_per_head, 100 + c), heads=heads)


def test_stream_batch_full_shape_identical_streams_shift_invariance():
    """Four streams with identical q, k, v at offsets 0, 1e3, 1e4, 1e5: each matches the oracle,
    and the outputs agree with each other (only relative positions matter)."""
    w = WORKLOADS["stream_batch"]
    ls = LockStep(w)
    rows = sample_rows(w.nq, 16, 7)
    for c in range(3):
        q_rot_o = ls.step([c] * 4, same_streams=True)
        ls.check_q_rot(q_rot_o)
        ls.check_cache()
        ls.check_attention(q_rot_o, rows=rows, heads=[0, 7])
    out = to_f64(ls.sess.out)
    for b in range(1, 4):
        err = np.abs(out[b] - out[0])
        assert err.max() <= 2 * MAX_ABS and err.mean() <= 2 * MEAN_ABS


@pytest.mark.parametrize("rerotate", [False, True])
def test_stream_batch_full_shape_through_the_first_refresh(rerotate):
    """The stream-batch workload at its own shape (4 streams, 12 heads, 30x52 tokens per frame,
    chunks of 3 frames, sink 3 + window 18, RoPE refresh every 64 chunks, start offsets 0, 1e3,
    1e4, 1e5), one layer streamed through chunks 0-66: the first chunks, the first window wrap and
    the chunks around the refresh at 64 are checked -- q_rot, every retained frame's K/V rows and
    all slot metadata bit-exact, attention on sampled rows of two heads.  With rerotate the
    window keys are turned back by F*R at the refresh chunk (second reading of the refresh)
    before its first append, on both sides."""
    w = WORKLOADS["stream_batch"]
    ls = LockStep(w)
    L = ls.sess.layers[0]
    check = {0, 6, 7, 62, 63, 64, 65, 66}
    for c in range(67):
        if rerotate:
            sd.rope_refresh_rerotate(ls.cfg, [c] * w.batch, L.k, L.meta)
            torch.cuda.synchronize()
            refresh = [o.refresh_rerotate(c) for o in ls.oracles]
            assert all(refresh) == (c == 64) and any(refresh) == (c == 64)
        q_rot_o = ls.step([c] * w.batch)
        if c in check:
            ls.check_q_rot(q_rot_o)
            ls.check_cache()
            ls.check_attention(q_rot_o, rows=sample_rows(w.nq, 20, 300 + c), heads=[0, 11])
            if c == 64:
                meta = L.meta.cpu().numpy()
                for b, s0 in enumerate(w.start_frames):
                    # the new chunk's frames restart at the stream's own start frame
                    assert {int(meta[b, oracle.slot_of_frame(64 * 3 + i, 3, 18), 1]) for i in range(3)} == \
                        {s0, s0 + 1, s0 + 2}


# ------------------------------------------------------------------------------------------
# motion
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,T,hp,wp,ch", [
    (1, 1, 1, 16, 1),          # smallest frame, one pair
    (2, 5, 48, 64, 3),
    (1, 33, 20, 24, 3),        # crosses a 32-frame run
    (3, 65, 16, 20, 3),
    (2, 20, 480, 832, 3),      # the 480p frame
    (2, 140, 480, 832, 3),     # long runs of 32 frame pairs and a ragged last run
])
def test_motion_exact(B, T, hp, wp, ch):
    frames = motion_frames_host(B, T + 1, hp, wp, ch, seed=B * 100 + T)
    ssd_ref = oracle.motion_ssd(frames.numpy())
    fd = frames.cuda()
    ssd = torch.empty((B, T), dtype=torch.int64, device="cuda")
    m = torch.empty((B, T), dtype=torch.float32, device="cuda")
    sd.motion_l2(fd, ssd, m)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ssd.cpu().numpy().view(np.uint64), ssd_ref)
    m_ref = oracle.motion_rms(ssd_ref, hp * wp * ch).astype(np.float32)
    np.testing.assert_array_equal(m.cpu().numpy(), m_ref)


@pytest.mark.parametrize("R", [0, 7])
def test_append_at_a_very_large_chunk_index(R):
    """A stream a million chunks in (time indices of several million, cache frame numbers past
    3e6): q_rot and the slot rows equal the oracle's bit-exact RoPE at the oracle's positions,
    and the slot metadata names the right frame and time index."""
    w = small_workload(WORKLOADS["tiny"], batch=2, heads=2, refresh_chunks=R, start_frames=[100000, 7])
    cfg = config(w)
    sess = sd.StreamSession(cfg, 1, w.start_frames, "cuda")
    L = sess.layers[0]
    c = 1_000_003
    q, k, v = qkv_chunk_host(w, w.batch, 3)
    sd.rope_append_kv(cfg, w.start_frames, [c, c], q.cuda(), k.cuda(), v.cuda(), sess.q_rot, L.k, L.v, L.meta,
                      sess.ws)
    torch.cuda.synchronize()
    qg, kg, vg, meta = bits(sess.q_rot), bits(L.k), bits(L.v), L.meta.cpu().numpy()
    hw = w.hw
    for b in range(w.batch):
        t, h, ww, frame = oracle.chunk_positions(w.start_frames[b], c, w.chunk_frames, w.grid_h, w.grid_w, R)
        rep = lambda a: np.repeat(a, w.heads)
        qo = oracle.rope_spec(bits(q[b]).reshape(-1, 128), rep(t), rep(h), rep(ww), w.rope_t, w.rope_h, w.rope_w,
                              w.rope_base).reshape(w.nq, w.heads, 128)
        ko = oracle.rope_spec(bits(k[b]).reshape(-1, 128), rep(t), rep(h), rep(ww), w.rope_t, w.rope_h, w.rope_w,
                              w.rope_base).reshape(w.nq, w.heads, 128)
        np.testing.assert_array_equal(qg[b].transpose(1, 0, 2), qo)
        for i in range(w.chunk_frames):
            f = int(frame[i * hw])
            s = oracle.slot_of_frame(f, w.sink_frames, w.window_frames)
            assert tuple(meta[b, s]) == (f, int(t[i * hw]))
            np.testing.assert_array_equal(kg[b][:, s * hw:(s + 1) * hw, :], ko[i * hw:(i + 1) * hw].transpose(1, 0, 2))
            np.testing.assert_array_equal(vg[b][:, s * hw:(s + 1) * hw, :], bits(v[b])[i * hw:(i + 1) * hw].transpose(1, 0, 2))
