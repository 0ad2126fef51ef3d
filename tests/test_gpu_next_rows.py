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


@pytest.mark.parametrize("window,sink_updates,rope", [(9, False, (44, 42, 42)), (9, True, (44, 42, 42)),
                                                     (4, True, (44, 42, 42)),
                                                     # a time axis of 72 dims spans 9 of a row's 16-byte vectors
                                                     (9, True, (72, 28, 28))])
def test_refresh_rerotation_and_sink_update_stream(window, sink_updates, rope):
    w = small_workload(WORKLOADS["tiny"], batch=2, heads=2, window_frames=window, refresh_chunks=3,
                       start_frames=[0, 777], rope_t=rope[0], rope_h=rope[1], rope_w=rope[2])
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


# ------------------------------------------------------------------------------------------
# fused QKV projection + Causal-RoPE + cache append
# ------------------------------------------------------------------------------------------

import math  # noqa: E402

from gpu_common import config, to_f64, MAX_ABS, MEAN_ABS  # noqa: E402


def _proj_inputs(w, c, seed=0):
    C = w.heads * w.head_dim
    g = torch.Generator().manual_seed(1000 * seed + c)
    x = torch.randn((w.batch, w.nq, C), generator=g).to(torch.bfloat16)
    W = (torch.randn((3 * C, C), generator=g) / math.sqrt(C)).to(torch.bfloat16)
    bias = (torch.randn(3 * C, generator=g) * 0.1).float()
    return x, W, bias


def _close(got, ref, what):
    """bf16 outputs against fp64: each element within 2^-8 of its rotation pair's norm (one bf16
    rounding of a value no larger than that norm, plus fp32 accumulation error far below it)."""
    pn = np.repeat(np.hypot(ref[..., 0::2], ref[..., 1::2]), 2, axis=-1)
    err = np.abs(got - ref)
    bad = err > 2.0 ** -8 * pn + 1e-6
    assert not bad.any(), "%s: %d elements off, worst %.3g (pair norm %.3g)" % (
        what, int(bad.sum()), float(err[bad].max()), float(pn[bad][np.argmax(err[bad])]))


def _fused_reference(w, start, c, x_b, W, bias):
    C = w.heads * w.head_dim
    y = oracle.qkv_project(bits(x_b), bits(W), bias.numpy())          # [Nq][3C]
    t, h, ww, frame = oracle.chunk_positions(start, c, w.chunk_frames, w.grid_h, w.grid_w, w.refresh_chunks)
    rep = lambda a: np.repeat(a.astype(np.float64), w.heads)
    rot = lambda z: oracle.rope_ideal(z.reshape(-1, w.head_dim), rep(t), rep(h), rep(ww), w.rope_t, w.rope_h,
                                      w.rope_w, w.rope_base).reshape(w.nq, w.heads, w.head_dim)
    q = rot(y[:, :C])
    k = rot(y[:, C:2 * C])
    v = y[:, 2 * C:].reshape(w.nq, w.heads, w.head_dim)
    return q, k, v, t, frame


@pytest.mark.parametrize("name,over,chunks,attend", [
    ("tiny", dict(heads=2, window_frames=4, refresh_chunks=3, batch=2, start_frames=[0, 500]), 7, True),
    # odd head count: 192-feature tiles straddle heads and the q|k|v boundaries; 405 tokens per
    # stream leave a ragged 256-token tile
    ("tiny", dict(heads=3, grid_h=9, grid_w=15, window_frames=5, refresh_chunks=2, batch=2,
                  start_frames=[7, 90000]), 4, True),
    ("wan13b_480p", dict(), 2, False),
    # cos/sin tables too large for the kernel's shared-memory copy (30 h and 30 w pairs over a
    # 40 x 80 grid: 28.8 KB): the epilogue reads them from global memory
    ("tiny", dict(heads=2, grid_h=40, grid_w=80, chunk_frames=1, sink_frames=1, window_frames=2,
                  rope_t=8, rope_h=60, rope_w=60, start_frames=[11]), 3, False),
])
def test_fused_qkv_rope_append_matches_fp64(name, over, chunks, attend):
    w = small_workload(WORKLOADS[name], **over)
    cfg = config(w)
    starts = list(w.start_frames)
    sess = sd.StreamSession(cfg, 1, starts, "cuda")
    L = sess.layers[0]
    hw = w.hw
    kept = [{} for _ in range(w.batch)]        # per stream: frame -> (k_ref, v_ref) of retained frames
    for c in range(chunks):
        x, W, bias = _proj_inputs(w, c)
        sd.qkv_rope_append(cfg, starts, [c] * w.batch, x.cuda(), W.cuda(), sess.q_rot, L.k, L.v, L.meta, sess.ws,
                           bias=bias.cuda())
        torch.cuda.synchronize()
        qg = to_f64(sess.q_rot)                  # [B][H][Nq][D]
        kg, vg = to_f64(L.k), to_f64(L.v)        # [B][H][rows][D]
        meta = L.meta.cpu().numpy()
        refs = []
        for b in range(w.batch):
            q, k, v, t, frame = _fused_reference(w, starts[b], c, x[b], W, bias)
            refs.append(q)
            _close(qg[b].transpose(1, 0, 2), q, "q_rot stream %d" % b)
            for i in range(w.chunk_frames):
                f = c * w.chunk_frames + i
                s = oracle.slot_of_frame(f, w.sink_frames, w.window_frames)
                assert tuple(meta[b, s]) == (f, int(t[i * hw])), (b, s, tuple(meta[b, s]))
                _close(kg[b][:, s * hw:(s + 1) * hw, :].transpose(1, 0, 2), k[i * hw:(i + 1) * hw], "k slot %d" % s)
                _close(vg[b][:, s * hw:(s + 1) * hw, :].transpose(1, 0, 2), v[i * hw:(i + 1) * hw], "v slot %d" % s)
                kept[b][f] = (k[i * hw:(i + 1) * hw], v[i * hw:(i + 1) * hw])
        if attend:
            lse = torch.empty((w.batch, w.heads, w.nq), dtype=torch.float32, device="cuda")
            sd.chunk_attention(cfg, [c] * w.batch, sess.q_rot, L.k, L.v, sess.out, sess.ws, lse=lse)
            torch.cuda.synchronize()
            out = to_f64(sess.out)
            for b in range(w.batch):
                n = (c + 1) * w.chunk_frames
                fr = list(range(min(w.sink_frames, n))) + \
                    [f for f in range(w.sink_frames, n)][-w.window_frames:]
                for hh in range(w.heads):
                    K = np.concatenate([kept[b][f][0][:, hh, :] for f in fr])
                    V = np.concatenate([kept[b][f][1][:, hh, :] for f in fr])
                    ref, _ = oracle.attention_f64(refs[b][:, hh, :], K, V, 1 / math.sqrt(w.head_dim))
                    err = np.abs(out[b, :, hh, :] - ref)
                    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (c, b, hh, err.max(), err.mean())


@pytest.mark.parametrize("name", ["wan14b_480p", "wan13b_720p", "stream_batch"])
def test_fused_qkv_rope_append_at_full_shape_sampled_rows(name):
    """Full workload shapes, sampled token rows of every stream's q_rot, k and v against the fp64
    projection + RoPE of those rows: Wan-14B 480p (40 heads, C = 5120, 80 feature tiles of 192,
    19 token tiles of 256); Wan-1.3B 720p (10800 tokens; its cos/sin tables, 21.5 KB, just fit
    the kernel's shared-memory copy); the 4-stream batch (tokens of four streams in the token
    tiles, start frames up to 1e5)."""
    w = WORKLOADS[name]
    cfg = config(w)
    starts = list(w.start_frames)
    sess = sd.StreamSession(cfg, 1, starts, "cuda")
    L = sess.layers[0]
    C = w.heads * w.head_dim
    c = 9                                           # window already wrapped: slots != frames
    x, W, bias = _proj_inputs(w, c, seed=3)
    sd.qkv_rope_append(cfg, starts, [c] * w.batch, x.cuda(), W.cuda(), sess.q_rot, L.k, L.v, L.meta, sess.ws,
                       bias=bias.cuda())
    torch.cuda.synchronize()
    sd.check_device_error(sess.ws)
    hw = w.hw
    rows = np.unique(np.concatenate([np.arange(0, 4), np.linspace(0, w.nq - 1, 60).astype(np.int64),
                                     np.arange(w.nq - 4, w.nq), np.arange(255, 258), np.arange(hw - 1, hw + 2)]))
    for b in range(w.batch):
        y = oracle.qkv_project(bits(x[b][torch.from_numpy(rows)].contiguous()), bits(W), bias.numpy())
        t, h, ww, frame = oracle.chunk_positions(starts[b], c, w.chunk_frames, w.grid_h, w.grid_w, w.refresh_chunks)
        rep = lambda a: np.repeat(a[rows].astype(np.float64), w.heads)
        rot = lambda z: oracle.rope_ideal(z.reshape(-1, w.head_dim), rep(t), rep(h), rep(ww), w.rope_t, w.rope_h,
                                          w.rope_w, w.rope_base).reshape(len(rows), w.heads, w.head_dim)
        q, k = rot(y[:, :C]), rot(y[:, C:2 * C])
        v = y[:, 2 * C:].reshape(len(rows), w.heads, w.head_dim)
        qg = to_f64(sess.q_rot[b][:, torch.from_numpy(rows).cuda()])        # [H][rows][D]
        _close(qg.transpose(1, 0, 2), q, "q_rot stream %d" % b)
        meta = L.meta.cpu().numpy()[b]
        slot_rows = []
        for n in rows:
            f = c * w.chunk_frames + int(n) // hw
            s = oracle.slot_of_frame(f, w.sink_frames, w.window_frames)
            assert tuple(meta[s]) == (f, int(t[(int(n) // hw) * hw])), (b, n, s, tuple(meta[s]))
            slot_rows.append(s * hw + int(n) % hw)
        idx = torch.tensor(slot_rows, device="cuda")
        _close(to_f64(L.k[b][:, idx]).transpose(1, 0, 2), k, "k rows stream %d" % b)
        _close(to_f64(L.v[b][:, idx]).transpose(1, 0, 2), v, "v rows stream %d" % b)
