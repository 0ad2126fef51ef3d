"""Robustness of the CUDA path: checkpoint/resume of the stream state, guard bands around
every buffer a call writes, and CUDA-graph capture of the per-layer calls."""
import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS, qkv_chunk_host
from gpu_common import bits, config, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


W = small_workload(WORKLOADS["tiny"], batch=2, heads=2, grid_h=5, grid_w=7, window_frames=5, sink_frames=2,
                   refresh_chunks=4, start_frames=[3, 9000])


def _inputs(c):
    return tuple(t.cuda() for t in qkv_chunk_host(W, W.batch, c, seed_offset=5))


def test_checkpoint_resume_is_bit_exact():
    """The stream state is the cache, its metadata and (S, c): restoring a snapshot into a fresh
    session and continuing gives the same outputs as never stopping."""
    cfg = config(W)
    a = sd.StreamSession(cfg, 1, W.start_frames, "cuda")
    outs_a = []
    snap = None
    for c in range(9):
        a.layer_step(0, [c, c], *_inputs(c))
        if c == 4:
            L = a.layers[0]
            snap = (L.k.clone(), L.v.clone(), L.meta.clone())
        if c > 4:
            outs_a.append(bits(a.out).copy())
    b = sd.StreamSession(cfg, 1, W.start_frames, "cuda")
    Lb = b.layers[0]
    Lb.k.copy_(snap[0]); Lb.v.copy_(snap[1]); Lb.meta.copy_(snap[2])
    for i, c in enumerate(range(5, 9)):
        b.layer_step(0, [c, c], *_inputs(c))
        np.testing.assert_array_equal(bits(b.out), outs_a[i])
    np.testing.assert_array_equal(bits(Lb.k), bits(a.layers[0].k))
    np.testing.assert_array_equal(Lb.meta.cpu().numpy(), a.layers[0].meta.cpu().numpy())


def _guarded(shape, dtype, fill):
    """A tensor view with a canary band of 4096 bytes on both sides."""
    pad = 4096 // torch.tensor([], dtype=dtype).element_size()
    n = int(np.prod(shape))
    base = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return base, base[pad:pad + n].view(shape), pad


def test_guard_bands_stay_untouched():
    cfg = config(W)
    B, H, nq, D = W.batch, W.heads, W.nq, 128
    rows = W.slots * W.hw
    ws_b, ws, wp = _guarded((sd.workspace_bytes(cfg),), torch.uint8, 0xA5)
    ws.zero_()
    sd.workspace_init(cfg, ws)
    bufs = {}
    for name, shape in (("q_rot", (B, H, nq, D)), ("k", (B, H, rows, D)), ("v", (B, H, rows, D)),
                        ("out", (B, nq, H, D))):
        bufs[name] = _guarded(shape, torch.int16, 0x5A5A)
    meta_b, meta, mp = _guarded((B, W.slots, 2), torch.int64, 0x1234567890)
    lse_b, lse, lp = _guarded((B, H, nq), torch.float32, 7.25)
    sd.cache_reset(cfg, bufs["k"][1], bufs["v"][1], meta)
    frames_b, frames, fp_ = _guarded((2, 5, 16, 32, 3), torch.uint8, 0x33)
    frames.copy_(torch.randint(0, 256, frames.shape, dtype=torch.uint8, device="cuda"))
    ssd_b, ssd, sp = _guarded((2, 4), torch.int64, 0x77)
    m_b, m, mp2 = _guarded((2, 4), torch.float32, 3.5)
    for c in range(6):
        q, k, v = _inputs(c)
        sd.rope_append_kv(cfg, W.start_frames, [c, c], q, k, v, bufs["q_rot"][1], bufs["k"][1], bufs["v"][1], meta, ws)
        sd.chunk_attention(cfg, [c, c], bufs["q_rot"][1], bufs["k"][1], bufs["v"][1], bufs["out"][1], ws, lse=lse)
        if c % 4 == 0 and c > 0:
            sd.rope_refresh_rerotate(cfg, [c, c], bufs["k"][1], meta)
            sd.sink_update(cfg, [c, c], [1, 1], bufs["k"][1], bufs["v"][1], meta)
    # the fused projection (reads x, W and bias; writes q_rot, the chunk's cache rows and meta),
    # the allocation-free attention (writes out and lse) and the noise controller (rate, state)
    C = H * D
    g = torch.Generator(device="cuda").manual_seed(11)
    x_b, x, xp = _guarded((B, nq, C), torch.bfloat16, 0.5)
    x.copy_(torch.randn((B, nq, C), generator=g, device="cuda").to(torch.bfloat16))
    wq_b, wq, wqp = _guarded((3 * C, C), torch.bfloat16, -0.25)
    wq.copy_((torch.randn((3 * C, C), generator=g, device="cuda") / C ** 0.5).to(torch.bfloat16))
    bias_b, bias, bp = _guarded((3 * C,), torch.float32, 1.5)
    bias.copy_(torch.randn(3 * C, generator=g, device="cuda") * 0.1)
    sd.qkv_rope_append(cfg, W.start_frames, [6, 6], x, wq, bufs["q_rot"][1], bufs["k"][1], bufs["v"][1], meta, ws,
                       bias=bias)
    sd.chunk_attention_noalloc(cfg, [6, 6], bufs["q_rot"][1], bufs["k"][1], bufs["v"][1], bufs["out"][1], lse=lse)
    sd.motion_l2(frames, ssd, m)
    rate_b, rate, rp = _guarded((2, 4), torch.float32, -2.0)
    state_b, state, stp = _guarded((2,), torch.float32, 9.0)
    state.fill_(-1.0)
    ctl = sd.NoiseCtl(motion_lo=1.0, motion_hi=80.0, rate_lo=0.2, rate_hi=0.9, ema=0.5, more_noise_when_fast=1)
    sd.noise_from_motion(ctl, m, rate, state)
    torch.cuda.synchronize()
    sd.check_device_error(ws)
    sd.noalloc_check_device_error()

    def bands_ok(base, pad, fill):
        h = base.cpu()
        ref = torch.full((pad,), fill, dtype=base.dtype)
        return torch.equal(h[:pad], ref) and torch.equal(h[-pad:], ref)
    for name, (base, _, pad) in bufs.items():
        assert bands_ok(base, pad, 0x5A5A), name
    assert bands_ok(meta_b, mp, 0x1234567890)
    assert bands_ok(lse_b, lp, 7.25)
    assert bands_ok(ws_b, wp, 0xA5)
    assert bands_ok(ssd_b, sp, 0x77)
    assert bands_ok(m_b, mp2, 3.5)
    assert bands_ok(frames_b, fp_, 0x33)
    assert bands_ok(x_b, xp, 0.5)
    assert bands_ok(wq_b, wqp, -0.25)
    assert bands_ok(bias_b, bp, 1.5)
    assert bands_ok(rate_b, rp, -2.0)
    assert bands_ok(state_b, stp, 9.0)


def test_cuda_graph_replay_equals_eager():
    """The per-layer calls (append + attention) launch kernels only, with their arguments in the
    launch parameters, so a captured graph replays them exactly."""
    cfg = config(W)
    eager = sd.StreamSession(cfg, 1, W.start_frames, "cuda")
    graphed = sd.StreamSession(cfg, 1, W.start_frames, "cuda")
    for c in range(3):
        eager.layer_step(0, [c, c], *_inputs(c))
        graphed.layer_step(0, [c, c], *_inputs(c))
    q, k, v = _inputs(3)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        graphed.layer_step(0, [3, 3], q, k, v, stream=s)
    g.replay()
    eager.layer_step(0, [3, 3], q, k, v)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(graphed.out), bits(eager.out))
    np.testing.assert_array_equal(bits(graphed.layers[0].k), bits(eager.layers[0].k))
    g.replay()                              # a second replay (the next denoise step) is idempotent
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(graphed.out), bits(eager.out))


def test_cuda_graph_replay_of_fused_projection_equals_eager():
    """The fused projection is launched as clusters of two CTAs (its first call on a device also
    sets the shared-memory limit and reads how many pairs fit); captured, as its first call in
    the process or not, it replays to exactly what the eager call writes."""
    cfg = config(W)
    C = W.heads * 128
    g = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randn((W.batch, W.nq, C), generator=g, device="cuda").to(torch.bfloat16)
    wq = (torch.randn((3 * C, C), generator=g, device="cuda") / C ** 0.5).to(torch.bfloat16)
    bias = torch.randn(3 * C, generator=g, device="cuda") * 0.1
    eager = sd.StreamSession(cfg, 1, W.start_frames, "cuda")
    graphed = sd.StreamSession(cfg, 1, W.start_frames, "cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        L = graphed.layers[0]
        sd.qkv_rope_append(cfg, W.start_frames, [2, 2], x, wq, graphed.q_rot, L.k, L.v, L.meta, graphed.ws,
                           bias=bias, stream=s)
    graph.replay()
    L = eager.layers[0]
    sd.qkv_rope_append(cfg, W.start_frames, [2, 2], x, wq, eager.q_rot, L.k, L.v, L.meta, eager.ws, bias=bias)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(graphed.q_rot), bits(eager.q_rot))
    np.testing.assert_array_equal(bits(graphed.layers[0].k), bits(eager.layers[0].k))
    np.testing.assert_array_equal(bits(graphed.layers[0].v), bits(eager.layers[0].v))
    np.testing.assert_array_equal(graphed.layers[0].meta.cpu().numpy(), eager.layers[0].meta.cpu().numpy())


def test_two_sessions_on_two_streams_equal_serial_runs():
    """Two independent sessions (different configurations, one of them large enough to use key
    splits) stepped concurrently on two CUDA streams give, bit for bit, what each gives when run
    alone: no state is shared between workspaces, caches or launches."""
    wa = W
    wb = small_workload(WORKLOADS["wan13b_480p"], heads=2, grid_h=10, grid_w=16)
    chunks = 8
    ins_a = [_inputs(c) for c in range(chunks)]
    ins_b = [tuple(t.cuda() for t in qkv_chunk_host(wb, wb.batch, c, seed_offset=9)) for c in range(chunks)]
    torch.cuda.synchronize()

    def run(concurrent):
        sa = torch.cuda.Stream()
        sb = torch.cuda.Stream() if concurrent else sa
        a = sd.StreamSession(config(wa), 1, wa.start_frames, "cuda", sa)
        b = sd.StreamSession(config(wb), 1, wb.start_frames, "cuda", sb)
        torch.cuda.synchronize()
        oa, ob = [], []
        for c in range(chunks):
            a.layer_step(0, [c] * wa.batch, *ins_a[c], stream=sa)
            with torch.cuda.stream(sa):
                oa.append(a.out.clone())
            b.layer_step(0, [c] * wb.batch, *ins_b[c], stream=sb)
            with torch.cuda.stream(sb):
                ob.append(b.out.clone())
        torch.cuda.synchronize()
        sd.check_device_error(a.ws)
        sd.check_device_error(b.ws)
        return [bits(t) for t in oa], [bits(t) for t in ob], sd.last_kv_splits()

    ca, cb, _ = run(True)
    sa_, sb_, splits_b = run(False)
    assert splits_b > 1, "the larger session should use key splits"
    for c in range(chunks):
        np.testing.assert_array_equal(ca[c], sa_[c], err_msg="session a, chunk %d" % c)
        np.testing.assert_array_equal(cb[c], sb_[c], err_msg="session b, chunk %d" % c)


def test_fused_projections_on_two_streams_equal_serial_runs():
    """Two fused projections (persistent CTA-pair grids sized to the whole GPU) issued on two
    streams at once -- at the 1.3B-480p shape and at a small one -- write, bit for bit, what each
    writes alone: pairs that cannot be resident together run later, nothing waits across grids."""
    shapes = [WORKLOADS["wan13b_480p"], W]
    sessions = {}

    def inputs(w, seed):
        C = w.heads * 128
        g = torch.Generator(device="cuda").manual_seed(seed)
        x = torch.randn((w.batch, w.nq, C), generator=g, device="cuda").to(torch.bfloat16)
        wq = (torch.randn((3 * C, C), generator=g, device="cuda") / C ** 0.5).to(torch.bfloat16)
        return x, wq, torch.randn(3 * C, generator=g, device="cuda") * 0.1
    ins = [inputs(w, 30 + i) for i, w in enumerate(shapes)]

    def run(concurrent):
        streams = [torch.cuda.Stream(), None]
        streams[1] = torch.cuda.Stream() if concurrent else streams[0]
        outs = []
        for i, w in enumerate(shapes):
            sessions[i] = sd.StreamSession(config(w), 1, list(w.start_frames), "cuda")
        torch.cuda.synchronize()
        for rep in range(20):
            for i, w in enumerate(shapes):
                S, L = sessions[i], sessions[i].layers[0]
                x, wq, bias = ins[i]
                sd.qkv_rope_append(config(w), list(w.start_frames), [5] * w.batch, x, wq, S.q_rot, L.k, L.v, L.meta,
                                   S.ws, bias=bias, stream=streams[i])
        torch.cuda.synchronize()
        for i in range(len(shapes)):
            sd.check_device_error(sessions[i].ws)
            outs.append((bits(sessions[i].q_rot).copy(), bits(sessions[i].layers[0].k).copy()))
        return outs

    conc = run(True)
    ser = run(False)
    for i in range(len(shapes)):
        np.testing.assert_array_equal(conc[i][0], ser[i][0])
        np.testing.assert_array_equal(conc[i][1], ser[i][1])


def test_undersized_or_offset_buffers_are_refused_on_the_host():
    """A buffer whose storage ends before the bytes a call touches raises ValueError in the
    binding; nothing is launched (the error word stays clear and a correct call follows)."""
    cfg = config(W)
    sess = sd.StreamSession(cfg, 1, list(W.start_frames), "cuda")
    L = sess.layers[0]
    q, k, v = (torch.randn((W.batch, W.nq, W.heads, 128), device="cuda").to(torch.bfloat16) for _ in range(3))
    short = torch.empty(sess.q_rot.numel() - 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="q_rot"):
        sd.rope_append_kv(cfg, W.start_frames, [0] * W.batch, q, k, v, short, L.k, L.v, L.meta, sess.ws)
    with pytest.raises(ValueError, match="k_cache"):
        sd.chunk_attention(cfg, [0] * W.batch, sess.q_rot, L.k.view(-1)[64:], L.v, sess.out, sess.ws)
    with pytest.raises(ValueError, match="q"):
        sd.rope_append_kv(cfg, W.start_frames, [0] * W.batch, q[:, 1:], k, v, sess.q_rot, L.k, L.v, L.meta, sess.ws)
    sd.rope_append_kv(cfg, W.start_frames, [0] * W.batch, q, k, v, sess.q_rot, L.k, L.v, L.meta, sess.ws)
    sd.chunk_attention(cfg, [0] * W.batch, sess.q_rot, L.k, L.v, sess.out, sess.ws)
    torch.cuda.synchronize()
    sd.check_device_error(sess.ws)
    assert torch.isfinite(sess.out.float()).all()
