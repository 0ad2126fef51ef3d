"""Seeded sweep of the fused QKV projection + Causal-RoPE + append against the fp64 oracle:
random head counts (odd and even), grids (ragged 256-token tiles), chunk sizes, stream counts, RoPE splits,
refresh periods, with and without bias, and padded input token strides.  Each chunk: q_rot, the
appended k and v rows within 2^-8 of each rotation pair's norm, slot metadata exact.
SDV2_SWEEP_QKV_CONFIGS sets the number of configurations (default 6)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS
from gpu_common import bits, config, small_workload, to_f64
from test_gpu_next_rows import _close

pytestmark = pytest.mark.gpu

N_CONFIGS = int(os.environ.get("SDV2_SWEEP_QKV_CONFIGS", "6"))


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def _random_case(seed):
    rng = np.random.default_rng(5000 + seed)
    F = int(rng.integers(1, 4))
    Fs = int(rng.integers(0, 4))
    W = int(rng.integers(F, F + 5))
    B = int(rng.choice([1, 2, 3]))
    rt = int(rng.choice([0, 8, 20, 44, 72, 128]))
    rh = 2 * int(rng.integers(0, (128 - rt) // 2 + 1))
    big = seed % 3 == 2
    gh = int(rng.integers(8, 20)) if big else int(rng.integers(1, 9))
    gw = int(rng.integers(8, 24)) if big else int(rng.integers(1, 11))
    w = small_workload(WORKLOADS["tiny"], batch=B, heads=int(rng.choice([1, 2, 3, 4, 5, 6])), grid_h=gh, grid_w=gw,
                       chunk_frames=F, sink_frames=Fs, window_frames=W, refresh_chunks=int(rng.choice([0, 2, 3])),
                       rope_t=rt, rope_h=rh, rope_w=128 - rt - rh,
                       start_frames=[int(x) for x in rng.integers(0, 120000, B)])
    pad = int(rng.choice([0, 8, 40]))
    with_bias = bool(rng.random() < 0.7)
    return w, pad, with_bias


@pytest.mark.parametrize("seed", range(N_CONFIGS))
def test_random_fused_projection_configs(seed):
    w, pad, with_bias = _random_case(seed)
    C = w.heads * w.head_dim
    ld = C + pad
    cfg = config(w)
    starts = list(w.start_frames)
    sess = sd.StreamSession(cfg, 1, starts, "cuda")
    L = sess.layers[0]
    hw = w.hw
    g = torch.Generator().manual_seed(6000 + seed)
    W = (torch.randn((3 * C, C), generator=g) / math.sqrt(C)).to(torch.bfloat16)
    bias = (torch.randn(3 * C, generator=g) * 0.1).float() if with_bias else None
    for c in range(3):
        x_full = torch.randn((w.batch, w.nq, ld), generator=g).to(torch.bfloat16)
        sd.qkv_rope_append(cfg, starts, [c] * w.batch, x_full.cuda(), W.cuda(), sess.q_rot, L.k, L.v, L.meta,
                           sess.ws, bias=None if bias is None else bias.cuda(), x_token_stride=ld)
        torch.cuda.synchronize()
        qg = to_f64(sess.q_rot)
        kg, vg = to_f64(L.k), to_f64(L.v)
        meta = L.meta.cpu().numpy()
        for b in range(w.batch):
            x = x_full[b, :, :C].contiguous()
            y = oracle.qkv_project(bits(x), bits(W), None if bias is None else bias.numpy())
            t, h, ww, frame = oracle.chunk_positions(starts[b], c, w.chunk_frames, w.grid_h, w.grid_w,
                                                     w.refresh_chunks)
            rep = lambda a: np.repeat(a.astype(np.float64), w.heads)
            rot = lambda z: oracle.rope_ideal(z.reshape(-1, 128), rep(t), rep(h), rep(ww), w.rope_t, w.rope_h,
                                              w.rope_w, w.rope_base).reshape(w.nq, w.heads, 128)
            q, k = rot(y[:, :C]), rot(y[:, C:2 * C])
            v = y[:, 2 * C:].reshape(w.nq, w.heads, 128)
            _close(qg[b].transpose(1, 0, 2), q, "q_rot seed %d chunk %d stream %d" % (seed, c, b))
            for i in range(w.chunk_frames):
                f = c * w.chunk_frames + i
                s = oracle.slot_of_frame(f, w.sink_frames, w.window_frames)
                assert tuple(meta[b, s]) == (f, int(t[i * hw])), (seed, c, b, s, tuple(meta[b, s]))
                _close(kg[b][:, s * hw:(s + 1) * hw, :].transpose(1, 0, 2), k[i * hw:(i + 1) * hw], "k slot %d" % s)
                _close(vg[b][:, s * hw:(s + 1) * hw, :].transpose(1, 0, 2), v[i * hw:(i + 1) * hw], "v slot %d" % s)
    sd.check_device_error(sess.ws)
