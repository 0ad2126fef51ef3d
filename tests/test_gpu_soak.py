"""Soak: the fused projection (CTA pairs: cross-CTA barriers, multicast commits) and the chunk
attention (key splits merged by the last arrival) called many times back to back at the
1.3B-480p shape.  Every repeat must be bit-identical to the first and no bounded wait may give
up: a race in the cross-CTA hand-offs would show as a differing repeat or a timeout."""
import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS
from gpu_common import bits, config

pytestmark = pytest.mark.gpu

REPEATS = 2000


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def test_fused_projection_repeats_bit_identically():
    w = WORKLOADS["wan13b_480p"]
    cfg = config(w)
    sess = sd.StreamSession(cfg, 1, list(w.start_frames), "cuda")
    L = sess.layers[0]
    C = w.heads * w.head_dim
    g = torch.Generator(device="cuda").manual_seed(21)
    x = torch.randn((1, w.nq, C), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((3 * C, C), generator=g, device="cuda") / C ** 0.5).to(torch.bfloat16)
    bias = torch.randn(3 * C, generator=g, device="cuda") * 0.1
    call = lambda: sd.qkv_rope_append(cfg, list(w.start_frames), [6], x, W, sess.q_rot, L.k, L.v, L.meta, sess.ws,
                                      bias=bias)
    call()
    torch.cuda.synchronize()
    ref = (bits(sess.q_rot).copy(), bits(L.k).copy(), bits(L.v).copy())
    for _ in range(REPEATS):
        call()
    torch.cuda.synchronize()
    sd.check_device_error(sess.ws)
    np.testing.assert_array_equal(bits(sess.q_rot), ref[0])
    np.testing.assert_array_equal(bits(L.k), ref[1])
    np.testing.assert_array_equal(bits(L.v), ref[2])


def test_chunk_attention_repeats_bit_identically():
    w = WORKLOADS["wan13b_480p"]
    cfg = config(w)
    sess = sd.StreamSession(cfg, 1, list(w.start_frames), "cuda")
    g = torch.Generator(device="cuda").manual_seed(22)
    for c in range(7):                                   # steady state: the window is full
        q, k, v = (torch.randn((1, w.nq, w.heads, 128), generator=g, device="cuda").to(torch.bfloat16)
                   for _ in range(3))
        sess.layer_step(0, [c], q, k, v)
    L = sess.layers[0]
    outs = [torch.empty_like(sess.out) for _ in range(2)]
    sd.chunk_attention(cfg, [6], sess.q_rot, L.k, L.v, outs[0], sess.ws)
    torch.cuda.synchronize()
    assert sd.last_kv_splits() >= 2                      # the split-merge path is the one repeated
    ref = bits(outs[0]).copy()
    for i in range(REPEATS // 4):
        sd.chunk_attention(cfg, [6], sess.q_rot, L.k, L.v, outs[1], sess.ws)
        if i % 25 == 24:
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(outs[1]), ref)
    torch.cuda.synchronize()
    sd.check_device_error(sess.ws)
    np.testing.assert_array_equal(bits(outs[1]), ref)
