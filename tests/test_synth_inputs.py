"""The seeded input generators shared by the oracle and the CUDA path (no method arithmetic):
deterministic, distinct per (layer, chunk, step), the stated distributions and shapes, and the
named workloads' geometry."""
import numpy as np
import torch

from synth_inputs import WORKLOADS, bf16_bits_to_f32, motion_frames_host, qkv_chunk_bits, qkv_chunk_host
from synth_inputs.generators import _seed


def test_seed_is_fnv1a_over_the_decimal_text():
    # FNV-1a 64 offset basis: the hash of the empty string (published constant), masked to 63 bits
    assert _seed() == 0xcbf29ce484222325 & 0x7FFFFFFFFFFFFFFF
    assert _seed(1, 2) == _seed(1, 2) and _seed(1, 2) != _seed(2, 1) and _seed(12) != _seed(1, 2)
    assert all(0 <= _seed(a, b) < 2 ** 63 for a in range(5) for b in range(5))


def test_qkv_chunks_are_deterministic_distinct_and_standard_normal():
    w = WORKLOADS["tiny"]
    a = qkv_chunk_host(w, 2, 3, layer=1, step=0)
    b = qkv_chunk_host(w, 2, 3, layer=1, step=0)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    for other in (qkv_chunk_host(w, 2, 4, layer=1), qkv_chunk_host(w, 2, 3, layer=2),
                  qkv_chunk_host(w, 2, 3, layer=1, step=1)):
        assert not torch.equal(a[0], other[0])
    q, k, v = a
    assert q.shape == (2, w.nq, w.heads, w.head_dim) and q.dtype == torch.bfloat16
    assert not torch.equal(q, k) and not torch.equal(k, v)
    big = qkv_chunk_host(WORKLOADS["wan13b_480p"], 1, 0)[0].float()
    assert abs(big.mean().item()) < 0.01 and abs(big.std().item() - 1.0) < 0.01
    s = qkv_chunk_host(w, 3, 0, same_streams=True)[0]
    assert torch.equal(s[0], s[1]) and torch.equal(s[0], s[2])


def test_bf16_bits_widen_exactly():
    t = torch.randn(4096).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf16_bits_to_f32(bits), t.float().numpy())
    qb = qkv_chunk_bits(WORKLOADS["tiny"], 1, 0)[0]
    np.testing.assert_array_equal(bf16_bits_to_f32(qb), qkv_chunk_host(WORKLOADS["tiny"], 1, 0)[0].float().numpy())


def test_motion_frames_follow_the_recipe():
    f = motion_frames_host(2, 6, 48, 64, 3, seed=9)
    assert f.shape == (2, 6, 48, 64, 3) and f.dtype == torch.uint8
    assert torch.equal(f, motion_frames_host(2, 6, 48, 64, 3, seed=9))
    assert not torch.equal(f[0], f[1])                      # streams differ
    assert not torch.equal(f, motion_frames_host(2, 6, 48, 64, 3, seed=10))
    still = motion_frames_host(1, 4, 48, 64, 3, seed=9, max_speed=0, noise_sigma=0.0)
    assert all(torch.equal(still[0, 0], still[0, t]) for t in range(4))   # no speed, no noise: static
    x = f.float()
    assert 40 < x.mean().item() < 215 and x.min().item() >= 0 and x.max().item() <= 255


def test_workload_geometry():
    w = WORKLOADS["wan13b_480p"]
    assert (w.grid_h, w.grid_w) == (480 // 16, 832 // 16) and w.heads * w.head_dim == 1536
    assert w.nq == 4680 and w.slots * w.hw == 32760
    assert (WORKLOADS["wan13b_720p"].grid_h, WORKLOADS["wan13b_720p"].grid_w) == (720 // 16, 1280 // 16)
    assert WORKLOADS["wan14b_480p"].heads * 128 == 5120
    for v in WORKLOADS.values():
        assert v.rope_t + v.rope_h + v.rope_w == v.head_dim and v.window_frames >= v.chunk_frames
        assert len(v.start_frames) == v.batch
