"""Pins of the oracle against facts that do not come from the oracle itself.

Every test here runs on the CPU.  Each one is chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign, a swapped index, an off-by-one in the ring) fails it:
exhaustive or closed-form checks, library routines on special cases, brute force on tiny
inputs, and the invariants that the pages' method relies on.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from synth_inputs import WORKLOADS, qkv_chunk_bits, bf16_bits_to_f32


# ------------------------------------------------------------------------------------------
# bf16 rounding (P9)
# ------------------------------------------------------------------------------------------

def test_bf16_rne_exhaustive_against_second_formulation():
    """All 2^32 fp32 bit patterns: the bit-trick RNE equals nearest-by-distance (ties to even)."""
    assert oracle.lib().orc_bf16_mismatches(0, 1 << 32) == 0


def test_bf16_rne_matches_torch_on_samples():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


@pytest.mark.parametrize("f32_bits,bf16_bits", [
    (0x3F800000, 0x3F80),   # 1.0
    (0x3F808000, 0x3F80),   # tie, lower code even -> down
    (0x3F818000, 0x3F82),   # tie, lower code odd -> up
    (0x3F808001, 0x3F81),   # just above the tie -> up
    (0x80000000, 0x8000),   # -0
    (0x7F7F7FFF, 0x7F7F),   # just below the overflow threshold
    (0x7F7F8000, 0x7F80),   # the overflow threshold itself rounds to +inf (tie to even)
    (0xFF800000, 0xFF80),   # -inf
    (0x00008000, 0x0000),   # smallest subnormal tie -> 0 (even)
    (0x00018000, 0x0002),   # subnormal tie -> up to even
])
def test_bf16_rne_special_values(f32_bits, bf16_bits):
    x = np.array([f32_bits], dtype=np.uint32).view(np.float32)
    assert int(oracle.f32_to_bf16(x)[0]) == bf16_bits


# ------------------------------------------------------------------------------------------
# RoPE (P1, P2, spec vs ideal)
# ------------------------------------------------------------------------------------------

DT, DH, DW, BASE = 44, 42, 42, 10000.0


def _rand(n, seed, d=128):
    return np.random.default_rng(seed).standard_normal((n, d))


def test_rope_matches_complex_rotation_per_pair():
    """Each pair (2j, 2j+1) of an axis segment is the complex number x + iy multiplied by
    exp(i * pos * base^(-2j/d_axis)); numpy's complex exp is the independent reference."""
    x = _rand(7, 1)
    tp = np.array([0, 1, 5, 37, 1000, 65535, 100191], np.float64)
    hp = np.array([0, 3, 29, 1, 12, 44, 7], np.float64)
    wp = np.array([0, 51, 2, 79, 13, 0, 40], np.float64)
    y = oracle.rope_ideal(x, tp, hp, wp, DT, DH, DW, BASE)
    off = 0
    for d_axis, pos in ((DT, tp), (DH, hp), (DW, wp)):
        j = np.arange(d_axis // 2)
        ang = pos[:, None] * np.power(BASE, -2.0 * j / d_axis)[None, :]
        z = (x[:, off:off + d_axis:2] + 1j * x[:, off + 1:off + d_axis:2]) * np.exp(1j * ang)
        np.testing.assert_allclose(y[:, off:off + d_axis:2], z.real, rtol=0, atol=1e-12)
        np.testing.assert_allclose(y[:, off + 1:off + d_axis:2], z.imag, rtol=0, atol=1e-12)
        off += d_axis


def test_rope_axis_segments_only_move_their_own_dims():
    """A position on one axis rotates only that axis's segment (t=[0,44), h=[44,86), w=[86,128))."""
    x = _rand(1, 2)
    for axis, seg in ((0, slice(0, 44)), (1, slice(44, 86)), (2, slice(86, 128))):
        pos = [np.zeros(1), np.zeros(1), np.zeros(1)]
        pos[axis] = np.array([3.0])
        y = oracle.rope_ideal(x, *pos, DT, DH, DW, BASE)
        moved = np.abs(y - x)[0] > 1e-12
        expect = np.zeros(128, bool)
        expect[seg] = True
        # pair j=0 of every segment has frequency 1, so every pair of the segment moves
        assert (moved == expect).all()


def test_rope_preserves_pair_norms():
    x = _rand(64, 3)
    rng = np.random.default_rng(4)
    tp, hp, wp = (rng.integers(0, 110000, 64).astype(np.float64) for _ in range(3))
    y = oracle.rope_ideal(x, tp, hp, wp, DT, DH, DW, BASE)
    nx = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    ny = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12, atol=0)


def test_rope_relative_position_property():
    """<R(p) q, R(p') k> = <R(p - p') q, k> for positions up to 1.1e5 on every axis."""
    q = _rand(16, 5)
    k = _rand(16, 6)
    rng = np.random.default_rng(7)
    for _ in range(4):
        p = rng.integers(0, 110000, (3, 16)).astype(np.float64)
        pp = rng.integers(0, 110000, (3, 16)).astype(np.float64)
        lhs = np.sum(oracle.rope_ideal(q, *p, DT, DH, DW, BASE) *
                     oracle.rope_ideal(k, *pp, DT, DH, DW, BASE), axis=1)
        rhs = np.sum(oracle.rope_ideal(q, *(p - pp), DT, DH, DW, BASE) * k, axis=1)
        np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-10 * 128)


def test_rope_spec_zero_position_is_identity_bit_exact():
    x = qkv_chunk_bits(WORKLOADS["tiny"], 1, 0)[0].reshape(-1, 128)
    z = np.zeros(x.shape[0], np.int64)
    np.testing.assert_array_equal(oracle.rope_spec(x, z, z, z, DT, DH, DW, BASE), x)


def test_rope_spec_within_one_bf16_ulp_of_rounded_ideal():
    w = WORKLOADS["tiny"]
    x = qkv_chunk_bits(w, 1, 3)[1].reshape(-1, 128)[:2000]
    rng = np.random.default_rng(8)
    tp = rng.integers(0, 110000, x.shape[0])
    hp = rng.integers(0, 45, x.shape[0])
    wp = rng.integers(0, 80, x.shape[0])
    spec = oracle.rope_spec(x, tp, hp, wp, DT, DH, DW, BASE)
    ideal = oracle.rope_ideal(bf16_bits_to_f32(x).astype(np.float64), tp, hp, wp, DT, DH, DW, BASE)
    ideal_b = oracle.f32_to_bf16(ideal.astype(np.float32))
    a = bf16_bits_to_f32(spec).astype(np.float64)
    b = bf16_bits_to_f32(ideal_b).astype(np.float64)
    ulp = np.maximum(np.abs(b), 2.0 ** -126) * 2.0 ** -7
    assert np.all(np.abs(a - b) <= ulp + 1e-30)
    # the spec is not the identity: positions do rotate
    assert np.mean(spec != x) > 0.5


def test_rope_cos_sin_table_values():
    """The fp32 table entries are the fp32 rounding of libm's fp64 cos/sin: for pair 0 the
    frequency is exactly 1, so the angle is the position itself."""
    for pos in (0, 1, 2, 7, 1000, 100002):
        c, s = oracle.rope_cos_sin_f32(pos, 0, 44, BASE)
        assert c == float(np.float32(math.cos(pos))) and s == float(np.float32(math.sin(pos)))
    # last pair of the 44-dim time axis: frequency base^(-42/44)
    assert oracle.rope_omega(21, 44, BASE) == pytest.approx(BASE ** (-42 / 44), rel=1e-15)


# ------------------------------------------------------------------------------------------
# Causal-RoPE with a global time index (P3) and the refresh reading
# ------------------------------------------------------------------------------------------

def _global_positions(start, n_frames, gh, gw):
    """Positions of every token of frames 0..n-1 of a stream computed over the whole sequence."""
    hw = gh * gw
    out = []
    for g in range(n_frames * hw):
        frame = g // hw
        r = g % hw
        out.append((start + frame, r // gw, r % gw))
    return np.array(out, np.int64)


@pytest.mark.parametrize("start", [0, 17, 100000])
def test_local_chunk_positions_equal_global_sequence_positions(start):
    F, gh, gw = 3, 4, 6
    chunks = 6
    glob = _global_positions(start, F * chunks, gh, gw)
    hw = gh * gw
    for c in range(chunks):
        t, h, w, frame = oracle.chunk_positions(start, c, F, gh, gw, 0)
        sl = glob[c * F * hw:(c + 1) * F * hw]
        np.testing.assert_array_equal(np.stack([t, h, w], 1), sl)
        np.testing.assert_array_equal(frame, np.arange(c * F, (c + 1) * F).repeat(hw))


def test_local_rope_equals_global_rope_bit_exact():
    w = WORKLOADS["tiny"]
    F, gh, gw, hw = w.chunk_frames, w.grid_h, w.grid_w, w.hw
    start = 12345
    chunks = 4
    xs = [qkv_chunk_bits(w, 1, c)[1][0] for c in range(chunks)]     # [Nq][H][D] per chunk
    whole = np.concatenate(xs, 0)
    glob = _global_positions(start, F * chunks, gh, gw)
    rot_glob = oracle.rope_spec(whole, glob[:, 0], glob[:, 1], glob[:, 2], DT, DH, DW, BASE)
    for c in range(chunks):
        t, h, ww, _ = oracle.chunk_positions(start, c, F, gh, gw, 0)
        rot = oracle.rope_spec(xs[c], t, h, ww, DT, DH, DW, BASE)
        np.testing.assert_array_equal(rot, rot_glob[c * F * hw:(c + 1) * F * hw])


def test_refresh_resets_time_offset_every_R_chunks():
    F, gh, gw, R, S = 3, 2, 3, 4, 1000
    for c in range(3 * R):
        t, _, _, frame = oracle.chunk_positions(S, c, F, gh, gw, R)
        t0, _, _, _ = oracle.chunk_positions(S, c % R, F, gh, gw, R)
        np.testing.assert_array_equal(t, t0)
        assert frame.min() == c * F           # the cache frame number keeps counting
    t, _, _, _ = oracle.chunk_positions(S, R, F, gh, gw, R)
    assert t.min() == S                       # back at the stream's anchor


# ------------------------------------------------------------------------------------------
# Sink + rolling window cache (P4)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("F,Fs,W,chunks", [
    (3, 3, 4, 10),       # tiny workload: window wraps inside a chunk
    (3, 3, 18, 140),     # 1.3B-480p / stream-batch shape, many wraps
    (3, 2, 3, 12),       # sink not a multiple of the chunk
    (3, 0, 6, 12),       # no sink
    (2, 5, 2, 12),       # window equal to the chunk
])
def test_ring_slots_equal_concatenate_then_truncate(F, Fs, W, chunks):
    cache = oracle.FrameListCache(Fs, W)
    for c in range(chunks):
        for i in range(F):
            cache.append(c * F + i, 0, None, None)
        n = (c + 1) * F
        kept = cache.frames()
        # brute-force retained set: first Fs frames, then the last W of the remaining ones
        allf = list(range(n))
        expect = allf[:Fs] + (allf[Fs:][-W:] if W and len(allf) > Fs else [])
        assert kept == expect
        ring = oracle.ring_pointer_slots(n, Fs, W)
        slots = [oracle.slot_of_frame(f, Fs, W) for f in kept]
        assert slots == [ring[f] for f in kept]
        # the retained frames fill exactly the first len(kept) slots: a contiguous prefix
        assert sorted(slots) == list(range(len(kept)))
        # the current chunk is always inside the window
        assert all(f in kept for f in range(c * F, n))


def test_reappending_a_chunk_replaces_contents_only():
    cache = oracle.FrameListCache(3, 4)
    for f in range(9):
        cache.append(f, f, np.full((1, 1, 1), f), np.full((1, 1, 1), f))
    before = cache.frames()
    for f in range(6, 9):
        cache.append(f, f + 100, np.full((1, 1, 1), -f), np.full((1, 1, 1), -f))
    assert cache.frames() == before
    assert [e[1] for e in cache.entries][-3:] == [106, 107, 108]
    with pytest.raises(ValueError):     # frame 4 was evicted; it cannot come back
        cache.append(4, 0, None, None)


# ------------------------------------------------------------------------------------------
# Softmax and attention (P5, P6, P7)
# ------------------------------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_match_scipy():
    rng = np.random.default_rng(9)
    for n in (1, 2, 17, 1000):
        s = rng.standard_normal(n) * 30
        p, lse = oracle.softmax(s)
        assert abs(p.sum() - 1.0) < 1e-12
        np.testing.assert_allclose(p, scipy.special.softmax(s), rtol=1e-12, atol=1e-300)
        assert lse == pytest.approx(scipy.special.logsumexp(s), rel=1e-14)
        p2, _ = oracle.softmax(s + 123.0)
        np.testing.assert_allclose(p2, p, rtol=1e-12, atol=1e-300)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((5, 8))
    k = rng.standard_normal((7, 8))
    v = rng.standard_normal((7, 8))
    scale = 1 / math.sqrt(8)
    out, lse = oracle.attention_f64(q, k, v, scale)
    for r in range(5):
        s = [scale * sum(q[r, d] * k[j, d] for d in range(8)) for j in range(7)]
        e = [math.exp(x) for x in s]
        z = sum(e)
        o = [sum(e[j] / z * v[j, d] for j in range(7)) for d in range(8)]
        np.testing.assert_allclose(out[r], o, rtol=1e-12, atol=1e-14)
        assert lse[r] == pytest.approx(math.log(z), rel=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((4, 16))
    k = rng.standard_normal((9, 16))
    v = rng.standard_normal((9, 16))
    # constant values -> output is that value
    vc = np.tile(rng.standard_normal(16), (9, 1))
    out, _ = oracle.attention_f64(q, k, vc, 0.25)
    np.testing.assert_allclose(out, np.tile(vc[0], (4, 1)), rtol=1e-13, atol=1e-13)
    # zero query -> uniform weights -> mean of the values; lse = log(n)
    out, lse = oracle.attention_f64(np.zeros((2, 16)), k, v, 0.25)
    np.testing.assert_allclose(out, np.tile(v.mean(0), (2, 1)), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(9), rtol=1e-14)
    # a single key -> its value
    out, _ = oracle.attention_f64(q, k[:1], v[:1], 0.25)
    np.testing.assert_allclose(out, np.tile(v[0], (4, 1)), rtol=0, atol=1e-14)
    # permuting the keys (with their values) changes nothing
    perm = rng.permutation(9)
    o1, _ = oracle.attention_f64(q, k, v, 0.25)
    o2, _ = oracle.attention_f64(q, k[perm], v[perm], 0.25)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)


def test_attention_bf16_entry_equals_fp64_entry_on_widened_inputs():
    w = WORKLOADS["tiny"]
    q, k, v = (x[0, :, 0, :] for x in qkv_chunk_bits(w, 1, 0))
    a, la = oracle.attention_bf16(q, k, v, 0.1, rows=np.array([0, 5, 71]))
    b, lb = oracle.attention_f64(bf16_bits_to_f32(q)[[0, 5, 71]].astype(np.float64),
                                 bf16_bits_to_f32(k).astype(np.float64),
                                 bf16_bits_to_f32(v).astype(np.float64), 0.1)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_shift_invariance_of_stream_offsets():
    """Identical q, k, v streamed from global offsets 0, 1e3, 1e4, 1e5 give the same fp64
    attention (only position differences matter); R = 0 so the offsets never reset."""
    w = WORKLOADS["tiny"]
    F, gh, gw, hw = w.chunk_frames, w.grid_h, w.grid_w, w.hw
    chunks = 3
    data = [tuple(bf16_bits_to_f32(x[0, :, 0, :]).astype(np.float64) for x in qkv_chunk_bits(w, 1, c))
            for c in range(chunks)]
    outs = []
    for S in (0, 1000, 10000, 100000):
        ks, vs = [], []
        for c in range(chunks):
            t, h, ww, _ = oracle.chunk_positions(S, c, F, gh, gw, 0)
            q, k, v = data[c]
            ks.append(oracle.rope_ideal(k, t, h, ww, DT, DH, DW, BASE))
            vs.append(v)
            qr = oracle.rope_ideal(q, t, h, ww, DT, DH, DW, BASE)
        o, _ = oracle.attention_f64(qr, np.concatenate(ks), np.concatenate(vs), 1 / math.sqrt(128))
        outs.append(o)
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-9)


def test_stream_oracle_tiny_chunk_shapes_and_visibility():
    w = WORKLOADS["tiny"]
    so = oracle.StreamOracle(w, 0)
    seen = []
    for c in range(w.chunks):
        q, k, v = (x[0] for x in qkv_chunk_bits(w, 1, c))
        q_rot = so.append_chunk(c, q, k, v)
        assert q_rot.shape == q.shape
        out, lse = so.attend(q_rot, 1, rows=np.array([0, 71]))
        assert out.shape == (2, 128) and np.all(np.isfinite(out))
        seen.append(len(so.cache.frames()))
    # 3, 6, then sink 3 + window 4 from chunk 2 on
    assert seen == [3, 6] + [7] * (w.chunks - 2)


# ------------------------------------------------------------------------------------------
# Motion (P8)
# ------------------------------------------------------------------------------------------

def test_motion_identical_frames_and_symmetry():
    rng = np.random.default_rng(12)
    f = rng.integers(0, 256, (2, 3, 8, 16, 3), dtype=np.uint8)
    f[:, 1] = f[:, 0]
    ssd = oracle.motion_ssd(f)
    assert (ssd[:, 0] == 0).all()
    rev = np.ascontiguousarray(f[:, ::-1])
    np.testing.assert_array_equal(oracle.motion_ssd(rev)[:, ::-1], ssd)


@pytest.mark.parametrize("a,d", [(1, 1), (1, 5), (2, 16), (3, 7)])
def test_motion_shifted_ramp_closed_form(a, d):
    hp, wp, ch = 6, 80, 3
    x = np.arange(wp)
    assert a * (wp - 1) < 256
    ramp = np.broadcast_to((a * x)[None, :, None], (hp, wp, ch)).astype(np.uint8)
    moved = np.roll(ramp, d, axis=1)          # moved(x) = ramp(x - d), cyclic
    f = np.stack([ramp, moved])[None]
    expect = hp * ch * ((wp - d) * (a * d) ** 2 + d * (a * (wp - d)) ** 2)
    assert int(oracle.motion_ssd(f)[0, 0]) == expect


def test_motion_noise_only_statistics():
    rng = np.random.default_rng(13)
    n = 200000
    sigma = 4.0
    frames = np.clip(np.round(128 + rng.standard_normal((1, 2, n)) * sigma), 0, 255).astype(np.uint8)
    ssd = int(oracle.motion_ssd(frames)[0, 0])
    # each frame carries N(0, sigma^2) plus rounding noise of variance 1/12
    expect = n * 2 * (sigma ** 2 + 1 / 12)
    assert abs(ssd - expect) / expect < 0.05
    m = oracle.motion_rms(ssd, n)
    assert abs(m - math.sqrt(2 * (sigma ** 2 + 1 / 12))) < 0.1
