"""Pins of the oracle's "next" rows: refresh re-rotation (second reading of the RoPE refresh),
sink update, and the motion-to-noise map.  CPU only."""
import math

import numpy as np
import pytest

import oracle
from synth_inputs import WORKLOADS, qkv_chunk_bits, bf16_bits_to_f32
from dataclasses import replace

DT, DH, DW, BASE = 44, 42, 42, 10000.0


def test_rerotation_keeps_distances_across_the_reset_fp64():
    """After a reset of F*R, a query at the reset time index t and a window key turned back by
    F*R give the same score as the never-reset query at t + F*R against the unturned key."""
    rng = np.random.default_rng(1)
    F, R = 3, 64
    q = rng.standard_normal((8, 128))
    k = rng.standard_normal((8, 128))
    t_new = rng.integers(0, 3, 8).astype(np.float64) + 1000            # reset positions
    tau = rng.integers(0, F * R, 8).astype(np.float64) + 1000          # old window positions
    h = rng.integers(0, 30, 8).astype(np.float64)
    w = rng.integers(0, 52, 8).astype(np.float64)
    hk = rng.integers(0, 30, 8).astype(np.float64)
    wk = rng.integers(0, 52, 8).astype(np.float64)
    k_old = oracle.rope_ideal(k, tau, hk, wk, DT, DH, DW, BASE)
    k_back = oracle.rope_ideal(k_old, np.full(8, -F * R, np.float64), np.zeros(8), np.zeros(8), DT, DH, DW, BASE)
    s_reset = np.sum(oracle.rope_ideal(q, t_new, h, w, DT, DH, DW, BASE) * k_back, axis=1)
    s_cont = np.sum(oracle.rope_ideal(q, t_new + F * R, h, w, DT, DH, DW, BASE) * k_old, axis=1)
    np.testing.assert_allclose(s_reset, s_cont, rtol=0, atol=1e-9)
    # turning the h and w axes as well would break it
    k_bad = oracle.rope_ideal(k_old, np.full(8, -F * R, np.float64), np.full(8, -F * R, np.float64),
                              np.zeros(8), DT, DH, DW, BASE)
    s_bad = np.sum(oracle.rope_ideal(q, t_new, h, w, DT, DH, DW, BASE) * k_bad, axis=1)
    assert np.abs(s_bad - s_cont).max() > 1e-3


def test_rerotation_spec_touches_only_time_dims():
    x = qkv_chunk_bits(WORKLOADS["tiny"], 1, 0)[1].reshape(-1, 128)[:500]
    n = x.shape[0]
    z = np.zeros(n, np.int64)
    y = oracle.rope_spec(x, np.full(n, -192, np.int64), z, z, DT, DH, DW, BASE)
    np.testing.assert_array_equal(y[:, 44:], x[:, 44:])
    assert np.mean(y[:, :44] != x[:, :44]) > 0.5
    # turning back and forth: each of the two roundings moves an element by at most half a
    # bf16 ulp of a value no larger than its pair's norm
    y2 = oracle.rope_spec(y, np.full(n, 192, np.int64), z, z, DT, DH, DW, BASE)
    a = bf16_bits_to_f32(y2).astype(np.float64)
    b = bf16_bits_to_f32(x).astype(np.float64)
    pair_norm = np.repeat(np.hypot(b[:, 0::2], b[:, 1::2]), 2, axis=1)
    assert np.all(np.abs(a - b) <= 2 * pair_norm * 2.0 ** -8 + 1e-30)
    assert np.mean(a != b) < 0.5


def _small(R=3, W=9):
    return replace(WORKLOADS["tiny"], heads=1, grid_h=2, grid_w=3, window_frames=W, refresh_chunks=R,
                   start_frames=[50])


def test_stream_tpos_after_resets_equals_continuous_tpos_minus_shifts():
    """With re-rotation, every retained window frame's time index is the never-reset index
    minus F*R per reset it went through, and so is the new chunk's."""
    w = _small(R=3, W=9)
    w0 = replace(w, refresh_chunks=0)
    so, s0 = oracle.StreamOracle(w, 50), oracle.StreamOracle(w0, 50)
    for c in range(10):
        q, k, v = (x[0] for x in qkv_chunk_bits(w, 1, c))
        so.refresh_rerotate(c)
        so.append_chunk(c, q, k, v)
        s0.append_chunk(c, q, k, v)
        resets = c // 3
        for e, e0 in zip(so.cache.entries[w.sink_frames:], s0.cache.entries[w0.sink_frames:]):
            assert e[0] == e0[0]
            assert e[1] == e0[1] - w.chunk_frames * 3 * resets


def test_stream_rerotated_keys_keep_scores_continuous():
    """Right after a reset, the new chunk's queries score the re-rotated window keys as a stream
    that never resets scores its unrotated keys (fp64 products of the bf16 cache contents; the
    only difference is bf16 rounding of the rotations)."""
    w = _small(R=3, W=9)
    w0 = replace(w, refresh_chunks=0)
    so, s0 = oracle.StreamOracle(w, 50), oracle.StreamOracle(w0, 50)
    for c in range(7):                                  # resets at chunks 3 and 6
        q, k, v = (x[0] for x in qkv_chunk_bits(w, 1, c))
        so.refresh_rerotate(c)
        qr = so.append_chunk(c, q, k, v)
        qr0 = s0.append_chunk(c, q, k, v)
    nwin = sum(1 for e in so.cache.entries[w.sink_frames:] if e[0] < 6 * w.chunk_frames) * w.hw
    assert nwin > 0
    worst = 0.0
    for h in range(w.heads):
        qa = bf16_bits_to_f32(qr[:, h, :]).astype(np.float64)
        qb = bf16_bits_to_f32(qr0[:, h, :]).astype(np.float64)
        ka = bf16_bits_to_f32(so.cache.keys(h)[w.sink_frames * w.hw:][:nwin]).astype(np.float64)
        kb = bf16_bits_to_f32(s0.cache.keys(h)[w0.sink_frames * w0.hw:][:nwin]).astype(np.float64)
        worst = max(worst, float(np.abs(qa @ ka.T - qb @ kb.T).max()))
    assert worst < 0.5, worst


def test_sink_update_copies_the_last_frames():
    w = _small(R=3, W=9)
    so = oracle.StreamOracle(w, 0)
    for c in range(4):
        q, k, v = (x[0] for x in qkv_chunk_bits(w, 1, c))
        so.append_chunk(c, q, k, v)
    so.sink_update()
    ids = [e[0] for e in so.cache.entries]
    assert ids[:3] == [9, 10, 11] and ids[-3:] == [9, 10, 11]
    for a, b in zip(so.cache.entries[:3], so.cache.entries[-3:]):
        np.testing.assert_array_equal(a[2], b[2])
        np.testing.assert_array_equal(a[3], b[3])
        assert a[1] == b[1] and a[2] is not b[2]
    # a later denoise step re-appends the window originals, not the sink copies
    q, k, v = (x[0] for x in qkv_chunk_bits(w, 1, 99))
    so.append_chunk(3, q, k, v)
    assert not np.array_equal(so.cache.entries[0][2], so.cache.entries[-3][2])


NOISE = dict(m_lo=2.0, m_hi=12.0, out_lo=0.1, out_hi=0.9)


@pytest.mark.parametrize("fast_more", [0, 1])
def test_noise_map_monotone_endpoints_and_direction(fast_more):
    m = np.linspace(-5, 20, 401, dtype=np.float32)[None, :]
    r = oracle.noise(m, **NOISE, ema=0.0, more_noise_when_fast=fast_more)[0]
    d = np.diff(r.astype(np.float64))
    assert np.all(d >= 0) if fast_more else np.all(d <= 0)
    lo_end, hi_end = (NOISE["out_lo"], NOISE["out_hi"]) if fast_more else (NOISE["out_hi"], NOISE["out_lo"])
    assert r[m[0] <= 2.0].tolist() == [np.float32(lo_end)] * int(np.sum(m[0] <= 2.0))
    assert r[m[0] >= 12.0].tolist() == [np.float32(hi_end)] * int(np.sum(m[0] >= 12.0))
    other = oracle.noise(m, **NOISE, ema=0.0, more_noise_when_fast=1 - fast_more)[0]
    np.testing.assert_allclose(r + other, NOISE["out_lo"] + NOISE["out_hi"], atol=1e-6)


def test_noise_smoothing_closed_form_and_state_carry():
    ema = 0.75
    m = np.array([[0.0] * 1 + [20.0] * 30], np.float32)           # a step from the low to the high end
    r = oracle.noise(m, **NOISE, ema=ema, more_noise_when_fast=1)[0].astype(np.float64)
    k = np.arange(31)
    expect = NOISE["out_hi"] + (NOISE["out_lo"] - NOISE["out_hi"]) * ema ** k
    np.testing.assert_allclose(r, expect, atol=1e-6)
    # two calls with the state carried equal one call over the concatenation
    state = np.full(1, -1.0, np.float32)
    a = oracle.noise(m[:, :10], **NOISE, ema=ema, more_noise_when_fast=1, state=state)
    b = oracle.noise(m[:, 10:], **NOISE, ema=ema, more_noise_when_fast=1, state=state)
    np.testing.assert_array_equal(np.concatenate([a, b], 1), oracle.noise(m, **NOISE, ema=ema, more_noise_when_fast=1))


def test_qkv_projection_brute_force():
    rng = np.random.default_rng(3)
    x = oracle.f32_to_bf16(rng.standard_normal((3, 5)).astype(np.float32))
    w = oracle.f32_to_bf16(rng.standard_normal((7, 5)).astype(np.float32))
    bias = rng.standard_normal(7).astype(np.float32)
    y = oracle.qkv_project(x, w, bias)
    xf, wf = bf16_bits_to_f32(x), bf16_bits_to_f32(w)
    for i in range(3):
        for j in range(7):
            ref = sum(float(xf[i, c]) * float(wf[j, c]) for c in range(5)) + float(bias[j])
            assert y[i, j] == pytest.approx(ref, rel=1e-14, abs=1e-14)
