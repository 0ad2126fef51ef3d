"""The oracle's pins catch plausible mistakes.

Each case below swaps one oracle function for a deliberately wrong version -- a slip of the
kind a hand-written reference could contain (a sign, a swapped axis, a missing factor of 2 in
a frequency exponent, a dropped term, an off-by-one in the ring, a wrong operand, a missing
scale) -- and runs the pins that guard that function.  At least one pin must fail for every
mutant.  The mutants live only here, on the CPU; nothing of them reaches the library.
"""
import math

import numpy as np
import pytest

import oracle
import test_oracle_pins as P
import test_oracle_pins_next as PN

DT, DH, DW, BASE = P.DT, P.DH, P.DW, P.BASE

_rope_ideal = oracle.rope_ideal
_chunk_positions = oracle.chunk_positions
_slot_of_frame = oracle.slot_of_frame
_attention_f64 = oracle.attention_f64
_softmax = oracle.softmax
_motion_ssd = oracle.motion_ssd
_noise = oracle.noise
_qkv_project = oracle.qkv_project
_rope_spec = oracle.rope_spec


# ------------------------------------------------------------------------------------------
# RoPE mutants
# ------------------------------------------------------------------------------------------

def _rope_np(x, tp, hp, wp, dt, dh, dw, base, pairing="adjacent", two=2.0, drop_term=False):
    """A numpy rotary embedding with switchable slips."""
    x = np.asarray(x, np.float64)
    y = x.copy()
    off = 0
    for d_axis, pos in ((dt, tp), (dh, hp), (dw, wp)):
        half = d_axis // 2
        j = np.arange(half)
        ang = np.asarray(pos, np.float64)[:, None] * np.power(base, -two * j / d_axis)[None, :]
        c, s = np.cos(ang), np.sin(ang)
        if pairing == "adjacent":
            a_idx, b_idx = off + 2 * j, off + 2 * j + 1
        else:                                   # first half of the segment paired with the second
            a_idx, b_idx = off + j, off + half + j
        xa, xb = x[:, a_idx], x[:, b_idx]
        y[:, a_idx] = xa * c if drop_term else xa * c - xb * s
        y[:, b_idx] = xa * s + xb * c
        off += d_axis
    return y


def rope_negated_angle(x, tp, hp, wp, dt, dh, dw, base):
    return _rope_ideal(x, -np.asarray(tp, np.float64), -np.asarray(hp, np.float64), -np.asarray(wp, np.float64),
                       dt, dh, dw, base)


def rope_h_w_swapped(x, tp, hp, wp, dt, dh, dw, base):
    return _rope_ideal(x, tp, wp, hp, dt, dh, dw, base)


def rope_missing_factor_two(x, tp, hp, wp, dt, dh, dw, base):
    return _rope_np(x, tp, hp, wp, dt, dh, dw, base, two=1.0)


def rope_half_split_pairs(x, tp, hp, wp, dt, dh, dw, base):
    return _rope_np(x, tp, hp, wp, dt, dh, dw, base, pairing="half")


def rope_dropped_term(x, tp, hp, wp, dt, dh, dw, base):
    return _rope_np(x, tp, hp, wp, dt, dh, dw, base, drop_term=True)


ROPE_PINS = [P.test_rope_matches_complex_rotation_per_pair, P.test_rope_axis_segments_only_move_their_own_dims,
             P.test_rope_preserves_pair_norms, P.test_rope_relative_position_property]


# ------------------------------------------------------------------------------------------
# position / refresh mutants
# ------------------------------------------------------------------------------------------

def positions_never_reset(start, chunk, F, gh, gw, R):
    return _chunk_positions(start, chunk, F, gh, gw, 0)


def positions_reset_period_off_by_one(start, chunk, F, gh, gw, R):
    return _chunk_positions(start, chunk, F, gh, gw, R + 1 if R > 0 else 0)


def positions_h_w_swapped(start, chunk, F, gh, gw, R):
    t, h, w, frame = _chunk_positions(start, chunk, F, gh, gw, R)
    n = np.arange(t.size) % (gh * gw)
    return t, n % gh, n // gh, frame          # column-major inside the frame


def positions_frame_number_off_by_one(start, chunk, F, gh, gw, R):
    t, h, w, frame = _chunk_positions(start, chunk, F, gh, gw, R)
    return t, h, w, frame + 1


POSITION_PINS = [lambda: P.test_local_chunk_positions_equal_global_sequence_positions(17),
                 P.test_refresh_resets_time_offset_every_R_chunks]


# ------------------------------------------------------------------------------------------
# cache mutants
# ------------------------------------------------------------------------------------------

def slot_ring_off_by_one(frame, Fs, W):
    return frame if frame < Fs else Fs + (frame - Fs + 1) % W


def slot_sink_in_ring(frame, Fs, W):
    return frame % (Fs + W)


class CacheForgetsSink(oracle.FrameListCache):
    """Truncates the whole list to its last F_s + W frames: the sink is evicted."""

    def append(self, frame, tpos, k, v):
        for e in self.entries:
            if e[0] == frame:
                e[1], e[2], e[3] = tpos, k, v
                return
        self.entries.append([frame, tpos, k, v])
        self.appended += 1
        keep = self.sink_frames + self.window_frames
        self.entries = self.entries[-keep:]


CACHE_PINS = [lambda: P.test_ring_slots_equal_concatenate_then_truncate(3, 3, 4, 10),
              lambda: P.test_ring_slots_equal_concatenate_then_truncate(3, 2, 3, 12)]


# ------------------------------------------------------------------------------------------
# softmax / attention mutants
# ------------------------------------------------------------------------------------------

def attention_missing_scale(q, k, v, scale):
    return _attention_f64(q, k, v, 1.0)


def attention_keys_as_values(q, k, v, scale):
    return _attention_f64(q, k, k, scale)


def attention_normalised_over_queries(q, k, v, scale):
    s = scale * np.asarray(q, np.float64) @ np.asarray(k, np.float64).T
    e = np.exp(s - s.max(axis=0, keepdims=True))
    p = e / e.sum(axis=0, keepdims=True)
    return p @ np.asarray(v, np.float64), np.log(np.exp(s).sum(axis=1))


def attention_lse_without_max(q, k, v, scale):
    out, lse = _attention_f64(q, k, v, scale)
    s = scale * np.asarray(q, np.float64) @ np.asarray(k, np.float64).T
    return out, lse - s.max(axis=1)


def softmax_lse_without_max(s):
    p, lse = _softmax(s)
    return p, lse - float(np.max(s))


ATTENTION_PINS = [P.test_attention_brute_force_tiny, P.test_attention_closed_forms]


# ------------------------------------------------------------------------------------------
# motion mutants
# ------------------------------------------------------------------------------------------

def ssd_absolute_difference(frames):
    f = np.asarray(frames, np.int64)
    return np.abs(f[:, 1:] - f[:, :-1]).reshape(f.shape[0], f.shape[1] - 1, -1).sum(-1).astype(np.uint64)


def ssd_against_first_frame(frames):
    f = np.asarray(frames, np.int64)
    d = f[:, 1:] - f[:, :1]
    return (d * d).reshape(f.shape[0], f.shape[1] - 1, -1).sum(-1).astype(np.uint64)


def ssd_first_channel_only(frames):
    f = np.asarray(frames, np.int64)
    d = (f[:, 1:] - f[:, :-1])[..., :1]
    return (d * d).reshape(f.shape[0], f.shape[1] - 1, -1).sum(-1).astype(np.uint64)


MOTION_PINS = [P.test_motion_identical_frames_and_symmetry,
               lambda: P.test_motion_shifted_ramp_closed_form(1, 5),
               lambda: P.test_motion_shifted_ramp_closed_form(3, 7)]


# ------------------------------------------------------------------------------------------
# next-row mutants: refresh re-rotation, sink update, noise map, projection
# ------------------------------------------------------------------------------------------

def _rerotate_with(shift_sign=-1, all_axes=False, lower_tpos=True):
    def refresh_rerotate(self, chunk):
        w = self.w
        R = w.refresh_chunks
        if not (R > 0 and chunk > 0 and chunk % R == 0):
            return False
        shift = w.chunk_frames * R
        for e in self.cache.entries[w.sink_frames:]:
            if 0 <= e[0] < chunk * w.chunk_frames:
                n = e[2].shape[0]
                z = np.zeros(n, np.int64)
                d = np.full(n, shift_sign * shift, np.int64)
                e[2] = _rope_spec(e[2], d, d if all_axes else z, d if all_axes else z, w.rope_t, w.rope_h,
                                  w.rope_w, w.rope_base)
                if lower_tpos:
                    e[1] -= shift
        return True
    return refresh_rerotate


def sink_update_oldest(self):
    fs = self.w.sink_frames
    first = self.cache.entries[fs:2 * fs]
    self.cache.entries[:fs] = [[e[0], e[1], e[2].copy(), e[3].copy()] for e in first]


def sink_update_aliased(self):
    fs = self.w.sink_frames
    self.cache.entries[:fs] = [[e[0], e[1], e[2], e[3]] for e in self.cache.entries[-fs:]]


def noise_direction_inverted(m, m_lo, m_hi, out_lo, out_hi, ema, more_noise_when_fast, state=None):
    return _noise(m, m_lo, m_hi, out_lo, out_hi, ema, 1 - int(more_noise_when_fast), state)


def noise_state_ignored(m, m_lo, m_hi, out_lo, out_hi, ema, more_noise_when_fast, state=None):
    return _noise(m, m_lo, m_hi, out_lo, out_hi, ema, more_noise_when_fast, None)


def qkv_bias_twice(x_bits, w_bits, bias=None):
    y = _qkv_project(x_bits, w_bits, bias)
    return y if bias is None else y + np.asarray(bias, np.float32).astype(np.float64)[None, :]


def qkv_bias_dropped(x_bits, w_bits, bias=None):
    return _qkv_project(x_bits, w_bits, None)


REROTATE_PINS = [PN.test_stream_tpos_after_resets_equals_continuous_tpos_minus_shifts,
                 PN.test_stream_rerotated_keys_keep_scores_continuous]
NOISE_PINS = [lambda: PN.test_noise_map_monotone_endpoints_and_direction(0),
              lambda: PN.test_noise_map_monotone_endpoints_and_direction(1),
              PN.test_noise_smoothing_closed_form_and_state_carry]

NEXT_MUTANTS = [
    ("rerotation: keys turned forward instead of back", oracle.StreamOracle, "refresh_rerotate",
     _rerotate_with(shift_sign=+1), REROTATE_PINS),
    ("rerotation: all three axes turned", oracle.StreamOracle, "refresh_rerotate",
     _rerotate_with(all_axes=True), REROTATE_PINS),
    ("rerotation: time index not lowered", oracle.StreamOracle, "refresh_rerotate",
     _rerotate_with(lower_tpos=False), REROTATE_PINS),
    ("sink update: oldest window frames copied", oracle.StreamOracle, "sink_update", sink_update_oldest,
     [PN.test_sink_update_copies_the_last_frames]),
    ("sink update: arrays shared instead of copied", oracle.StreamOracle, "sink_update", sink_update_aliased,
     [PN.test_sink_update_copies_the_last_frames]),
    ("noise: direction flag inverted", oracle, "noise", noise_direction_inverted, NOISE_PINS),
    ("noise: smoothing state not carried", oracle, "noise", noise_state_ignored, NOISE_PINS),
    ("projection: bias added twice", oracle, "qkv_project", qkv_bias_twice, [PN.test_qkv_projection_brute_force]),
    ("projection: bias dropped", oracle, "qkv_project", qkv_bias_dropped, [PN.test_qkv_projection_brute_force]),
]


@pytest.mark.parametrize("name,owner,attr,mutant,pins", NEXT_MUTANTS, ids=[m[0] for m in NEXT_MUTANTS])
def test_next_row_pins_reject_mutant(monkeypatch, name, owner, attr, mutant, pins):
    monkeypatch.setattr(owner, attr, mutant)
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, "no pin caught the mutant: " + name


MUTANTS = [
    ("rope: negated angle", "rope_ideal", rope_negated_angle, ROPE_PINS),
    ("rope: h and w positions swapped", "rope_ideal", rope_h_w_swapped, ROPE_PINS),
    ("rope: frequency exponent missing its factor 2", "rope_ideal", rope_missing_factor_two, ROPE_PINS),
    ("rope: pairs (j, j + d/2) instead of adjacent", "rope_ideal", rope_half_split_pairs, ROPE_PINS),
    ("rope: the -y sin term dropped", "rope_ideal", rope_dropped_term, ROPE_PINS),
    ("positions: offset never reset", "chunk_positions", positions_never_reset, POSITION_PINS),
    ("positions: reset period off by one", "chunk_positions", positions_reset_period_off_by_one, POSITION_PINS),
    ("positions: tokens column-major in a frame", "chunk_positions", positions_h_w_swapped, POSITION_PINS),
    ("positions: cache frame number off by one", "chunk_positions", positions_frame_number_off_by_one,
     POSITION_PINS),
    ("cache: ring index off by one", "slot_of_frame", slot_ring_off_by_one, CACHE_PINS),
    ("cache: sink slots taken into the ring", "slot_of_frame", slot_sink_in_ring, CACHE_PINS),
    ("cache: list truncation evicts the sink", "FrameListCache", CacheForgetsSink, CACHE_PINS),
    ("attention: softmax scale missing", "attention_f64", attention_missing_scale, ATTENTION_PINS),
    ("attention: keys used as values", "attention_f64", attention_keys_as_values, ATTENTION_PINS),
    ("attention: normalised over queries", "attention_f64", attention_normalised_over_queries, ATTENTION_PINS),
    ("attention: log-sum-exp without the max", "attention_f64", attention_lse_without_max, ATTENTION_PINS),
    ("softmax: log-sum-exp without the max", "softmax", softmax_lse_without_max,
     [P.test_softmax_rows_sum_to_one_and_match_scipy]),
    ("motion: absolute instead of squared difference", "motion_ssd", ssd_absolute_difference, MOTION_PINS),
    ("motion: every frame against the first", "motion_ssd", ssd_against_first_frame, MOTION_PINS),
    ("motion: one colour channel only", "motion_ssd", ssd_first_channel_only, MOTION_PINS),
]


@pytest.mark.parametrize("name,target,mutant,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(monkeypatch, name, target, mutant, pins):
    monkeypatch.setattr(oracle, target, mutant)
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, "no pin caught the mutant: " + name


def test_unmutated_oracle_passes_the_same_pins():
    for pins in (ROPE_PINS, POSITION_PINS, CACHE_PINS, ATTENTION_PINS, MOTION_PINS, REROTATE_PINS, NOISE_PINS):
        for pin in pins:
            pin()
