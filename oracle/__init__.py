"""Oracle: a plain, slow, obviously-correct CPU model of the streaming chunk-attention path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU-baseline leg
may import this package.  It shares no code with the CUDA library and never calls it.

What each function follows (pages are cited by title and section):

* chunk_positions -- "Accelerating Video Generation Inference with Sequential-Parallel 3D
  Positional Encoding Using a Global Time Index", technical summary 2(나): each generated block
  computes its tokens' time index locally from the block's start frame (the global time
  index), so no gather of the whole sequence is needed.  The periodic offset reset of
  "StreamDiffusionV2" (review page, section 三, "RoPE 刷新"; technical summary section 2 part A item 2) is read as: the
  chunk offset inside the time index restarts every R chunks, t = S + F*(c mod R) + i.
* FrameListCache -- the same review page, section 三 ("Sink Token 引导的滚动 KV 缓存"): the KV of
  the first frames is kept as a sink, and a fixed-size window of the most recent frames rolls.
  Modelled literally as a list: append the chunk's frames, then keep the first F_s entries and
  the last W of the rest (concatenate-then-truncate with the sink kept).
* ring_pointer_slots -- an explicit ring buffer with a wrapping write pointer, used to pin the
  closed-form slot of a frame.
* rope_spec / rope_ideal -- 3D RoPE over (t, h, w) segments (C code, see sdv2_oracle.c).
* attention -- softmax(q k^T / sqrt(D)) v over every retained key, fp64.
* motion_ssd -- squared L2 distance of adjacent frames, exact integers ("L2 运动估计").
* StreamOracle.refresh_rerotate -- second reading of the RoPE refresh: at a refresh chunk the
  window frames' keys are turned back by F*R on the time axis (rope_spec with positions
  (-F*R, 0, 0)), and their time index decreases by F*R.
* StreamOracle.sink_update -- reading of "sink tokens updated from recent visual context": the
  sink entries become copies of the last F_s appended frames.
* qkv_project -- the QKV projection W x + bias in fp64 (numpy's matmul as the product
  primitive), for the fused projection + Causal-RoPE path of the Causal-RoPE page, technical
  summary 2(다); its output is rotated with rope_ideal.
* noise -- the motion-to-noise-rate map.  PARITY UNPINNED with respect to the pages: they give
  no formula and disagree on its direction (technical summary section 2 part A item 3 vs review page section 三); the
  map is a declared reading, pinned only to its own stated properties (monotone, end points,
  direction flag, smoothing closed form).
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

_LIB = None


def lib():
    """The oracle's compiled C library (built on first use with gcc)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, u64, dbl, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
        L.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16_ref.restype = ctypes.c_uint16
        L.orc_f32_to_bf16_ref.argtypes = [ctypes.c_float]
        L.orc_bf16_mismatches.restype = i64
        L.orc_bf16_mismatches.argtypes = [u64, u64]
        L.orc_f32_to_bf16_array.argtypes = [vp, vp, i64]
        L.orc_rope_omega.restype = dbl
        L.orc_rope_omega.argtypes = [i32, i32, dbl]
        L.orc_rope_cos_sin_f32.argtypes = [i64, i32, i32, dbl, vp, vp]
        L.orc_rope_spec.argtypes = [vp, vp, i64, i32, i32, i32, dbl, vp, vp, vp]
        L.orc_rope_ideal.argtypes = [vp, vp, i64, i32, i32, i32, dbl, vp, vp, vp]
        L.orc_softmax.restype = dbl
        L.orc_softmax.argtypes = [vp, i64, vp]
        L.orc_attention_f64.argtypes = [vp, i64, vp, vp, i64, i32, dbl, vp, vp]
        L.orc_attention_bf16.argtypes = [vp, vp, i64, vp, vp, i64, i32, dbl, vp, vp]
        L.orc_ssd_u8.restype = u64
        L.orc_ssd_u8.argtypes = [vp, vp, i64]
        L.orc_motion_ssd.argtypes = [vp, i64, i64, i64, vp]
        L.orc_noise.argtypes = [vp, i64, i64, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                ctypes.c_float, i32, vp, vp]
        L.orc_num_threads.restype = i32
        L.orc_set_num_threads.argtypes = [i32]
        _LIB = L
    return _LIB


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ------------------------------------------------------------------------------------------
# bf16
# ------------------------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_p(x), _p(y), x.size)
    return y


# ------------------------------------------------------------------------------------------
# positions, slots, cache
# ------------------------------------------------------------------------------------------

def chunk_positions(start_frame: int, chunk: int, chunk_frames: int, grid_h: int, grid_w: int,
                    refresh_chunks: int):
    """Positions of the F*HW tokens of chunk c of a stream that starts at global frame S.

    Token n lies in frame i = n // HW of the chunk, at grid row (n % HW) // gw and column
    n % gw (tokens row-major inside a frame).  Returns int64 arrays (t, h, w, frame) where t is
    the RoPE time index S + F*(c mod R) + i (R = 0: S + F*c + i) and frame is the
    stream-relative frame number c*F + i that names the frame in the cache."""
    hw = grid_h * grid_w
    n = np.arange(chunk_frames * hw, dtype=np.int64)
    i = n // hw
    r = n % hw
    h = r // grid_w
    w = r % grid_w
    frame = chunk * chunk_frames + i
    c_eff = chunk % refresh_chunks if refresh_chunks > 0 else chunk
    t = start_frame + c_eff * chunk_frames + i
    return t, h, w, frame


def slot_of_frame(frame: int, sink_frames: int, window_frames: int) -> int:
    """Closed-form cache slot of stream-relative frame f: the sink keeps frames 0..F_s-1 in
    slots 0..F_s-1; later frames cycle through the W window slots after them."""
    if frame < sink_frames:
        return frame
    return sink_frames + (frame - sink_frames) % window_frames


def ring_pointer_slots(n_frames: int, sink_frames: int, window_frames: int):
    """Slots given to frames 0..n-1 by a ring buffer with a write pointer (no modular formula):
    the sink slots are filled in order; afterwards a pointer walks the window slots and jumps
    back to the first window slot after the last one."""
    out = []
    ptr = sink_frames
    for f in range(n_frames):
        if f < sink_frames:
            out.append(f)
        else:
            out.append(ptr)
            ptr += 1
            if ptr == sink_frames + window_frames:
                ptr = sink_frames
    return out


class FrameListCache:
    """Explicit list model of one stream's (one layer's) KV cache.

    Each entry is one whole latent frame: (frame, tpos, k_rot[HW][H][D], v[HW][H][D]) as bf16
    bits.  Appending a frame concatenates it to the list and truncates: the first F_s entries
    (the sink) stay, and of the rest only the last W remain.  Appending a frame that is already
    retained replaces its contents (a later denoise step of the same chunk)."""

    def __init__(self, sink_frames: int, window_frames: int):
        self.sink_frames = sink_frames
        self.window_frames = window_frames
        self.entries = []
        self.appended = 0          # frames ever appended (distinct frame numbers)

    def append(self, frame: int, tpos: int, k, v):
        # A frame that is already retained is replaced where it lives: sink frames (frame < F_s)
        # in the sink part, later frames in the window part.  (After a sink update the sink
        # holds copies of window frames; a later denoise step re-appends the window original.)
        home = self.entries[:self.sink_frames] if frame < self.sink_frames else self.entries[self.sink_frames:]
        for e in home:
            if e[0] == frame:
                e[1], e[2], e[3] = tpos, k, v
                return
        if frame != self.appended:
            raise ValueError("frames must be appended in order (got %d, expected %d)"
                             % (frame, self.appended))
        self.entries.append([frame, tpos, k, v])
        self.appended += 1
        sink = self.entries[:self.sink_frames]
        rest = self.entries[self.sink_frames:]
        if len(rest) > self.window_frames:
            rest = rest[len(rest) - self.window_frames:]
        self.entries = sink + rest

    def frames(self):
        return [e[0] for e in self.entries]

    def keys(self, head: int) -> np.ndarray:
        """Retained keys of one head in list order, [n_frames*HW][D] bf16 bits."""
        return np.ascontiguousarray(np.concatenate([e[2][:, head, :] for e in self.entries], 0))

    def values(self, head: int) -> np.ndarray:
        return np.ascontiguousarray(np.concatenate([e[3][:, head, :] for e in self.entries], 0))


# ------------------------------------------------------------------------------------------
# RoPE
# ------------------------------------------------------------------------------------------

def rope_spec(x_bits: np.ndarray, tpos, hpos, wpos, dt: int, dh: int, dw: int, base: float):
    """bf16 3D RoPE of vectors x[..., D] (bf16 bits) whose leading index n has positions
    tpos[n], hpos[n], wpos[n]; any further axes between n and D (e.g. heads) share n's
    position."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    D = dt + dh + dw
    assert x.shape[-1] == D
    n0 = x.shape[0]
    per = int(np.prod(x.shape[1:-1])) if x.ndim > 2 else 1
    rep = lambda a: np.ascontiguousarray(np.repeat(np.asarray(a, dtype=np.int64), per))
    t, h, w = rep(tpos), rep(hpos), rep(wpos)
    assert t.size == n0 * per
    y = np.empty_like(x)
    lib().orc_rope_spec(_p(x), _p(y), n0 * per, dt, dh, dw, float(base), _p(t), _p(h), _p(w))
    return y


def rope_ideal(x: np.ndarray, tpos, hpos, wpos, dt: int, dh: int, dw: int, base: float):
    """fp64 3D RoPE with no rounding; x[n][D] fp64, positions fp64 per n."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    n = x.shape[0]
    y = np.empty_like(x)
    t = np.ascontiguousarray(np.broadcast_to(np.asarray(tpos, np.float64), (n,)))
    h = np.ascontiguousarray(np.broadcast_to(np.asarray(hpos, np.float64), (n,)))
    w = np.ascontiguousarray(np.broadcast_to(np.asarray(wpos, np.float64), (n,)))
    lib().orc_rope_ideal(_p(x), _p(y), n, dt, dh, dw, float(base), _p(t), _p(h), _p(w))
    return y


def rope_cos_sin_f32(pos: int, j: int, d_axis: int, base: float):
    c = ctypes.c_float()
    s = ctypes.c_float()
    lib().orc_rope_cos_sin_f32(int(pos), j, d_axis, float(base), ctypes.byref(c), ctypes.byref(s))
    return c.value, s.value


def rope_omega(j: int, d_axis: int, base: float) -> float:
    return lib().orc_rope_omega(j, d_axis, float(base))


# ------------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------------

def softmax(s: np.ndarray):
    s = np.ascontiguousarray(s, dtype=np.float64)
    p = np.empty_like(s)
    lse = lib().orc_softmax(_p(s), s.size, _p(p))
    return p, lse


def attention_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """softmax(scale * q k^T) v in fp64; q [nq][D], k, v [nkv][D]. Returns (out, lse)."""
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    nq, D = q.shape
    out = np.empty((nq, D), np.float64)
    lse = np.empty(nq, np.float64)
    lib().orc_attention_f64(_p(q), nq, _p(k), _p(v), k.shape[0], D, float(scale), _p(out), _p(lse))
    return out, lse


def attention_bf16(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, scale: float,
                   rows=None):
    """fp64 attention on bf16 inputs (widened exactly).  q [nq][D]; rows selects query rows."""
    q = np.ascontiguousarray(q_bits, np.uint16)
    k = np.ascontiguousarray(k_bits, np.uint16)
    v = np.ascontiguousarray(v_bits, np.uint16)
    D = q.shape[-1]
    if rows is None:
        rows = np.arange(q.shape[0], dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, D), np.float64)
    lse = np.empty(rows.size, np.float64)
    lib().orc_attention_bf16(_p(q), _p(rows), rows.size, _p(k), _p(v), k.shape[0], D, float(scale),
                             _p(out), _p(lse))
    return out, lse


# ------------------------------------------------------------------------------------------
# one stream, chunk by chunk
# ------------------------------------------------------------------------------------------

class StreamOracle:
    """One stream of the hot path for one layer: Causal-RoPE, cache append, chunk attention."""

    def __init__(self, w, start_frame: int):
        self.w = w
        self.start_frame = int(start_frame)
        self.cache = FrameListCache(w.sink_frames, w.window_frames)

    def append_chunk(self, chunk: int, q_bits, k_bits, v_bits):
        """q, k, v: [Nq][H][D] bf16 bits.  Returns q_rot [Nq][H][D] and appends k_rot, v."""
        w = self.w
        t, h, ww, frame = chunk_positions(self.start_frame, chunk, w.chunk_frames, w.grid_h,
                                          w.grid_w, w.refresh_chunks)
        q_rot = rope_spec(q_bits, t, h, ww, w.rope_t, w.rope_h, w.rope_w, w.rope_base)
        k_rot = rope_spec(k_bits, t, h, ww, w.rope_t, w.rope_h, w.rope_w, w.rope_base)
        hw = w.hw
        for i in range(w.chunk_frames):
            sl = slice(i * hw, (i + 1) * hw)
            self.cache.append(int(frame[i * hw]), int(t[i * hw]), k_rot[sl].copy(),
                              np.ascontiguousarray(v_bits[sl]).copy())
        return q_rot

    def refresh_rerotate(self, chunk: int):
        """At a refresh chunk (R > 0, c > 0, c mod R == 0), before the chunk is appended: every
        window entry of an earlier chunk has its keys turned back by F*R on the time axis and
        its time index lowered by F*R.  Returns True if anything changed."""
        w = self.w
        R = w.refresh_chunks
        if not (R > 0 and chunk > 0 and chunk % R == 0):
            return False
        shift = w.chunk_frames * R
        for e in self.cache.entries[w.sink_frames:]:
            if 0 <= e[0] < chunk * w.chunk_frames:
                n = e[2].shape[0]
                z = np.zeros(n, np.int64)
                e[2] = rope_spec(e[2], np.full(n, -shift, np.int64), z, z, w.rope_t, w.rope_h, w.rope_w,
                                 w.rope_base)
                e[1] = e[1] - shift
        return True

    def sink_update(self):
        """Replace the sink entries by copies of the last F_s appended frames."""
        fs = self.w.sink_frames
        if fs == 0:
            return
        last = self.cache.entries[-fs:]
        assert len(self.cache.entries) >= 2 * fs and all(e[0] >= fs for e in last)
        self.cache.entries[:fs] = [[e[0], e[1], e[2].copy(), e[3].copy()] for e in last]

    def attend(self, q_rot, head: int, rows=None, scale=None):
        """Attention of query rows of q_rot[:, head, :] to every retained key of that head."""
        D = self.w.head_dim
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        q = np.ascontiguousarray(q_rot[:, head, :])
        return attention_bf16(q, self.cache.keys(head), self.cache.values(head), scale, rows)


# ------------------------------------------------------------------------------------------
# motion
# ------------------------------------------------------------------------------------------

def motion_ssd(frames: np.ndarray) -> np.ndarray:
    """frames [B][T+1][...] uint8 -> ssd [B][T] uint64 (frame t+1 against frame t)."""
    f = np.ascontiguousarray(frames, np.uint8)
    nb, t1 = f.shape[0], f.shape[1]
    npix = int(np.prod(f.shape[2:]))
    out = np.empty((nb, t1 - 1), np.uint64)
    lib().orc_motion_ssd(_p(f), nb, t1 - 1, npix, _p(out))
    return out


def qkv_project(x_bits: np.ndarray, w_bits: np.ndarray, bias=None) -> np.ndarray:
    """fp64 [M][N] = x [M][C] (bf16 bits) times w [N][C]^T (bf16 bits) plus bias [N] (fp32)."""
    x = bf16_to_f32(x_bits).astype(np.float64)
    w = bf16_to_f32(w_bits).astype(np.float64)
    y = x @ w.T
    if bias is not None:
        y = y + np.asarray(bias, np.float32).astype(np.float64)[None, :]
    return y


def noise(m: np.ndarray, m_lo, m_hi, out_lo, out_hi, ema, more_noise_when_fast, state=None):
    """Noise rate per frame (see orc_noise).  m: [B][T] float32; state: [B] float32 or None
    (updated in place).  Returns rate [B][T] float32."""
    m = np.ascontiguousarray(m, np.float32)
    B, T = m.shape
    rate = np.empty_like(m)
    st = None if state is None else state
    if st is not None:
        assert st.dtype == np.float32 and st.flags["C_CONTIGUOUS"]
    lib().orc_noise(_p(m), B, T, m_lo, m_hi, out_lo, out_hi, ema, int(more_noise_when_fast),
                    None if st is None else _p(st), _p(rate))
    return rate


def motion_rms(ssd: np.ndarray, npix: int) -> np.ndarray:
    """RMS pixel difference sqrt(SSD / N) in fp64."""
    return np.sqrt(np.asarray(ssd, np.float64) / float(npix))
