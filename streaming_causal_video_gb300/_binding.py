"""ctypes binding of libsdv2.so (argument marshalling only)."""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libsdv2.so")
_LIB = None

SDV2_OK = 0
STATUS_NAMES = {0: "SDV2_OK", 1: "SDV2_ERR_INVALID_ARG", 2: "SDV2_ERR_UNSUPPORTED", 3: "SDV2_ERR_CUDA",
                4: "SDV2_ERR_TIMEOUT"}

# Every symbol that include/sdv2.h declares.
EXPORTS = ["sdv2_workspace_bytes", "sdv2_cache_bytes", "sdv2_meta_bytes", "sdv2_visible_tokens",
           "sdv2_workspace_init", "sdv2_cache_reset", "sdv2_rope_append_kv", "sdv2_qkv_rope_append", "sdv2_chunk_attention",
           "sdv2_chunk_attention_noalloc", "sdv2_noalloc_check_device_error",
           "sdv2_motion_l2", "sdv2_rope_refresh_rerotate", "sdv2_sink_update", "sdv2_noise_from_motion",
           "sdv2_check_device_error", "sdv2_set_wait_timeout_ns",
           "sdv2_debug_drop_kv_tile", "sdv2_debug_set_kv_splits", "sdv2_last_kv_splits", "sdv2_debug_kv_schedule",
           "sdv2_status_string", "sdv2_last_error"]


class SDV2Error(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, STATUS_NAMES.get(status, str(status)), detail))


class NoiseCtl(ctypes.Structure):
    """Mirror of sdv2_noise_ctl."""
    _fields_ = [("motion_lo", ctypes.c_float), ("motion_hi", ctypes.c_float), ("rate_lo", ctypes.c_float),
                ("rate_hi", ctypes.c_float), ("ema", ctypes.c_float), ("more_noise_when_fast", ctypes.c_int32)]


class StreamConfig(ctypes.Structure):
    """Mirror of sdv2_stream_cfg."""
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_t", ctypes.c_int32), ("rope_h", ctypes.c_int32), ("rope_w", ctypes.c_int32),
                ("rope_base", ctypes.c_double), ("grid_h", ctypes.c_int32), ("grid_w", ctypes.c_int32),
                ("chunk_frames", ctypes.c_int32), ("sink_frames", ctypes.c_int32),
                ("window_frames", ctypes.c_int32), ("refresh_chunks", ctypes.c_int32),
                ("qkv_token_stride", ctypes.c_int64)]

    @classmethod
    def make(cls, **kw):
        c = cls()
        for k, v in kw.items():
            setattr(c, k, v)
        return c

    @property
    def hw(self):
        return self.grid_h * self.grid_w

    @property
    def nq(self):
        return self.chunk_frames * self.hw

    @property
    def slots(self):
        return self.sink_frames + self.window_frames


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded library.  Raises if libsdv2.so has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libsdv2.so is not built; run __graft_entry__.build() or "
                               "python -m streaming_causal_video_gb300.build")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, u64, i32, cfgp = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32,
                                   ctypes.POINTER(StreamConfig))
        i64p = ctypes.POINTER(ctypes.c_int64)
        for name in ("sdv2_workspace_bytes", "sdv2_cache_bytes", "sdv2_meta_bytes"):
            getattr(L, name).restype = ctypes.c_size_t
            getattr(L, name).argtypes = [cfgp]
        L.sdv2_visible_tokens.restype = i64
        L.sdv2_visible_tokens.argtypes = [cfgp, i64]
        L.sdv2_workspace_init.restype = ctypes.c_int
        L.sdv2_workspace_init.argtypes = [cfgp, vp, vp]
        L.sdv2_cache_reset.restype = ctypes.c_int
        L.sdv2_cache_reset.argtypes = [cfgp, vp, vp, vp, vp]
        L.sdv2_rope_append_kv.restype = ctypes.c_int
        L.sdv2_rope_append_kv.argtypes = [cfgp, i64p, i64p, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sdv2_qkv_rope_append.restype = ctypes.c_int
        L.sdv2_qkv_rope_append.argtypes = [cfgp, i64p, i64p, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp]
        L.sdv2_chunk_attention.restype = ctypes.c_int
        L.sdv2_chunk_attention.argtypes = [cfgp, i64p, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
        L.sdv2_chunk_attention_noalloc.restype = ctypes.c_int
        L.sdv2_chunk_attention_noalloc.argtypes = [cfgp, i64p, vp, vp, vp, ctypes.c_float, vp, vp, vp]
        L.sdv2_noalloc_check_device_error.restype = ctypes.c_int
        L.sdv2_noalloc_check_device_error.argtypes = [vp]
        L.sdv2_motion_l2.restype = ctypes.c_int
        L.sdv2_motion_l2.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp, vp]
        L.sdv2_rope_refresh_rerotate.restype = ctypes.c_int
        L.sdv2_rope_refresh_rerotate.argtypes = [cfgp, i64p, vp, vp, vp]
        L.sdv2_sink_update.restype = ctypes.c_int
        L.sdv2_sink_update.argtypes = [cfgp, i64p, ctypes.POINTER(ctypes.c_int32), vp, vp, vp, vp]
        L.sdv2_noise_from_motion.restype = ctypes.c_int
        L.sdv2_noise_from_motion.argtypes = [ctypes.POINTER(NoiseCtl), vp, i32, i64, vp, vp, vp]
        L.sdv2_check_device_error.restype = ctypes.c_int
        L.sdv2_check_device_error.argtypes = [vp, vp]
        L.sdv2_set_wait_timeout_ns.restype = None
        L.sdv2_set_wait_timeout_ns.argtypes = [u64]
        L.sdv2_debug_drop_kv_tile.restype = None
        L.sdv2_debug_drop_kv_tile.argtypes = [i64]
        L.sdv2_debug_set_kv_splits.restype = None
        L.sdv2_debug_set_kv_splits.argtypes = [i32]
        L.sdv2_last_kv_splits.restype = i32
        L.sdv2_last_kv_splits.argtypes = []
        L.sdv2_debug_kv_schedule.restype = i32
        L.sdv2_debug_kv_schedule.argtypes = [i64, i32, i32, ctypes.POINTER(ctypes.c_int32)]
        L.sdv2_status_string.restype = ctypes.c_char_p
        L.sdv2_status_string.argtypes = [ctypes.c_int]
        L.sdv2_last_error.restype = ctypes.c_char_p
        L.sdv2_last_error.argtypes = []
        _LIB = L
    return _LIB


def exported_symbols():
    """Names from include/sdv2.h that the loaded library resolves."""
    L = lib()
    return [n for n in EXPORTS if hasattr(L, n)]


def _check(status: int, where: str):
    if status != SDV2_OK:
        raise SDV2Error(status, where, lib().sdv2_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dev(t, name, nbytes):
    """Device pointer of a CUDA tensor, checked to reach at least `nbytes` bytes from its first
    element within its storage (views such as packed q/k/v slices pass).  Raw integer pointers
    and None pass through unchecked: the C ABI cannot see buffer sizes."""
    if t is None or isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    avail = t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()
    if avail < nbytes:
        raise ValueError("%s: %d bytes from its first element, the call touches %d" % (name, avail, nbytes))
    return t.data_ptr()


def _row_span(rows, stride, width, elem):
    """Bytes from the first element of `rows` rows `stride` elements apart, `width` used each."""
    return 0 if rows <= 0 else ((rows - 1) * stride + width) * elem


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i64_array(values, n):
    vals = [int(x) for x in values]
    if len(vals) != n:
        raise ValueError("expected %d values, got %d" % (n, len(vals)))
    return (ctypes.c_int64 * n)(*vals)


def workspace_bytes(cfg: StreamConfig) -> int:
    return lib().sdv2_workspace_bytes(ctypes.byref(cfg))


def cache_bytes(cfg: StreamConfig) -> int:
    return lib().sdv2_cache_bytes(ctypes.byref(cfg))


def meta_bytes(cfg: StreamConfig) -> int:
    return lib().sdv2_meta_bytes(ctypes.byref(cfg))


def visible_tokens(cfg: StreamConfig, chunk_index: int) -> int:
    return lib().sdv2_visible_tokens(ctypes.byref(cfg), int(chunk_index))


def workspace_init(cfg, ws, stream=None):
    _check(lib().sdv2_workspace_init(ctypes.byref(cfg), _dev(ws, "ws", workspace_bytes(cfg)), _stream(stream)),
           "sdv2_workspace_init")


def cache_reset(cfg, k_cache, v_cache, meta, stream=None):
    _, cb, mb, _, _ = _sizes(cfg)
    _check(lib().sdv2_cache_reset(ctypes.byref(cfg), _dev(k_cache, "k_cache", cb), _dev(v_cache, "v_cache", cb),
                                  _dev(meta, "meta", mb), _stream(stream)), "sdv2_cache_reset")


def _sizes(cfg):
    """Bytes each per-layer buffer spans: q_rot/out, caches, metadata, workspace, lse."""
    rows = max(cfg.batch, 0) * max(cfg.heads, 0) * cfg.nq          # (stream, head, query) rows
    return rows * 128 * 2, cache_bytes(cfg), meta_bytes(cfg), workspace_bytes(cfg), rows * 4


def rope_append_kv(cfg, start_frame, chunk_index, q, k, v, q_rot, k_cache, v_cache, meta, ws, stream=None):
    B = cfg.batch
    qo, cb, mb, wb, _ = _sizes(cfg)
    C = max(cfg.heads, 0) * 128
    span = _row_span(max(B, 0) * cfg.nq, cfg.qkv_token_stride or C, C, 2)
    _check(lib().sdv2_rope_append_kv(ctypes.byref(cfg), _i64_array(start_frame, B), _i64_array(chunk_index, B),
                                     _dev(q, "q", span), _dev(k, "k", span), _dev(v, "v", span),
                                     _dev(q_rot, "q_rot", qo), _dev(k_cache, "k_cache", cb),
                                     _dev(v_cache, "v_cache", cb), _dev(meta, "meta", mb), _dev(ws, "ws", wb),
                                     _stream(stream)), "sdv2_rope_append_kv")


def qkv_rope_append(cfg, start_frame, chunk_index, x, w_qkv, q_rot, k_cache, v_cache, meta, ws, bias=None,
                    x_token_stride=0, stream=None):
    """x: [B][Nq][H*D] bf16; w_qkv: [3*H*D][H*D] bf16; bias: fp32 [3*H*D] or None."""
    B = cfg.batch
    qo, cb, mb, wb, _ = _sizes(cfg)
    C = max(cfg.heads, 0) * 128
    span = _row_span(max(B, 0) * cfg.nq, int(x_token_stride) or C, C, 2)
    _check(lib().sdv2_qkv_rope_append(ctypes.byref(cfg), _i64_array(start_frame, B), _i64_array(chunk_index, B),
                                      _dev(x, "x", span), int(x_token_stride), _dev(w_qkv, "w_qkv", 3 * C * C * 2),
                                      _dev(bias, "bias", 3 * C * 4), _dev(q_rot, "q_rot", qo),
                                      _dev(k_cache, "k_cache", cb), _dev(v_cache, "v_cache", cb),
                                      _dev(meta, "meta", mb), _dev(ws, "ws", wb), _stream(stream)),
           "sdv2_qkv_rope_append")


def chunk_attention(cfg, chunk_index, q_rot, k_cache, v_cache, out, ws, lse=None, scale=0.0, stream=None):
    qo, cb, _, wb, lb = _sizes(cfg)
    _check(lib().sdv2_chunk_attention(ctypes.byref(cfg), _i64_array(chunk_index, cfg.batch),
                                      _dev(q_rot, "q_rot", qo), _dev(k_cache, "k_cache", cb),
                                      _dev(v_cache, "v_cache", cb), float(scale), _dev(out, "out", qo),
                                      _dev(lse, "lse", lb), _dev(ws, "ws", wb), _stream(stream)),
           "sdv2_chunk_attention")


def chunk_attention_noalloc(cfg, chunk_index, q_rot, k_cache, v_cache, out, lse=None, scale=0.0, stream=None):
    """sdv2_chunk_attention_noalloc: the same attention without a caller-owned workspace."""
    qo, cb, _, _, lb = _sizes(cfg)
    _check(lib().sdv2_chunk_attention_noalloc(ctypes.byref(cfg), _i64_array(chunk_index, cfg.batch),
                                              _dev(q_rot, "q_rot", qo), _dev(k_cache, "k_cache", cb),
                                              _dev(v_cache, "v_cache", cb), float(scale), _dev(out, "out", qo),
                                              _dev(lse, "lse", lb), _stream(stream)), "sdv2_chunk_attention_noalloc")


def noalloc_check_device_error(stream=None):
    """sdv2_noalloc_check_device_error: raises SDV2Error (status 4) after a timed-out no-alloc call."""
    _check(lib().sdv2_noalloc_check_device_error(_stream(stream)), "sdv2_noalloc_check_device_error")


def motion_l2(frames, ssd, m=None, stream=None):
    """frames: uint8 [B][T+1][Hp][Wp][C] on the device; ssd: uint64-sized [B][T]; m: fp32 [B][T]."""
    B, T1, Hp, Wp, C = frames.shape
    if not frames.is_contiguous():
        raise ValueError("frames must be contiguous")
    n = B * max(T1 - 1, 0)
    _check(lib().sdv2_motion_l2(_dev(frames, "frames", frames.numel()), B, T1 - 1, Hp, Wp, C, _dev(ssd, "ssd", n * 8),
                                _dev(m, "m", n * 4), _stream(stream)), "sdv2_motion_l2")


def rope_refresh_rerotate(cfg, chunk_index, k_cache, meta, stream=None):
    _, cb, mb, _, _ = _sizes(cfg)
    _check(lib().sdv2_rope_refresh_rerotate(ctypes.byref(cfg), _i64_array(chunk_index, cfg.batch),
                                            _dev(k_cache, "k_cache", cb), _dev(meta, "meta", mb), _stream(stream)),
           "sdv2_rope_refresh_rerotate")


def sink_update(cfg, chunk_index, update, k_cache, v_cache, meta, stream=None):
    upd = (ctypes.c_int32 * cfg.batch)(*[int(u) for u in update])
    _, cb, mb, _, _ = _sizes(cfg)
    _check(lib().sdv2_sink_update(ctypes.byref(cfg), _i64_array(chunk_index, cfg.batch), upd,
                                  _dev(k_cache, "k_cache", cb), _dev(v_cache, "v_cache", cb), _dev(meta, "meta", mb),
                                  _stream(stream)), "sdv2_sink_update")


def noise_from_motion(ctl, m, rate, state=None, stream=None):
    """m, rate: device fp32 [B][T]; state: device fp32 [B] or None."""
    B, T = m.shape
    _check(lib().sdv2_noise_from_motion(ctypes.byref(ctl), _dev(m, "m", B * T * 4), B, T, _dev(state, "state", B * 4),
                                        _dev(rate, "rate", B * T * 4), _stream(stream)), "sdv2_noise_from_motion")


def check_device_error(ws, stream=None):
    _check(lib().sdv2_check_device_error(_dev(ws, "ws", 16), _stream(stream)), "sdv2_check_device_error")


def set_wait_timeout_ns(ns: int):
    lib().sdv2_set_wait_timeout_ns(int(ns))


def debug_drop_kv_tile(tile: int):
    lib().sdv2_debug_drop_kv_tile(int(tile))


def debug_set_kv_splits(n: int):
    lib().sdv2_debug_set_kv_splits(int(n))


def debug_kv_schedule(items: int, min_tiles: int, sms: int):
    """(full_items, splits) of the attention's automatic schedule; host only."""
    full = ctypes.c_int32(0)
    sp = lib().sdv2_debug_kv_schedule(int(items), int(min_tiles), int(sms), ctypes.byref(full))
    if sp < 0:
        raise ValueError("invalid schedule arguments")
    return full.value, sp


def last_kv_splits() -> int:
    return lib().sdv2_last_kv_splits()
