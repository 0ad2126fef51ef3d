"""Named workloads: shapes, seeds and stream offsets only.

The shapes follow the Wan-style DiT that the StreamDiffusionV2 review page names in
"六、实现细节" (Wan 2.1 1.3B and Wan 2.2 14B at 480p = 832x480 and 720p): a latent grid of
(H/16) x (W/16) tokens per latent frame, 12 heads (hidden 1536) for 1.3B and 40 heads
(hidden 5120) for 14B, head_dim 128, chunks of 3 latent frames, a sink of one chunk and a
rolling window that, together with the sink, spans 21 latent frames.
"""
from dataclasses import dataclass, field
from typing import List, Optional


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int            # independent streams B
    heads: int            # H
    head_dim: int         # D
    rope_t: int           # head dims given to the time axis
    rope_h: int           # head dims given to the height axis
    rope_w: int           # head dims given to the width axis
    rope_base: float
    grid_h: int           # latent tokens per frame along height
    grid_w: int           # latent tokens per frame along width
    chunk_frames: int     # F, latent frames per chunk
    sink_frames: int      # F_s, pinned sink frames
    window_frames: int    # W, rolling window frames (includes the current chunk)
    refresh_chunks: int   # R, RoPE offset reset period in chunks (0 = never)
    chunks: int           # chunks streamed
    layers: int           # DiT layers (one KV cache each)
    denoise_steps: int    # denoise steps per chunk (each re-runs every layer)
    seed: int
    start_frames: List[int] = field(default_factory=lambda: [0])
    motion_frame_shape: Optional[tuple] = None   # (Hp, Wp, C) of the pixel frames, if any

    @property
    def hw(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def nq(self) -> int:
        return self.chunk_frames * self.hw

    @property
    def slots(self) -> int:
        return self.sink_frames + self.window_frames


_COMMON = dict(head_dim=128, rope_t=44, rope_h=42, rope_w=42, rope_base=10000.0)

WORKLOADS = {
    # Tiny stream: full oracle parity at every chunk; the window (4 frames) is not a multiple of
    # the chunk (3 frames), so the ring wraps in the middle of a chunk.
    "tiny": Workload(name="tiny", batch=1, heads=2, grid_h=4, grid_w=6, chunk_frames=3,
                     sink_frames=3, window_frames=4, refresh_chunks=0, chunks=10, layers=1,
                     denoise_steps=1, seed=1, **_COMMON),
    # Wan-1.3B-shaped 480p: 832x480 pixels -> 52x30 latent tokens per frame.
    "wan13b_480p": Workload(name="wan13b_480p", batch=1, heads=12, grid_h=30, grid_w=52,
                            chunk_frames=3, sink_frames=3, window_frames=18, refresh_chunks=0,
                            chunks=40, layers=30, denoise_steps=2, seed=2, **_COMMON),
    # Wan-1.3B-shaped 720p: 1280x720 pixels -> 80x45 latent tokens per frame.
    "wan13b_720p": Workload(name="wan13b_720p", batch=1, heads=12, grid_h=45, grid_w=80,
                            chunk_frames=3, sink_frames=3, window_frames=18, refresh_chunks=0,
                            chunks=20, layers=30, denoise_steps=2, seed=3, **_COMMON),
    # Wan-14B-shaped 480p: 40 heads x 128 (hidden 5120).
    "wan14b_480p": Workload(name="wan14b_480p", batch=1, heads=40, grid_h=30, grid_w=52,
                            chunk_frames=3, sink_frames=3, window_frames=18, refresh_chunks=0,
                            chunks=20, layers=40, denoise_steps=2, seed=4, **_COMMON),
    # Four independent 1.3B-480p streams with distinct global start offsets, RoPE refresh every
    # 64 chunks, and per-frame L2 motion on 480x832x3 uint8 frames.
    "stream_batch": Workload(name="stream_batch", batch=4, heads=12, grid_h=30, grid_w=52,
                             chunk_frames=3, sink_frames=3, window_frames=18, refresh_chunks=64,
                             chunks=500, layers=30, denoise_steps=2, seed=5,
                             start_frames=[0, 1000, 10000, 100000],
                             motion_frame_shape=(480, 832, 3), **_COMMON),
}


def stream_config_dict(w: Workload, batch: Optional[int] = None, qkv_token_stride: int = 0) -> dict:
    """Fields of the library's stream configuration struct for workload w."""
    return dict(batch=w.batch if batch is None else batch, heads=w.heads, head_dim=w.head_dim,
                rope_t=w.rope_t, rope_h=w.rope_h, rope_w=w.rope_w, rope_base=w.rope_base,
                grid_h=w.grid_h, grid_w=w.grid_w, chunk_frames=w.chunk_frames,
                sink_frames=w.sink_frames, window_frames=w.window_frames,
                refresh_chunks=w.refresh_chunks, qkv_token_stride=qkv_token_stride)
