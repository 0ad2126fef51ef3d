"""Seeded random inputs.  No arithmetic of the method lives here."""
import numpy as np
import torch


def _seed(*parts: int) -> int:
    """A stable 63-bit seed from integers (FNV-1a over their decimal text)."""
    h = 0xcbf29ce484222325
    for ch in ",".join(str(int(p)) for p in parts).encode():
        h ^= ch
        h = (h * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def qkv_chunk_host(w, batch: int, chunk: int, layer: int = 0, step: int = 0, seed_offset: int = 0,
                   same_streams: bool = False):
    """q, k, v of one chunk as CPU torch bf16 tensors of shape [B][F*HW][H][D].

    Values are N(0, 1) drawn in fp32 and rounded to bf16 by torch.  With same_streams every
    stream receives identical data (the shift-invariance case)."""
    g = torch.Generator().manual_seed(_seed(w.seed, seed_offset, layer, chunk, step))
    nb = 1 if same_streams else batch
    shape = (nb, w.nq, w.heads, w.head_dim)
    out = []
    for _ in range(3):
        t = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
        if same_streams:
            t = t.expand(batch, *shape[1:]).contiguous()
        out.append(t)
    return tuple(out)


def qkv_chunk_bits(w, batch: int, chunk: int, **kw):
    """Same as qkv_chunk_host, as numpy uint16 arrays holding the bf16 bit patterns."""
    return tuple(t.view(torch.int16).numpy().view(np.uint16) for t in qkv_chunk_host(w, batch, chunk, **kw))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact: the bf16 bits are the top half of the fp32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def motion_frames_host(batch: int, frames: int, hp: int, wp: int, ch: int, seed: int,
                       max_speed: int = 16, noise_sigma: float = 4.0, device="cpu") -> torch.Tensor:
    """Video frames [B][frames][hp][wp][ch] uint8.

    Per stream: a smooth texture (uniform noise on a grid 1/16 of the frame, bilinearly
    upsampled to the frame size, range 0..255), moved each frame by an integer displacement
    whose per-frame speed in x and in y follows a random walk clipped to [0, max_speed] pixels;
    then Gaussian noise of the given sigma is added and the result is rounded and clamped to
    0..255.  The motion is a cyclic shift, so the frame content stays defined everywhere."""
    out = torch.empty((batch, frames, hp, wp, ch), dtype=torch.uint8, device=device)
    for b in range(batch):
        g = torch.Generator().manual_seed(_seed(seed, b, 7))
        coarse = torch.rand((1, ch, max(2, hp // 16), max(2, wp // 16)), generator=g) * 255.0
        tex = torch.nn.functional.interpolate(coarse, size=(hp, wp), mode="bilinear",
                                              align_corners=False)[0].permute(1, 2, 0)
        tex = tex.to(device)
        steps = torch.randint(-2, 3, (frames, 2), generator=g)
        speed = torch.zeros(2, dtype=torch.int64)
        pos = torch.zeros(2, dtype=torch.int64)
        gd = torch.Generator(device=device).manual_seed(_seed(seed, b, 11))
        for t in range(frames):
            if t > 0:
                speed = (speed + steps[t]).clamp(0, max_speed)
                pos = pos + speed
            shifted = torch.roll(tex, shifts=(int(pos[0]) % hp, int(pos[1]) % wp), dims=(0, 1))
            noise = torch.randn(shifted.shape, generator=gd, device=device) * noise_sigma
            out[b, t] = (shifted + noise).round().clamp(0, 255).to(torch.uint8)
    return out
