"""Device buffers for a stream batch, allocated with torch, and the per-layer call sequence.

A StreamSession owns the workspace, one LayerCache (k, v, slot metadata) per DiT layer and the
q_rot / out buffers; layer_step() issues sdv2_rope_append_kv then sdv2_chunk_attention for one
layer of one denoise step.  Nothing here computes: it allocates and calls the library.
"""
import torch

from . import _binding as sd


class LayerCache:
    """One layer's KV cache: k and v [B][H][(F_s+W)*HW][D] bf16, meta [B][F_s+W][2] int64."""

    def __init__(self, cfg: sd.StreamConfig, device, stream=None):
        B, H, D = cfg.batch, cfg.heads, cfg.head_dim
        rows = cfg.slots * cfg.hw
        assert sd.cache_bytes(cfg) == B * H * rows * D * 2
        self.k = torch.empty((B, H, rows, D), dtype=torch.bfloat16, device=device)
        self.v = torch.empty((B, H, rows, D), dtype=torch.bfloat16, device=device)
        self.meta = torch.empty((B, cfg.slots, 2), dtype=torch.int64, device=device)
        sd.cache_reset(cfg, self.k, self.v, self.meta, stream)


class StreamSession:
    def __init__(self, cfg: sd.StreamConfig, layers: int, start_frames, device="cuda", stream=None):
        self.cfg = cfg
        self.start_frames = [int(s) for s in start_frames]
        B, H, D, nq = cfg.batch, cfg.heads, cfg.head_dim, cfg.nq
        self.ws = torch.zeros(sd.workspace_bytes(cfg), dtype=torch.uint8, device=device)
        sd.workspace_init(cfg, self.ws, stream)
        self.layers = [LayerCache(cfg, device, stream) for _ in range(layers)]
        self.q_rot = torch.empty((B, H, nq, D), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((B, nq, H, D), dtype=torch.bfloat16, device=device)

    def layer_step(self, layer: int, chunk_index, q, k, v, out=None, lse=None, stream=None):
        """Causal-RoPE + cache append, then chunk attention, for one layer.  q, k, v: [B][Nq][H][D]."""
        L = self.layers[layer]
        out = self.out if out is None else out
        sd.rope_append_kv(self.cfg, self.start_frames, chunk_index, q, k, v, self.q_rot, L.k, L.v, L.meta,
                          self.ws, stream)
        sd.chunk_attention(self.cfg, chunk_index, self.q_rot, L.k, L.v, out, self.ws, lse=lse, stream=stream)
        return out
