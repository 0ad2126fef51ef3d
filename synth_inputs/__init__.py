"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module holds no arithmetic of the method (no RoPE, no cache indexing, no attention,
no motion metric).  It only names the workloads and draws their random inputs:

* q, k, v activations: N(0, 1) in fp32, rounded to bf16 by torch's own conversion;
* video frames for the motion reduction: a smooth random texture moved by a random walk of
  integer displacements, plus Gaussian pixel noise, rounded and clamped to uint8.

Both the oracle side and the CUDA side receive the same arrays from here.
"""
from .workloads import WORKLOADS, Workload, stream_config_dict  # noqa: F401
from .generators import (  # noqa: F401
    qkv_chunk_host,
    qkv_chunk_bits,
    motion_frames_host,
    bf16_bits_to_f32,
)
