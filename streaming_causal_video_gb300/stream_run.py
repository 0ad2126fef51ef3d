"""A whole streaming run through the library's public calls, timed chunk by chunk.

For every chunk of a stream batch, every denoise step and every DiT layer (one KV cache per
layer), the run issues sdv2_rope_append_kv then sdv2_chunk_attention, exactly as a model would.
CUDA events around each attention call give the attention time; events at chunk boundaries give
the path time (append + attention).  The first chunks attend to a cache that is still filling
(fewer visible keys); once sink and window are full every chunk costs the same, so warm-up and
steady state are reported separately.

Reported per run (one JSON line):
  run_pflop       sum over calls of 4 * H * D * Nq * Nkv(c) * B (the two GEMMs, no mask);
  attention_tflops  run_pflop / total attention time;
  t_path_s, latent_frames_per_s  path time of the timed chunks and chunks * F * B / t_path;
  warmup / steady  the same per group of chunks.
A long stream batch (hundreds of chunks) is timed on windows of chunks at full layers x steps;
the chunks between windows advance the stream state with one layer and one step (the cache
shapes depend only on the chunk index, so this does not change what the windows measure).

Run: python -m streaming_causal_video_gb300.stream_run [--workload NAME] [--chunks N]
"""
import argparse
import json
import os
import sys

import torch

from . import _binding as sd
from .layer import StreamSession

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
from synth_inputs import WORKLOADS, stream_config_dict  # noqa: E402

# timed windows for streams longer than this many chunks
LONG_STREAM = 100
WINDOWS = ((0, 10), (60, 70), (490, 500))


def timed_chunks(w, chunks):
    if chunks <= LONG_STREAM:
        return set(range(chunks))
    return {c for lo, hi in WINDOWS for c in range(lo, min(hi, chunks))}


def run(w, chunks=None, device="cuda"):
    chunks = w.chunks if chunks is None else chunks
    dev = torch.device(device)
    st = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(st)
    cfg = sd.StreamConfig.make(**stream_config_dict(w))
    sess = StreamSession(cfg, w.layers, w.start_frames, dev, st)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    shape = (w.batch, w.nq, w.heads, w.head_dim)
    qkv = [tuple(torch.randn(shape, generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
           for _ in range(w.layers)]
    steady_nkv = w.slots * w.hw
    timed = timed_chunks(w, chunks)

    def call(layer, c, ev=None):
        L = sess.layers[layer]
        q, k, v = qkv[layer]
        cidx = [c] * w.batch
        sd.rope_append_kv(cfg, w.start_frames, cidx, q, k, v, sess.q_rot, L.k, L.v, L.meta, sess.ws, st)
        if ev is not None:
            ev[0].record(st)
        sd.chunk_attention(cfg, cidx, sess.q_rot, L.k, L.v, sess.out, sess.ws, stream=st)
        if ev is not None:
            ev[1].record(st)

    # warm-up: a few calls on chunk 0 of layer 0, whose cache is then reset
    for _ in range(3):
        call(0, 0)
    sd.cache_reset(cfg, sess.layers[0].k, sess.layers[0].v, sess.layers[0].meta, st)
    st.synchronize()

    records = []   # (chunk, nkv, chunk start event, chunk end event, [(attn start, attn end)])
    for c in range(chunks):
        if c in timed:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            pairs = []
            e0.record(st)
            for _step in range(w.denoise_steps):
                for layer in range(w.layers):
                    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    call(layer, c, ev)
                    pairs.append(ev)
            e1.record(st)
            records.append((c, sd.visible_tokens(cfg, c), e0, e1, pairs))
        else:
            call(0, c)
    st.synchronize()
    sd.check_device_error(sess.ws)

    def summarize(recs):
        if not recs:
            return None
        path_ms = sum(r[2].elapsed_time(r[3]) for r in recs)
        attn_ms = sum(a.elapsed_time(b) for r in recs for a, b in r[4])
        flops = sum(4.0 * w.heads * w.head_dim * w.nq * r[1] * w.batch * len(r[4]) for r in recs)
        return {"chunks": len(recs), "path_ms": round(path_ms, 3), "attention_ms": round(attn_ms, 3),
                "ms_per_chunk": round(path_ms / len(recs), 4),
                "attention_tflops": round(flops / (attn_ms * 1e-3) / 1e12, 1),
                "latent_frames_per_s": round(len(recs) * w.chunk_frames * w.batch / (path_ms * 1e-3), 2),
                "pflop": round(flops / 1e15, 4)}

    warm = [r for r in records if r[1] < steady_nkv]
    steady = [r for r in records if r[1] == steady_nkv]
    total = summarize(records)
    return {"workload": w.name, "streams": w.batch, "chunks": chunks, "timed_chunks": len(records),
            "layers": w.layers, "denoise_steps": w.denoise_steps, "calls_timed": sum(len(r[4]) for r in records),
            "run_pflop": total["pflop"], "attention_tflops": total["attention_tflops"],
            "t_path_s": round(total["path_ms"] * 1e-3, 4), "latent_frames_per_s": total["latent_frames_per_s"],
            "warmup": summarize(warm), "steady": summarize(steady),
            "timed_windows": None if chunks <= LONG_STREAM else [list(x) for x in WINDOWS]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="wan13b_480p", choices=sorted(k for k in WORKLOADS if k != "tiny"))
    ap.add_argument("--chunks", type=int, default=0, help="chunks to stream (default: the workload's)")
    args = ap.parse_args()
    res = run(WORKLOADS[args.workload], args.chunks or None)
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
