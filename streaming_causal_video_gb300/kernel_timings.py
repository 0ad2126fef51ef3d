"""Per-entry-point timings at the workload shapes (CUDA events on the launch stream).

For each HBM-bound call: algorithmic bytes per call, mean time over repeated calls on buffers
larger than L2 (several distinct layer caches are cycled), achieved GB/s and the fraction of
the copy-bandwidth peak.  For attention: flops per call and TFLOP/s.  Prints one JSON line per
measurement.  Run: python -m streaming_causal_video_gb300.kernel_timings [--peak-gbs X] [--only qkv,...]
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
from synth_inputs import WORKLOADS, motion_frames_host, stream_config_dict  # noqa: E402


def _time(fn, reps, stream):
    for _ in range(3):
        fn(0)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    stream.synchronize()
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--peak-gbs", type=float, default=0.0, help="HBM peak (GB/s); default: MEASURED_PEAKS.json or 6800")
    ap.add_argument("--layers", type=int, default=8, help="distinct layer caches cycled (more than L2 in total)")
    ap.add_argument("--only", default="", help="comma-separated subset of: append, attention, rerotate, sink, "
                    "qkv, cublas, unfused, qkv14b, motion, noise, copies (default: all)")
    args = ap.parse_args()
    only = {x.strip() for x in args.only.split(",") if x.strip()}

    def want(k):
        return not only or k in only
    peak = args.peak_gbs
    src = "given"
    if not peak:
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
                d = json.load(fh)
            peak = float(d.get("hbm_gbs") or d["hbm"]["gbs"])
            src = "measured"
        except Exception:
            peak, src = 6800.0, "fallback"

    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    out = []

    def report(name, workload, bytes_per_call=None, flops_per_call=None, ms=None, extra=None):
        rec = {"entry_point": name, "workload": workload, "ms_per_call": round(ms, 5)}
        if bytes_per_call:
            gbs = bytes_per_call / (ms * 1e-3) / 1e9
            rec.update({"bytes_per_call": int(bytes_per_call), "GB_per_s": round(gbs, 1),
                        "frac_of_hbm_peak": round(gbs / peak, 3), "peak_GB_per_s": peak, "peak_source": src})
        if flops_per_call:
            rec.update({"flops_per_call": flops_per_call, "TFLOP_per_s": round(flops_per_call / (ms * 1e-3) / 1e12, 1)})
        if extra:
            rec.update(extra)
        out.append(rec)
        print(json.dumps(rec), flush=True)

    # ---- 1.3B-480p: rope_append, re-rotation, sink update, attention
    w = WORKLOADS["wan13b_480p"]
    cfg = sd.StreamConfig.make(**stream_config_dict(w))
    nl = args.layers
    sess = StreamSession(cfg, nl, w.start_frames, dev, stream)
    g = torch.Generator(device=dev).manual_seed(1)
    qkv = [tuple(torch.randn((1, w.nq, w.heads, 128), generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
           for _ in range(nl)]
    steady = 6
    for c in range(steady + 1):
        for l in range(nl):
            sess.layer_step(l, [c], *qkv[l], stream=stream)
    stream.synchronize()

    def rope(i):
        l = i % nl
        L = sess.layers[l]
        sd.rope_append_kv(cfg, w.start_frames, [steady], *qkv[l], sess.q_rot, L.k, L.v, L.meta, sess.ws, stream)
    if want("append"):
        report("sdv2_rope_append_kv", w.name, bytes_per_call=w.nq * w.heads * 1536, ms=_time(rope, 60, stream))

    def attn(i):
        L = sess.layers[i % nl]
        sd.chunk_attention(cfg, [steady], sess.q_rot, L.k, L.v, sess.out, sess.ws, stream=stream)
    nkv = sd.visible_tokens(cfg, steady)
    if want("attention"):
        report("sdv2_chunk_attention", w.name, flops_per_call=4.0 * w.heads * 128 * w.nq * nkv,
               ms=_time(attn, 30, stream), extra={"kv_splits": sd.last_kv_splits()})

    # re-rotation at a refresh chunk: every window slot holds an earlier frame (R = 7 chunks so
    # that chunk 7 is a refresh chunk); time-axis vectors of the window keys are read and written
    cfg_r = sd.StreamConfig.make(**stream_config_dict(w))
    cfg_r.refresh_chunks = 7
    tvecs = (w.rope_t // 2 + 3) // 4
    rr_bytes = w.window_frames * w.hw * w.heads * tvecs * 16 * 2

    def rerot(i):
        L = sess.layers[i % nl]
        sd.rope_refresh_rerotate(cfg_r, [7], L.k, L.meta, stream)
    if want("rerotate"):
        report("sdv2_rope_refresh_rerotate", w.name + " (window of 18 frames)", bytes_per_call=rr_bytes,
               ms=_time(rerot, 60, stream))

    sink_bytes = w.sink_frames * w.hw * w.heads * 256 * 2 * 2

    def sink(i):
        L = sess.layers[i % nl]
        sd.sink_update(cfg, [steady], [1], L.k, L.v, L.meta, stream)
    if want("sink"):
        report("sdv2_sink_update", w.name + " (3 sink frames)", bytes_per_call=sink_bytes, ms=_time(sink, 60, stream))
    # fused QKV projection + RoPE + append vs the unfused sequence (projection GEMM through
    # torch/cuBLAS to bf16, then sdv2_rope_append_kv)
    C = w.heads * w.head_dim
    xs = [torch.randn((1, w.nq, C), generator=g, device=dev).to(torch.bfloat16) for _ in range(nl)]
    Wq = (torch.randn((3 * C, C), generator=g, device=dev) / C ** 0.5).to(torch.bfloat16)
    bq = torch.randn(3 * C, generator=g, device=dev).float() * 0.1
    gemm_flops = 2.0 * w.nq * 3 * C * C

    def fused(i):
        L = sess.layers[i % nl]
        sd.qkv_rope_append(cfg, w.start_frames, [steady], xs[i % nl], Wq, sess.q_rot, L.k, L.v, L.meta, sess.ws,
                           bias=bq, stream=stream)
    if want("qkv"):
        report("sdv2_qkv_rope_append", w.name + " (x [4680][1536] @ W[4608][1536]^T + bias, RoPE, append)",
               flops_per_call=gemm_flops, ms=_time(fused, 60, stream),
               extra={"bytes_min": int((w.nq * C + 3 * C * C) * 2 + w.nq * 3 * C * 2)})
    ybuf = torch.empty((1, w.nq, 3 * C), dtype=torch.bfloat16, device=dev)

    def gemm_only(i):
        torch.matmul(xs[i % nl][0], Wq.t(), out=ybuf[0])
    if want("cublas"):
        report("projection GEMM alone: torch.matmul (cuBLAS), bf16 out, no bias or RoPE", w.name,
               flops_per_call=gemm_flops, ms=_time(gemm_only, 60, stream))

    def unfused(i):
        l = i % nl
        L = sess.layers[l]
        torch.matmul(xs[l][0], Wq.t(), out=ybuf[0])
        ybuf.add_(bq.to(torch.bfloat16))
        y = ybuf.view(1, w.nq, 3, w.heads, w.head_dim)
        cfg_s = sd.StreamConfig.make(**stream_config_dict(w, qkv_token_stride=3 * C))
        sd.rope_append_kv(cfg_s, w.start_frames, [steady], y[:, :, 0], y[:, :, 1], y[:, :, 2], sess.q_rot, L.k, L.v,
                          L.meta, sess.ws, stream)
    if want("unfused"):
        report("unfused: torch.matmul (cuBLAS) + bias + sdv2_rope_append_kv", w.name, flops_per_call=gemm_flops,
               ms=_time(unfused, 60, stream))
    del sess, qkv
    torch.cuda.empty_cache()

    # fused projection at the Wan-14B 480p shape (C = 5120, 40 heads: 80 feature tiles, a
    # 5120-long hidden dimension) against the library GEMM of the same shape
    if want("qkv14b"):
        w14 = WORKLOADS["wan14b_480p"]
        cfg14 = sd.StreamConfig.make(**stream_config_dict(w14))
        nl14 = max(1, min(nl, 4))
        sess14 = StreamSession(cfg14, nl14, w14.start_frames, dev, stream)
        C14 = w14.heads * w14.head_dim
        xs14 = [torch.randn((1, w14.nq, C14), generator=g, device=dev).to(torch.bfloat16) for _ in range(nl14)]
        W14 = (torch.randn((3 * C14, C14), generator=g, device=dev) / C14 ** 0.5).to(torch.bfloat16)
        b14 = torch.randn(3 * C14, generator=g, device=dev).float() * 0.1
        flops14 = 2.0 * w14.nq * 3 * C14 * C14

        def fused14(i):
            L = sess14.layers[i % nl14]
            sd.qkv_rope_append(cfg14, w14.start_frames, [steady], xs14[i % nl14], W14, sess14.q_rot, L.k, L.v, L.meta,
                               sess14.ws, bias=b14, stream=stream)
        report("sdv2_qkv_rope_append", w14.name + " (x [4680][5120] @ W[15360][5120]^T + bias, RoPE, append)",
               flops_per_call=flops14, ms=_time(fused14, 30, stream))
        y14 = torch.empty((1, w14.nq, 3 * C14), dtype=torch.bfloat16, device=dev)

        def gemm14(i):
            torch.matmul(xs14[i % nl14][0], W14.t(), out=y14[0])
        report("projection GEMM alone: torch.matmul (cuBLAS), bf16 out, no bias or RoPE", w14.name,
               flops_per_call=flops14, ms=_time(gemm14, 30, stream))
        del sess14, xs14, W14, y14
        torch.cuda.empty_cache()

    # size-matched reference: a plain device-to-device copy (torch copy_) moving the same bytes
    # (half read, half written) as each HBM-bound call, over 8 buffer pairs cycled so that the
    # set is larger than L2 -- the bandwidth a copy of that size reaches on this GPU
    if want("copies"):
        for label, nbytes in (("rope_append_kv", w.nq * w.heads * 1536), ("rope_refresh_rerotate", rr_bytes),
                              ("sink_update", sink_bytes)):
            half = nbytes // 2
            srcs = [torch.empty(half, dtype=torch.uint8, device=dev) for _ in range(nl)]
            dsts = [torch.empty(half, dtype=torch.uint8, device=dev) for _ in range(nl)]

            def cp(i):
                dsts[i % nl].copy_(srcs[i % nl])
            report("reference copy_ of the bytes of sdv2_" + label, w.name, bytes_per_call=2 * half,
                   ms=_time(cp, 60, stream))
            del srcs, dsts
        torch.cuda.empty_cache()
    if not (want("motion") or want("noise")):
        return out

    # ---- stream batch: motion over 4 x 501 frames of 480x832x3, then the noise controller
    wb = WORKLOADS["stream_batch"]
    hp, wp, ch = wb.motion_frame_shape
    frames = motion_frames_host(wb.batch, 501, hp, wp, ch, seed=wb.seed, device=dev)
    ssd = torch.empty((wb.batch, 500), dtype=torch.int64, device=dev)
    m = torch.empty((wb.batch, 500), dtype=torch.float32, device=dev)

    def motion(i):
        sd.motion_l2(frames, ssd, m, stream)
    if want("motion"):
        report("sdv2_motion_l2", "stream_batch: 4 x 501 frames of 480x832x3", bytes_per_call=frames.numel(),
               ms=_time(motion, 10, stream))
    ctl = sd.NoiseCtl(motion_lo=2.0, motion_hi=12.0, rate_lo=0.1, rate_hi=0.9, ema=0.5, more_noise_when_fast=1)
    rate = torch.empty_like(m)

    def noise(i):
        sd.noise_from_motion(ctl, m, rate, None, stream)
    if want("noise"):
        report("sdv2_noise_from_motion", "stream_batch: 4 x 500 motion values", ms=_time(noise, 100, stream))
    return out


if __name__ == "__main__":
    main()
