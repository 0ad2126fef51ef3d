#!/usr/bin/env python
"""Benchmark of the streaming chunk-attention hot path on one GB300 (replicas for N > 1).

One step = one streamed chunk of the Wan-1.3B-shaped 480p stream at steady state (full sink +
window): the motion magnitude of the chunk's video frames, then for each of 2 denoise steps and
each of 30 layers, sdv2_rope_append_kv followed by sdv2_chunk_attention.

value   : chunk-attention TFLOP/s over the whole step (4*H*D*Nq*Nkv flops per attention call,
          divided by the step's wall time on the device; inputs resident in HBM).
e2e     : the same metric when every call's q, k, v come from pinned host buffers and every
          attention output and the motion result go back to pinned host buffers, copies timed.
roofline: the attention kernel, its flops per launch over its mean launch time (CUDA events on
          the launch stream, inside the timed region), against the measured dense bf16 peak.
cpu_baseline / --impl reference: the CPU oracle on the same workload, on a bounded sample of
          query rows (its cost per row is fixed at a given key count).

roofline_rope_append: the same for sdv2_rope_append_kv against the measured HBM copy bandwidth.
workloads: steady-state lines of the 1.3B-720p, 14B-480p and stream-batch shapes (same step and
          timing code, a few steps each), each with the oracle's attention on sampled rows.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--workload NAME] [--no-e2e] [--no-cpu-baseline] [--no-workloads] [--workload-steps K]
"""
import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth_inputs import WORKLOADS, stream_config_dict  # noqa: E402

METRIC = "chunk-attention TFLOP/s & latent frames/s (Wan-1.3B 480p shape); % BF16 peak"
PEAK_FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
VIDEO_FRAMES_PER_LATENT = 4          # Wan VAE: 4 video frames per latent frame in time
VIDEO_SHAPE = (480, 832, 3)


def describe(w):
    return ("%s: %d streams, %d heads x %d, %dx%d = %d tokens/latent frame, chunk %d frames (%d queries), "
            "sink %d + window %d frames (%d KV), %d layers x %d denoise steps per chunk"
            % (w.name, w.batch, w.heads, w.head_dim, w.grid_h, w.grid_w, w.hw, w.chunk_frames, w.nq,
               w.sink_frames, w.window_frames, w.slots * w.hw, w.layers, w.denoise_steps))


# ------------------------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ------------------------------------------------------------------------------------------

class Dist:
    def __init__(self, gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl"
            try:
                import torch
                if not torch.cuda.is_available():
                    backend = "gloo"
            except Exception:
                backend = "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------------------------
# peaks, clocks, profile evidence
# ------------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except Exception:
        return dict(PEAK_FALLBACK), "fallback"


def peak_value(d, key):
    """Find a numeric peak in MEASURED_PEAKS.json whatever its nesting."""
    if isinstance(d, dict):
        if key in d and isinstance(d[key], (int, float)):
            return float(d[key])
        for v in d.values():
            r = peak_value(v, key)
            if r is not None:
                return r
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            try:
                power.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def code_only(text):
    """C/CUDA source without comments and with whitespace collapsed, so that an edit to comments
    does not count as a change of the kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


ATTN_SECTION = ("// ---- chunk attention", "// ---- motion")


def attention_source_hash(read=None):
    """Hash of the code (not the comments) the attention kernel is built from: attention.cu,
    ptx.cuh, tmem_io.cuh and the chunk-attention section of internal.h (the other sections of
    that header describe other kernels)."""
    h = hashlib.sha256()
    for f in ("attention.cu", "ptx.cuh", "tmem_io.cuh", "internal.h"):
        if read is None:
            with open(os.path.join(ROOT, "streaming_causal_video_gb300", "csrc", f)) as fh:
                text = fh.read()
        else:
            text = read(f)
        if f == "internal.h":
            a = text.index(ATTN_SECTION[0])
            text = text[a:text.index(ATTN_SECTION[1], a)]
        h.update(code_only(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """dram bytes per attention launch from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "chunk_attention_%s.json" % workload)
    try:
        with open(path) as fh:
            d = json.load(fh)
    except Exception:
        return None
    if d.get("source_hash") != attention_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------------
# CPU oracle baseline
# ------------------------------------------------------------------------------------------

def oracle_sample(w, seconds_target, seed=0, max_rows=4096):
    """Time the oracle's fp64 attention on query rows of the steady-state key count, growing the
    sample until it has run about `seconds_target`.  Returns (flops, seconds, rows, threads)."""
    import numpy as np
    import oracle
    from synth_inputs import qkv_chunk_bits
    rng = np.random.default_rng(seed)
    nkv = w.slots * w.hw
    D = w.head_dim
    # keys/values: N(0,1) bf16 bits for one head, the chunk's queries for the rows
    q, k, _ = qkv_chunk_bits(w, 1, 0)
    keys = np.ascontiguousarray(np.resize(k[0, :, 0, :], (nkv, D)))
    vals = np.ascontiguousarray(np.resize(q[0, :, 1 % w.heads, :], (nkv, D)))
    qrows = np.ascontiguousarray(q[0, :, 0, :])
    rows_done, t_total, n = 0, 0.0, min(8, w.nq)
    while t_total < seconds_target and rows_done < max_rows:
        rows = rng.choice(w.nq, size=n, replace=False)
        t0 = time.perf_counter()
        oracle.attention_bf16(qrows, keys, vals, 1.0 / math.sqrt(D), rows=rows)
        t_total += time.perf_counter() - t0
        rows_done += n
        n = min(n * 2, 512, w.nq)
    flops = 4.0 * D * nkv * rows_done
    return flops, t_total, rows_done, oracle.num_threads()


def oracle_rope_append_sample(w, seconds_target):
    """Time the oracle's Causal-RoPE + cache append of whole chunks of workload w: rope_spec of
    the chunk's q and k (every head) and FrameListCache.append of its frames.  Returns
    (chunks, seconds, bytes per chunk)."""
    import oracle
    from synth_inputs import qkv_chunk_bits
    q, k, v = qkv_chunk_bits(w, 1, 0)
    so = oracle.StreamOracle(w, w.start_frames[0])
    done, t_total, c = 0, 0.0, 0
    while t_total < seconds_target or done == 0:
        t0 = time.perf_counter()
        so.append_chunk(c, q[0], k[0], v[0])
        t_total += time.perf_counter() - t0
        done += 1
        c += 1
    return done, t_total, 1536.0 * w.nq * w.heads


def oracle_tiny_run():
    """The oracle's whole tiny-stream run: every chunk appended (Causal-RoPE + list cache) and
    every query row of every head attended.  Returns (attention flops, seconds)."""
    import numpy as np
    import oracle
    from synth_inputs import qkv_chunk_bits
    w = WORKLOADS["tiny"]
    so = oracle.StreamOracle(w, w.start_frames[0])
    flops, secs = 0.0, 0.0
    for c in range(w.chunks):
        q, k, v = qkv_chunk_bits(w, 1, c)
        t0 = time.perf_counter()
        q_rot = so.append_chunk(c, q[0], k[0], v[0])
        nkv = sum(e[2].shape[0] for e in so.cache.entries)
        for h in range(w.heads):
            so.attend(q_rot, h)
        secs += time.perf_counter() - t0
        flops += 4.0 * w.heads * w.head_dim * w.nq * nkv
    return flops, secs


def oracle_motion_sample(frames_np, seconds_target):
    """Time the oracle's exact SSD over the given frames [B][T+1][...] repeatedly.  Returns
    (passes, seconds, bytes per pass)."""
    import oracle
    done, t_total = 0, 0.0
    while t_total < seconds_target or done == 0:
        t0 = time.perf_counter()
        oracle.motion_ssd(frames_np)
        t_total += time.perf_counter() - t0
        done += 1
    return done, t_total, float(frames_np.size)


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

class SteadyStream:
    """Device state of one workload at steady state (full sink + window in every layer's cache),
    and one bench step: motion over the chunk's video frames, then for each denoise step and
    layer, sdv2_rope_append_kv followed by sdv2_chunk_attention."""

    def __init__(self, w, dev, stream):
        import torch
        import streaming_causal_video_gb300 as sd
        from synth_inputs import motion_frames_host
        self.sd = sd
        self.w = w
        self.stream = stream
        self.cfg = sd.StreamConfig.make(**stream_config_dict(w))
        B, H, D, nq = w.batch, w.heads, w.head_dim, w.nq
        self.sess = sd.StreamSession(self.cfg, w.layers, w.start_frames, dev, stream)
        g = torch.Generator(device=dev).manual_seed(w.seed)
        self.qkv = [tuple(torch.randn((B, nq, H, D), generator=g, device=dev, dtype=torch.float32)
                          .to(torch.bfloat16) for _ in range(3)) for _ in range(w.layers)]
        self.outs = [torch.empty((B, nq, H, D), dtype=torch.bfloat16, device=dev) for _ in range(w.layers)]
        self.vf = VIDEO_FRAMES_PER_LATENT * w.chunk_frames
        Hp, Wp, Cc = VIDEO_SHAPE
        self.frames = motion_frames_host(B, self.vf + 1, Hp, Wp, Cc, seed=w.seed, device=dev)
        self.ssd = torch.empty((B, self.vf), dtype=torch.int64, device=dev)
        self.mrms = torch.empty((B, self.vf), dtype=torch.float32, device=dev)
        steady = 0
        while sd.visible_tokens(self.cfg, steady) < w.slots * w.hw:
            steady += 1
        for c in range(steady):
            for l in range(w.layers):
                q, k, v = self.qkv[l]
                self.sess.layer_step(l, [c] * B, q, k, v, out=self.outs[l], stream=stream)
        stream.synchronize()
        sd.check_device_error(self.sess.ws, stream)
        self.chunk = steady
        self.attn_flops = 4.0 * H * D * nq * sd.visible_tokens(self.cfg, steady) * B
        self.rope_bytes = 1536.0 * B * nq * H          # read q, k, v; write q_rot, k, v rows
        self.launches_per_step = 3 + 2 * w.denoise_steps * w.layers

    def step(self, attn_ev=None, rope_ev=None):
        """One chunk; returns its attention flops.  attn_ev / rope_ev, if lists, receive a pair
        of CUDA events around every attention / rope_append call (recorded on the launch
        stream)."""
        import torch
        sd, w, st, S = self.sd, self.w, self.stream, self.sess
        c = self.chunk
        B = w.batch

        def ev():
            e = torch.cuda.Event(enable_timing=True)
            e.record(st)
            return e
        sd.motion_l2(self.frames, self.ssd, self.mrms, stream=st)
        for _s in range(w.denoise_steps):
            for l in range(w.layers):
                q, k, v = self.qkv[l]
                L = S.layers[l]
                r0 = ev() if rope_ev is not None else None
                sd.rope_append_kv(self.cfg, w.start_frames, [c] * B, q, k, v, S.q_rot, L.k, L.v, L.meta, S.ws, st)
                a0 = ev() if (rope_ev is not None or attn_ev is not None) else None
                sd.chunk_attention(self.cfg, [c] * B, S.q_rot, L.k, L.v, self.outs[l], S.ws, stream=st)
                if rope_ev is not None:
                    rope_ev.append((r0, a0))
                if attn_ev is not None:
                    attn_ev.append((a0, ev()))
        self.chunk += 1
        return w.denoise_steps * w.layers * self.attn_flops

    def close(self):
        import torch
        self.sd.check_device_error(self.sess.ws, self.stream)
        del self.sess, self.qkv, self.outs, self.frames
        torch.cuda.empty_cache()


def timed_steps(state, steps, dist, dev, clock_gpu, attn_ev=None, rope_ev=None):
    """Barrier + synchronize, time `steps` steps with CUDA events on the launch stream, barrier +
    synchronize; clocks sampled during the region.  Returns (flops, ms max over ranks, clocks)."""
    import torch
    clocks = ClockSampler(clock_gpu)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(state.stream)
    flops = 0.0
    h0 = time.perf_counter()
    for _ in range(steps):
        flops += state.step(attn_ev, rope_ev)
    clocks.host_issue_ms_per_step = (time.perf_counter() - h0) * 1e3 / max(1, steps)
    t1.record(state.stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clk = clocks.stop()
    clk["host_issue_ms_per_step"] = round(clocks.host_issue_ms_per_step, 3)
    return flops, dist.max(t0.elapsed_time(t1)), clk


def measure_other_workload(name, steps, warmup, dist, dev, stream, oracle_seconds):
    """Steady-state attention TFLOP/s and latent frames/s of another workload (same step and
    timing code as the headline), with the oracle's attention on sampled rows beside it."""
    w = WORKLOADS[name]
    state = SteadyStream(w, dev, stream)
    for _ in range(warmup):
        state.step()
    stream.synchronize()
    attn_ev = []
    flops, ms, clk = timed_steps(state, steps, dist, dev, dist.local, attn_ev=attn_ev)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in attn_ev)
    splits = state.sd.last_kv_splits()
    state.close()
    res = {"workload": describe(w), "steps": steps, "ms_per_step": round(ms / steps, 3),
           "attention_tflops": round(flops * dist.world / (ms * 1e-3) / 1e12, 3),
           "latent_frames_per_s": round(steps * w.chunk_frames * w.batch * dist.world / (ms * 1e-3), 3),
           "attention_ms_per_call": round(attn_ms, 4),
           "attention_call_tflops": round(state.attn_flops / (attn_ms * 1e-3) / 1e12, 2),
           "kv_splits": splits, "clocks": clk}
    if dist.world == 1 and oracle_seconds > 0:
        f, secs, rows, threads = oracle_sample(w, oracle_seconds, seed=7)
        res["cpu_baseline"] = {"value": round(f / secs / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
                               "kind": "oracle",
                               "sample": "fp64 oracle attention of %d query rows against the steady-state %d keys "
                                         "(%.1f s)" % (rows, w.slots * w.hw, secs)}
    return res


def run_ours(args, dist):
    import torch
    import streaming_causal_video_gb300 as sd

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    w = WORKLOADS[args.workload]
    B, H, D, nq = w.batch, w.heads, w.head_dim, w.nq
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    state = SteadyStream(w, dev, stream)
    cfg, sess, qkv, outs = state.cfg, state.sess, state.qkv, state.outs
    frames, ssd, mrms, vf = state.frames, state.ssd, state.mrms, state.vf
    flops_per_call = state.attn_flops
    launches_per_step = state.launches_per_step
    warmup = max(3, args.warmup)
    for _ in range(warmup):
        state.step()
    stream.synchronize()
    sd.check_device_error(sess.ws, stream)

    # ---- device-resident timed region (events around every attention and rope_append call)
    attn_ev, rope_ev = [], []
    flops, ms_max, clk = timed_steps(state, args.steps, dist, dev, dist.local, attn_ev=attn_ev, rope_ev=rope_ev)
    sd.check_device_error(sess.ws, stream)
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    rope_ms = [a.elapsed_time(b) for a, b in rope_ev]
    attn_mean_ms = statistics.mean(attn_ms)
    rope_mean_ms = statistics.mean(rope_ms)
    total_flops = flops * dist.world
    value = total_flops / (ms_max * 1e-3) / 1e12
    latent_fps = args.steps * w.chunk_frames * B * dist.world / (ms_max * 1e-3)

    # ---- end-to-end through the C ABI with host buffers
    # Every call's q, k, v come from pinned host memory and every attention output (and the
    # motion result) goes back to pinned host memory.  Copies run on two copy streams,
    # double-buffered against the compute stream and ordered with events, as a serving loop
    # that receives activations from the host would run them.
    e2e = None
    if not args.no_e2e:
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
        h_qkv = [tuple(pin(t) for t in qkv[l]) for l in range(w.layers)]
        h_out = [torch.empty((B, nq, H, D), dtype=torch.bfloat16, pin_memory=True) for _ in range(w.layers)]
        h_frames = pin(frames)
        h_ssd = torch.empty((B, vf), dtype=torch.int64, pin_memory=True)
        nbuf = 2
        d_in = [tuple(torch.empty_like(t) for t in qkv[0]) for _ in range(nbuf)]
        h2d_stream = torch.cuda.Stream(device=dev)
        d2h_stream = torch.cuda.Stream(device=dev)
        in_free = [torch.cuda.Event() for _ in range(nbuf)]      # staging buffer consumed
        in_ready = [torch.cuda.Event() for _ in range(nbuf)]     # staging buffer filled
        out_ready = [torch.cuda.Event() for _ in range(w.layers)]
        out_free = [torch.cuda.Event() for _ in range(w.layers)]
        ssd_free = torch.cuda.Event()
        for e in in_free + out_free + [ssd_free]:
            e.record(stream)
        h2d = sum(t.numel() * t.element_size() for t in h_qkv[0]) * w.layers * w.denoise_steps + \
            h_frames.numel()
        d2h = h_out[0].numel() * 2 * w.layers * w.denoise_steps + h_ssd.numel() * 8
        counter = [0]

        def e2e_step():
            c = state.chunk
            with torch.cuda.stream(h2d_stream):
                frames.copy_(h_frames, non_blocking=True)
                fr_ready = torch.cuda.Event()
                fr_ready.record(h2d_stream)
            stream.wait_event(fr_ready)
            stream.wait_event(ssd_free)
            sd.motion_l2(frames, ssd, mrms, stream=stream)
            ssd_ready = torch.cuda.Event()
            ssd_ready.record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ssd_ready)
                h_ssd.copy_(ssd, non_blocking=True)
                ssd_free.record(d2h_stream)
            for _s in range(w.denoise_steps):
                for l in range(w.layers):
                    i = counter[0] % nbuf
                    counter[0] += 1
                    q, k, v = d_in[i]
                    hq, hk, hv = h_qkv[l]
                    with torch.cuda.stream(h2d_stream):
                        h2d_stream.wait_event(in_free[i])
                        if e2e_copy_ev is not None:
                            c0 = torch.cuda.Event(enable_timing=True)
                            c0.record(h2d_stream)
                        q.copy_(hq, non_blocking=True)
                        k.copy_(hk, non_blocking=True)
                        v.copy_(hv, non_blocking=True)
                        in_ready[i].record(h2d_stream)
                        if e2e_copy_ev is not None:
                            c1 = torch.cuda.Event(enable_timing=True)
                            c1.record(h2d_stream)
                            e2e_copy_ev.append((c0, c1))
                    stream.wait_event(in_ready[i])
                    L = sess.layers[l]
                    sd.rope_append_kv(cfg, w.start_frames, [c] * B, q, k, v, sess.q_rot, L.k, L.v, L.meta,
                                      sess.ws, stream)
                    in_free[i].record(stream)
                    stream.wait_event(out_free[l])
                    if e2e_attn_ev is not None:
                        a0 = torch.cuda.Event(enable_timing=True)
                        a0.record(stream)
                    sd.chunk_attention(cfg, [c] * B, sess.q_rot, L.k, L.v, outs[l], sess.ws, stream=stream)
                    out_ready[l].record(stream)
                    if e2e_attn_ev is not None:
                        a1 = torch.cuda.Event(enable_timing=True)
                        a1.record(stream)
                        e2e_attn_ev.append((a0, a1))
                    with torch.cuda.stream(d2h_stream):
                        d2h_stream.wait_event(out_ready[l])
                        h_out[l].copy_(outs[l], non_blocking=True)
                        out_free[l].record(d2h_stream)
            state.chunk += 1
            return w.denoise_steps * w.layers * flops_per_call

        e2e_attn_ev = None
        e2e_copy_ev = None
        for _ in range(warmup):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_attn_ev = []
        e2e_copy_ev = []
        clocks2 = ClockSampler(dist.local)
        clocks2.start()
        dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        f2 = 0.0
        h0 = time.perf_counter()
        for _ in range(args.steps):
            f2 += e2e_step()
        host_issue_ms = (time.perf_counter() - h0) * 1e3 / args.steps
        # the step's results are on the host only when both copy streams have drained
        done_h2d = torch.cuda.Event()
        done_h2d.record(h2d_stream)
        done_d2h = torch.cuda.Event()
        done_d2h.record(d2h_stream)
        stream.wait_event(done_h2d)
        stream.wait_event(done_d2h)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
        clk2 = clocks2.stop()
        ms2 = dist.max(e0.elapsed_time(e1))
        e2e_attn_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_attn_ev)
        e2e_h2d_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_copy_ev)
        sd.check_device_error(sess.ws, stream)
        e2e = {"value": round(f2 * dist.world / (ms2 * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(ms2 / args.steps, 3),
               "host_issue_ms_per_step": round(host_issue_ms, 3),
               "attention_mean_launch_ms": round(e2e_attn_ms, 4),
               "h2d_ms_per_layer": round(e2e_h2d_ms, 4),
               "h2d_GBs_per_layer": round(3 * qkv[0][0].numel() * 2 / (e2e_h2d_ms * 1e-3) / 1e9, 1),
               "clocks": clk2,
               "latent_frames_per_s": round(args.steps * w.chunk_frames * B * dist.world / (ms2 * 1e-3), 3),
               "copies": "pinned host buffers; H2D and D2H on two copy streams overlapped with compute"}
        del h_qkv, h_out, d_in

    peaks, peak_src = load_peaks()
    peak = peak_value(peaks, "bf16_tflops_sustained") or PEAK_FALLBACK["bf16_tflops_sustained"]
    hbm = peak_value(peaks, "hbm_gbs") or PEAK_FALLBACK["hbm_gbs"]
    achieved = flops_per_call / (attn_mean_ms * 1e-3) / 1e12
    traffic = profiled_traffic(args.workload)
    roofline = {"bound": "tensor", "kernel": "chunk_attention_kernel", "achieved": round(achieved, 2),
                "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": "%s bf16_tflops_sustained (kernel timed inside a long step)" % peak_src,
                "flops_per_launch": flops_per_call, "mean_launch_ms": round(attn_mean_ms, 4),
                "launches_timed": len(attn_ms),
                "joules_per_launch_est": (round(clk["power_w"] * attn_mean_ms * 1e-3, 4)
                                          if clk.get("power_w") else None),
                "joules_note": "median board power sampled by nvidia-smi during the timed region x mean "
                               "attention launch time (the step is ~97 % attention)"}
    rope_gbs = state.rope_bytes / (rope_mean_ms * 1e-3) / 1e9
    roofline_rope = {"bound": "hbm", "kernel": "rope_append_kernel", "achieved": round(rope_gbs, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(rope_gbs / hbm, 4), "traffic": None,
                     "peak_source": "%s hbm_gbs" % peak_src,
                     "bytes_per_launch": state.rope_bytes, "mean_launch_ms": round(rope_mean_ms, 5),
                     "launches_timed": len(rope_ms), "sm_mhz": clk.get("sm_mhz"),
                     "note": "CUDA events around each sdv2_rope_append_kv call inside the step; the call's "
                             "43 MB of writes may still sit in L2 when its end event is recorded (the next "
                             "attention launch reads them from there)"}

    res = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": dist.world,
           "steps": args.steps, "warmup": warmup, "ms_per_step": round(ms_max / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded N(0,1) bf16 q/k/v per layer; seeded moving-texture uint8 frames)",
           "config": {"workload": describe(w), "global_batch": B * dist.world,
                      "parallelism": "replicas" if dist.world > 1 else "single GPU",
                      "l2": "inputs larger than L2: %d distinct layer caches (%.1f GB)"
                            % (w.layers, 2 * sd.cache_bytes(cfg) * w.layers / 1e9),
                      "step": "1 chunk: motion over %d video frames + %d denoise steps x %d layers x "
                              "(rope_append_kv + chunk_attention) at steady state (Nkv=%d)"
                              % (vf, w.denoise_steps, w.layers, w.slots * w.hw),
                      "kv_splits": sd.last_kv_splits()},
           "latent_frames_per_s": round(latent_fps, 3),
           "pct_bf16_peak": round(100.0 * value / peak, 2),
           "gpu_launches": launches_per_step * args.steps,
           "clocks": clk, "roofline": roofline, "roofline_rope_append": roofline_rope, "e2e": e2e,
           "impl": "ours"}
    motion_np = frames.cpu().numpy() if dist.world == 1 and not args.no_cpu_baseline else None
    state.close()
    del cfg, sess, qkv, outs, frames, ssd, mrms
    if not args.no_workloads:
        others = [n for n in ("wan13b_720p", "wan14b_480p", "stream_batch") if n != args.workload]
        res["workloads"] = {n: measure_other_workload(n, args.workload_steps, 3, dist, dev, stream,
                                                      0 if args.no_cpu_baseline else 2.5) for n in others}
    res["_motion_frames"] = motion_np
    return res


def cpu_baseline_entry(w, motion_np, seconds=10.0, single_seconds=3.0, rope_seconds=2.0, motion_seconds=1.5):
    """The oracle on all host cores (the reported value) and, for scale, on one thread: the
    attention on sampled rows, plus the Causal-RoPE + append of whole chunks and the motion SSD
    of the step's frames."""
    import oracle
    flops, secs, rows, threads = oracle_sample(w, seconds)
    all_threads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        f1, s1, r1, _ = oracle_sample(w, single_seconds, seed=1, max_rows=256)
    finally:
        oracle.set_num_threads(all_threads)
    out = {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "single_thread_value": round(f1 / s1 / 1e12, 7),
           "sample": "fp64 oracle attention of %d query rows against the steady-state %d keys of one head "
                     "(bf16 inputs), %.1f s on %d threads; single_thread_value: %d rows, %.1f s on 1 thread; "
                     "TFLOP/s counts the same 4*D*Nkv flops per row as the GPU metric"
                     % (rows, w.slots * w.hw, secs, threads, r1, s1)}

    def both(fn, unit_scale, unit, what):
        n, t, per = fn()
        oracle.set_num_threads(1)
        try:
            n1, t1, _ = fn()
        finally:
            oracle.set_num_threads(all_threads)
        return {"value": round(n * per / t / unit_scale, 4), "unit": unit, "cores": all_threads,
                "single_thread_value": round(n1 * per / t1 / unit_scale, 5), "kind": "oracle",
                "sample": "%s: %d passes in %.2f s on %d threads; %d in %.2f s on 1 thread"
                          % (what, n, t, all_threads, n1, t1)}
    out["rope_append"] = both(lambda: oracle_rope_append_sample(w, rope_seconds), 1e9, "GB/s",
                              "rope_spec of the chunk's q and k (%d tokens x %d heads) + FrameListCache.append "
                              "of its %d frames; GB/s counts the kernel's 1536 algorithmic bytes per token-head"
                              % (w.nq, w.heads, w.chunk_frames))
    f_all, s_all = oracle_tiny_run()
    oracle.set_num_threads(1)
    try:
        f_one, s_one = oracle_tiny_run()
    finally:
        oracle.set_num_threads(all_threads)
    out["tiny_run"] = {"value": round(s_all, 4), "unit": "s per run", "cores": all_threads,
                       "single_thread_value": round(s_one, 4), "kind": "oracle",
                       "tflops": round(f_all / s_all / 1e12, 6), "single_thread_tflops": round(f_one / s_one / 1e12, 7),
                       "sample": "the whole tiny stream (10 chunks, 2 heads, 72 queries per chunk): Causal-RoPE + "
                                 "list-cache append of every chunk and attention of every query row"}
    if motion_np is not None:
        out["motion"] = both(lambda: oracle_motion_sample(motion_np, motion_seconds), 1e9, "GB/s",
                             "motion_ssd of the step's %d frames of %s per stream (exact uint64), GB/s of "
                             "frame bytes read" % (motion_np.shape[1], "x".join(map(str, motion_np.shape[2:]))))
    return out


def run_reference(args, dist):
    """The oracle as the reference arm: each step is a bounded sample of the workload's attention."""
    import oracle
    w = WORKLOADS[args.workload]
    warmup = max(3, args.warmup)
    per_step = 2.0
    for _ in range(warmup):
        oracle_sample(w, per_step / 4, seed=1, max_rows=64)
    flops = secs = 0.0
    rows = 0
    for s in range(args.steps):
        f, t, r, threads = oracle_sample(w, per_step, seed=100 + s, max_rows=2048)
        flops += f
        secs += t
        rows += r
    value = flops / secs / 1e12
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": warmup, "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(w)}, "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": "per step: fp64 oracle attention of query rows against the steady-state "
                                       "%d keys for about %.0f s; %d rows in all" % (w.slots * w.hw, per_step, rows)},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wan13b_480p", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the steady-state lines of the other workloads (1.3B-720p, 14B-480p, stream batch)")
    ap.add_argument("--workload-steps", type=int, default=3, help="timed steps of each other workload")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count (profiling runs only; 0 = workload's)")
    args = ap.parse_args()
    if args.layers:
        import dataclasses
        WORKLOADS[args.workload] = dataclasses.replace(WORKLOADS[args.workload], layers=args.layers)

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, None)), flush=True)
        return 0

    dist = Dist(args.gpus)
    res = run_ours(args, dist)
    motion_np = res.pop("_motion_frames", None)
    if dist.rank == 0:
        if dist.world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline_entry(WORKLOADS[args.workload], motion_np)
        print(json.dumps(res), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
