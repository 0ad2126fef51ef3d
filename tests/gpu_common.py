"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle in lock-step and
compare them (bit-exact for q_rot, cache rows and slot metadata; attention within the stated
tolerance: max-abs 2e-2 and mean-abs 2e-3 against the fp64 oracle)."""
import math
from dataclasses import replace

import numpy as np
import torch

import oracle
import streaming_causal_video_gb300 as sd
from synth_inputs import qkv_chunk_host, stream_config_dict

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def config(w, **over):
    return sd.StreamConfig.make(**stream_config_dict(w, **over))


class LockStep:
    """One layer of a stream batch on the GPU next to one StreamOracle per stream."""

    def __init__(self, w, start_frames=None, device="cuda"):
        self.w = w
        self.starts = list(w.start_frames if start_frames is None else start_frames)
        assert len(self.starts) == w.batch
        self.cfg = config(w)
        self.sess = sd.StreamSession(self.cfg, 1, self.starts, device)
        self.oracles = [oracle.StreamOracle(w, s) for s in self.starts]
        self.lse = torch.empty((w.batch, w.heads, w.nq), dtype=torch.float32, device=device)
        self.steps = []

    def step(self, chunks, qkv=None, seed_offset=0, same_streams=False):
        """Append + attend chunk chunks[b] of every stream b on both sides.  Returns the host
        copies (q_rot_oracle[b], q, k, v) for the comparisons."""
        w = self.w
        if qkv is None:
            q, k, v = qkv_chunk_host(w, w.batch, int(chunks[0]), step=int(sum(chunks)) + 7 * len(self.steps),
                                     seed_offset=seed_offset, same_streams=same_streams)
        else:
            q, k, v = qkv
        self.steps.append(list(chunks))
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        self.sess.layer_step(0, chunks, qd, kd, vd, lse=self.lse)
        torch.cuda.synchronize()
        q_rot_o = []
        for b in range(w.batch):
            q_rot_o.append(self.oracles[b].append_chunk(int(chunks[b]), bits(q[b]), bits(k[b]), bits(v[b])))
        return q_rot_o

    def check_q_rot(self, q_rot_o):
        g = bits(self.sess.q_rot)                       # [B][H][Nq][D]
        for b in range(self.w.batch):
            np.testing.assert_array_equal(g[b].transpose(1, 0, 2), q_rot_o[b], err_msg="q_rot stream %d" % b)

    def check_cache(self, only_frames=None):
        w = self.w
        L = self.sess.layers[0]
        kc, vc = bits(L.k), bits(L.v)                  # [B][H][rows][D]
        meta = L.meta.cpu().numpy()                     # [B][slots][2]
        hw = w.hw
        for b in range(w.batch):
            filled = set()
            for frame, tpos, kf, vf in self.oracles[b].cache.entries:
                s = oracle.slot_of_frame(frame, w.sink_frames, w.window_frames)
                assert s not in filled
                filled.add(s)
                assert tuple(meta[b, s]) == (frame, tpos), (b, s, tuple(meta[b, s]), frame, tpos)
                if only_frames is not None and frame not in only_frames:
                    continue
                np.testing.assert_array_equal(kc[b][:, s * hw:(s + 1) * hw, :], kf.transpose(1, 0, 2),
                                              err_msg="k slot %d stream %d" % (s, b))
                np.testing.assert_array_equal(vc[b][:, s * hw:(s + 1) * hw, :], vf.transpose(1, 0, 2),
                                              err_msg="v slot %d stream %d" % (s, b))
            assert filled == set(range(len(filled)))   # a contiguous prefix of slots
            for s in range(w.slots):
                if s not in filled:
                    assert tuple(meta[b, s]) == (-1, 0)
                    if only_frames is None:
                        assert not kc[b][:, s * hw:(s + 1) * hw, :].any()
                        assert not vc[b][:, s * hw:(s + 1) * hw, :].any()

    def check_cache_entries_in_slots(self):
        """Sink entries live in slots 0..F_s-1 in list order (after a sink update they are
        copies of window frames); window entries live in their ring slots.  Bit-exact rows
        and metadata, and nothing else is filled."""
        w = self.w
        L = self.sess.layers[0]
        kc, vc = bits(L.k), bits(L.v)
        meta = L.meta.cpu().numpy()
        hw = w.hw
        for b in range(w.batch):
            entries = self.oracles[b].cache.entries
            filled = set()
            for idx, (frame, tpos, kf, vf) in enumerate(entries):
                s = idx if idx < w.sink_frames else oracle.slot_of_frame(frame, w.sink_frames, w.window_frames)
                assert s not in filled
                filled.add(s)
                assert tuple(meta[b, s]) == (frame, tpos), (b, s, tuple(meta[b, s]), frame, tpos)
                np.testing.assert_array_equal(kc[b][:, s * hw:(s + 1) * hw, :], kf.transpose(1, 0, 2),
                                              err_msg="k slot %d stream %d" % (s, b))
                np.testing.assert_array_equal(vc[b][:, s * hw:(s + 1) * hw, :], vf.transpose(1, 0, 2),
                                              err_msg="v slot %d stream %d" % (s, b))
            assert filled == set(range(len(filled)))

    def check_attention(self, q_rot_o, rows=None, heads=None, check_lse=True):
        w = self.w
        out = to_f64(self.sess.out)                     # [B][Nq][H][D]
        lse = self.lse.cpu().numpy().astype(np.float64)
        worst = (0.0, 0.0)
        for b in range(w.batch):
            for h in (range(w.heads) if heads is None else heads):
                r = np.arange(w.nq) if rows is None else np.asarray(rows)
                ref, lse_ref = self.oracles[b].attend(q_rot_o[b], h, rows=r)
                got = out[b, r, h, :]
                err = np.abs(got - ref)
                assert np.all(np.isfinite(got))
                mx, mean = float(err.max()), float(err.mean())
                worst = (max(worst[0], mx), max(worst[1], mean))
                assert mx <= MAX_ABS and mean <= MEAN_ABS, \
                    "attention b=%d h=%d: max-abs %.3g mean-abs %.3g" % (b, h, mx, mean)
                if check_lse:
                    le = np.abs(lse[b, h, r] - lse_ref).max()
                    assert le <= LSE_ABS, "lse b=%d h=%d: %.3g" % (b, h, le)
        return worst


def sample_rows(nq: int, n: int, seed: int) -> np.ndarray:
    """Edges of the 128-row query tiles and of the chunk, plus seeded random rows."""
    fixed = [0, 1, 127, 128, 255, 256, nq - 1, nq - 2, (nq // 128) * 128, (nq // 128) * 128 - 1]
    rng = np.random.default_rng(seed)
    extra = rng.choice(nq, size=max(0, n - len(fixed)), replace=False)
    return np.unique(np.clip(np.array(fixed + list(extra)), 0, nq - 1))


def small_workload(base, **over):
    return replace(base, **over)
