"""sdv2_chunk_attention_noalloc: attention without a caller-owned workspace.

Callers that cannot allocate device memory (a memory pool they do not own, a plugin host that
forbids allocation after start-up, a real-time loop that must never reach the allocator) use
this entry point; its scratch is a static array inside the library.  These tests call it
through the C ABI and check, on two calls in a row, that its output matches the workspace
entry point's within the parity tolerance, and that sizes its array cannot serve are
rejected.  The file is collected last so that a run stopping at the first failure has run
every other test already; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS
from gpu_common import LockStep, MAX_ABS, MEAN_ABS, config, small_workload, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


@pytest.mark.parametrize("w,chunks", [
    (WORKLOADS["tiny"], 4),                                                                   # 2 key splits
    (small_workload(WORKLOADS["wan13b_480p"], heads=2, grid_h=10, grid_w=16, chunks=8), 8),   # 4 key splits
    (small_workload(WORKLOADS["stream_batch"], heads=3, grid_h=6, grid_w=8, chunks=3), 3),    # 4 streams
])
def test_noalloc_matches_workspace_entry_point_on_two_calls(w, chunks):
    ls = LockStep(w)
    for c in range(chunks):
        ls.step([c] * w.batch)
    L = ls.sess.layers[0]
    cidx = [chunks - 1] * w.batch
    ref = torch.empty_like(ls.sess.out)
    ref_lse = torch.empty_like(ls.lse)
    sd.chunk_attention(ls.cfg, cidx, ls.sess.q_rot, L.k, L.v, ref, ls.sess.ws, lse=ref_lse)
    torch.cuda.synchronize()
    sd.check_device_error(ls.sess.ws)
    r = to_f64(ref)
    for call in range(2):
        out = torch.full_like(ls.sess.out, float("nan"))
        lse = torch.full_like(ls.lse, float("nan"))
        sd.chunk_attention_noalloc(ls.cfg, cidx, ls.sess.q_rot, L.k, L.v, out, lse=lse)
        torch.cuda.synchronize()
        got = to_f64(out)
        assert np.all(np.isfinite(got)), "call %d left unwritten outputs" % call
        err = np.abs(got - r)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, \
            "call %d: max-abs %.3g mean-abs %.3g" % (call, err.max(), err.mean())
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=1e-3, rtol=0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 16 streams x 64 heads x ceil(4352/256) = 17408 items > 16384
    w = small_workload(WORKLOADS["tiny"], batch=16, heads=64, grid_h=32, grid_w=34, chunk_frames=4,
                       sink_frames=4, window_frames=4)
    cfg = config(w)
    fake = 1 << 20      # never dereferenced: the call is rejected before anything is enqueued
    with pytest.raises(sd.SDV2Error) as e:
        sd.chunk_attention_noalloc(cfg, [0] * 16, fake, fake, fake, fake)
    assert e.value.status == 2
    assert "16384" in str(e.value)
