"""sdv2_chunk_attention_noalloc: attention without a caller-owned workspace.

Callers that cannot allocate device memory (a memory pool they do not own, a plugin host that
forbids allocation after start-up, a real-time loop that must never reach the allocator) use
this entry point; its scratch is a static array inside the library.  These tests call it
through the C ABI and check, on two calls in a row:
* its output against the fp64 oracle (the parity tolerance) and against the workspace entry
  point's output (same tolerance);
* that when the key splits' partial rows would not fit in the array the split count is reduced
  and the result still matches;
* that a bounded wait which gives up is reported by sdv2_noalloc_check_device_error, even after
  a later call, and that the next call is correct again;
* that sizes its array cannot serve are rejected.
The file is collected last so that a run stopping at the first failure has run every other
test already; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS
from gpu_common import LockStep, MAX_ABS, MEAN_ABS, config, sample_rows, small_workload, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def _stream_to(w, chunks):
    ls = LockStep(w)
    q_rot_o = None
    for c in range(chunks):
        q_rot_o = ls.step([c] * w.batch)
    return ls, q_rot_o


def _workspace_reference(ls, cidx):
    L = ls.sess.layers[0]
    ref = torch.empty_like(ls.sess.out)
    ref_lse = torch.empty_like(ls.lse)
    sd.chunk_attention(ls.cfg, cidx, ls.sess.q_rot, L.k, L.v, ref, ls.sess.ws, lse=ref_lse)
    torch.cuda.synchronize()
    sd.check_device_error(ls.sess.ws)
    return to_f64(ref), ref_lse.cpu().numpy()


def _noalloc_into_session(ls, cidx):
    """One no-alloc call writing the session's out and lse (what LockStep.check_attention reads),
    both poisoned with NaN first so that an unwritten element cannot pass."""
    L = ls.sess.layers[0]
    ls.sess.out.fill_(float("nan"))
    ls.lse.fill_(float("nan"))
    sd.chunk_attention_noalloc(ls.cfg, cidx, ls.sess.q_rot, L.k, L.v, ls.sess.out, lse=ls.lse)
    torch.cuda.synchronize()


@pytest.mark.parametrize("w,chunks", [
    (WORKLOADS["tiny"], 4),                                                                   # 2 key splits
    (small_workload(WORKLOADS["wan13b_480p"], heads=2, grid_h=10, grid_w=16, chunks=8), 8),   # 4 key splits
    (small_workload(WORKLOADS["stream_batch"], heads=3, grid_h=6, grid_w=8, chunks=3), 3),    # 4 streams
])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(w, chunks):
    ls, q_rot_o = _stream_to(w, chunks)
    cidx = [chunks - 1] * w.batch
    r, r_lse = _workspace_reference(ls, cidx)
    for call in range(2):
        _noalloc_into_session(ls, cidx)
        got = to_f64(ls.sess.out)
        assert np.all(np.isfinite(got)), "call %d left unwritten outputs" % call
        ls.check_attention(q_rot_o)                      # fp64 oracle, parity tolerance, lse
        err = np.abs(got - r)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, \
            "call %d: max-abs %.3g mean-abs %.3g" % (call, err.max(), err.mean())
        np.testing.assert_allclose(ls.lse.cpu().numpy(), r_lse, atol=1e-3, rtol=0)
    sd.noalloc_check_device_error()


# 12 heads x ceil(960/256) = 48 items: the automatic choice is 3 key splits (144 CTAs, one wave),
# whose partial rows (48 * 3 * 256) exceed the array's 32000 rows; 2 splits fit.
REDUCED = small_workload(WORKLOADS["wan13b_480p"], heads=12, grid_h=16, grid_w=20, chunks=8)


@pytest.mark.parametrize("forced", [0, 4])
def test_key_splits_are_reduced_to_fit_the_static_array(forced):
    ls, q_rot_o = _stream_to(REDUCED, REDUCED.chunks)
    cidx = [REDUCED.chunks - 1]
    rows = sample_rows(REDUCED.nq, 40, 3)
    try:
        sd.debug_set_kv_splits(forced)
        _workspace_reference(ls, cidx)
        assert sd.last_kv_splits() == (forced or 3)
        for call in range(2):
            _noalloc_into_session(ls, cidx)
            assert sd.last_kv_splits() == 2, "call %d used %d splits" % (call, sd.last_kv_splits())
            assert np.all(np.isfinite(to_f64(ls.sess.out)))
            ls.check_attention(q_rot_o, rows=rows)
        sd.noalloc_check_device_error()
    finally:
        sd.debug_set_kv_splits(0)


def test_timeout_is_reported_after_a_later_call_and_cleared_by_the_check():
    w = WORKLOADS["tiny"]
    ls, q_rot_o = _stream_to(w, 3)                       # 168 keys: two KV tiles
    cidx = [2]
    sd.noalloc_check_device_error()                       # clean so far
    try:
        sd.set_wait_timeout_ns(50_000_000)                # 50 ms
        sd.debug_drop_kv_tile(1)                          # tile 1's copy is skipped: its waits run out
        _noalloc_into_session(ls, cidx)
    finally:
        sd.debug_drop_kv_tile(-1)
        sd.set_wait_timeout_ns(2_000_000_000)
    # a later, correct call does not hide the earlier timeout
    _noalloc_into_session(ls, cidx)
    ls.check_attention(q_rot_o)
    with pytest.raises(sd.SDV2Error) as e:
        sd.noalloc_check_device_error()
    assert e.value.status == 4
    # the check cleared the error word: the next call is correct and reports nothing
    _noalloc_into_session(ls, cidx)
    ls.check_attention(q_rot_o)
    sd.noalloc_check_device_error()


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
