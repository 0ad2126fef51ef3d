"""The attention kernel's bounded waits: when a K/V tile never arrives (its copy is skipped on
purpose through the library's fault-injection switch), every waiting role gives up after the
configured limit, the kernel records a timeout in the workspace error word and returns; the
host reads SDV2_ERR_TIMEOUT and the context stays usable for the next, correct call.
Nothing here faults, traps or spins without a limit."""
import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from synth_inputs import WORKLOADS, qkv_chunk_host
from gpu_common import LockStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def test_missing_tile_times_out_and_context_survives():
    w = WORKLOADS["tiny"]
    ls = LockStep(w)
    for c in range(3):                      # 168 keys: two KV tiles
        q_rot_o = ls.step([c])
    ls.check_attention(q_rot_o)
    sd.check_device_error(ls.sess.ws)       # clean so far
    try:
        sd.set_wait_timeout_ns(50_000_000)  # 50 ms
        sd.debug_drop_kv_tile(1)
        sd.chunk_attention(ls.cfg, [2], ls.sess.q_rot, ls.sess.layers[0].k, ls.sess.layers[0].v,
                           ls.sess.out, ls.sess.ws)
        with pytest.raises(sd.SDV2Error) as e:
            sd.check_device_error(ls.sess.ws)
        assert e.value.status == 4
    finally:
        sd.debug_drop_kv_tile(-1)
        sd.set_wait_timeout_ns(2_000_000_000)
    # the error word was cleared by the check; a normal call works and is correct again
    sd.chunk_attention(ls.cfg, [2], ls.sess.q_rot, ls.sess.layers[0].k, ls.sess.layers[0].v,
                       ls.sess.out, ls.sess.ws, lse=ls.lse)
    sd.check_device_error(ls.sess.ws)
    ls.check_attention(q_rot_o)
