"""The attention softmax's FMA-pipe 2^x on the GPU (through sdv2_debug_exp2), against the exact
2^x, against CUDA's ex2.approx.ftz.f32 on the same inputs, and against the CPU model of its
fp32 arithmetic."""
import numpy as np
import pytest
import torch

import streaming_causal_video_gb300 as sd
from streaming_causal_video_gb300 import exp2_poly
from test_exp2_poly import kernel_coefficients

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()


def _run(x):
    xd = torch.from_numpy(x).cuda()
    yf = torch.empty_like(xd)
    ym = torch.empty_like(xd)
    sd.debug_exp2(xd, yf, ym)
    torch.cuda.synchronize()
    return yf.cpu().numpy(), ym.cpu().numpy()


def test_fma_exp2_matches_exact_mufu_and_model():
    rng = np.random.default_rng(5)
    x = np.concatenate([np.linspace(-125, 8, 2_000_000), rng.uniform(-20, 8, 1_000_000),
                        -np.arange(0, 126)]).astype(np.float32)
    x = x[: x.size // 2 * 2]
    yf, ym = _run(x)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(yf / exact - 1)
    assert rel.max() <= 7.6e-5, (rel.max(), x[rel.argmax()])
    rel_m = np.abs(ym / exact - 1)
    assert rel_m.max() <= 1e-6                          # ex2.approx itself, for scale
    assert np.abs(yf / ym.astype(np.float64) - 1).max() <= 7.7e-5
    model = exp2_poly.model_f32(x, kernel_coefficients())
    same = yf.view(np.uint32) == model.view(np.uint32)
    assert same.mean() >= 1 - 1e-6, same.mean()
    ulp = np.abs(yf.view(np.int32).astype(np.int64) - model.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1


def test_fma_exp2_far_below_the_range_and_masked_scores():
    x = np.array([-np.inf, -1e30, -1000, -127, -126.5, -126, 0, 8], np.float32)
    yf, _ = _run(x)
    assert np.all(np.isfinite(yf)) and np.all(yf > 0)
    assert np.all(yf[:6] <= np.float32(2.0 ** -125))
    np.testing.assert_allclose(yf[6:], [1.0, 256.0], rtol=7.6e-5)
