"""The scale grid's power on the GPU: s = max(m, 1e-6)^alpha in fp32, formed from an fp64
logarithm and product and an fp32 exp2f of the fractional part, lies within 3 fp32 spacings of
the exact power (the kernel's stated bound) over statistics spread log-uniformly from below the
floor to the fp16 maximum, for alphas across the grid; 1/s is the IEEE quotient of that s. The
search is fed each alpha alone with the statistic given, so the s it returns is that alpha's."""

import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from post_weight_quantization_stats_b300 import awq, build  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    awq.lib()
    torch.cuda.set_device(0)
    yield
    awq.awq_stream_status()


def _ulps(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Distance in fp32 spacings at the exact value's binade."""
    e = np.floor(np.log2(want))
    return np.abs(got.astype(np.float64) - want) / np.exp2(e - 23)


def test_scale_grid_power_within_three_spacings():
    K = 4096
    rng = np.random.Generator(np.random.PCG64(41))
    m = np.exp(rng.uniform(math.log(1e-7), math.log(65504.0), K)).astype(np.float32)
    m[:4] = [0.0, 1e-6, 1.0, 65504.0]
    base = np.maximum(m.astype(np.float64), 1e-6)
    W = torch.randn((128, K), device="cuda").half()
    X = torch.randn((64, K), device="cuda").half()
    mean_abs = torch.from_numpy(m).cuda()
    worst = 0.0
    for a in (0.0, 0.05, 0.35, 0.5, 0.65, 0.95, 1.0 / 3.0):
        a32 = np.float32(a)
        _, _, s, inv_s = awq.search_scale(W, X, [float(a32)], mean_abs=mean_abs)
        awq.awq_stream_status()
        sg = s.cpu().numpy()
        want = base ** float(a32)
        u = _ulps(sg, want)
        worst = max(worst, float(u.max()))
        assert np.all(u <= 3.0), (a, float(u.max()), int(np.argmax(u)))
        np.testing.assert_array_equal(inv_s.cpu().numpy(), (np.float32(1) / sg).astype(np.float32))
    print(f"scale grid: worst distance {worst:.2f} fp32 spacings")
