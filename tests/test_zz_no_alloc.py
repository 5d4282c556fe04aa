"""awq_search_scale_static against awq_search_scale (collected last on purpose).

The static variant serves callers that cannot allocate device memory where they run the search
(a fixed memory budget set at start-up, a plug-in given a device but no allocator, a process
whose allocations belong to another runtime): its scratch is a static array inside the library.
It must give the same results as the workspace entry point, call after call, and must not
allocate. This file sorts last so that a run stopping at the first failure has already run every
other test.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from post_weight_quantization_stats_b300 import awq, build, synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    awq.lib()
    torch.cuda.set_device(0)


def _outputs(n_alpha, K):
    return (torch.full((n_alpha,), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((K,), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((K,), float("nan"), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("which", ["tiny-512", "ragged"])
def test_static_search_matches_workspace_search_on_two_calls(which):
    d = synth.make_layer("tiny-512") if which == "tiny-512" else \
        synth.random_layer(11, 1000, 2048, 300, n_out=10)
    W = torch.from_numpy(d["W"]).cuda()
    X = torch.from_numpy(d["X"]).cuda()
    N, K = W.shape
    T = X.shape[0]
    alphas = synth.alpha_grid(20)
    ref_err, ref_best, ref_s, ref_inv = awq.search_scale(W, X, alphas)
    awq.awq_stream_status()
    for call in range(2):
        err, best, s, inv = _outputs(len(alphas), K)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        awq.awq_search_scale_static(W, N, K, X, T, None, alphas, len(alphas), 128, False, err,
                                    best, s, inv)
        awq.awq_stream_status()
        if call == 1:   # the first call may load the library's device code; later ones allocate nothing
            assert torch.cuda.mem_get_info()[0] == free_before
        np.testing.assert_allclose(err.cpu().numpy(), ref_err.cpu().numpy(), rtol=1e-3, atol=0)
        assert int(best.item()) == int(ref_best.item())
        np.testing.assert_allclose(s.cpu().numpy(), ref_s.cpu().numpy(), rtol=1e-6, atol=0)
        np.testing.assert_allclose(inv.cpu().numpy(), ref_inv.cpu().numpy(), rtol=1e-6, atol=0)


def test_static_search_rejects_shapes_beyond_its_scratch():
    W = torch.zeros((16, 256), dtype=torch.float16, device="cuda")
    X = torch.zeros((16, 256), dtype=torch.float16, device="cuda")
    err, best, s, inv = _outputs(20, 256)
    need = awq.awq_search_workspace_bytes(8192, 8192, 4096, 20)
    assert need > awq.SEARCH_STATIC_SCRATCH_BYTES
    with pytest.raises(awq.AwqError) as ei:
        awq.awq_search_scale_static(W, 8192, 8192, X, 4096, None, synth.alpha_grid(20), 20, 128,
                                    False, err, best, s, inv)
    assert ei.value.name == "AWQ_ERR_WORKSPACE"
    assert torch.isnan(err).all()          # nothing was launched
