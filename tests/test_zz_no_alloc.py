"""awq_search_scale_static against awq_search_scale (collected last on purpose).

The static variant serves callers that cannot allocate device memory where they run the search
(a fixed memory budget set at start-up, a plug-in given a device but no allocator, a process
whose allocations belong to another runtime): its scratch is a static array inside the library.
It must give the same results as the workspace entry point, call after call, and must not
allocate. Where both entry points take the same schedule (every case here: the workspace
search gets the workspace it asks for, and the static array holds that schedule's workspace),
the results are the same bits. This file sorts last so that a run stopping at the first
failure has already run every other test.
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


# AUTO scores these layers through H = X^T X in the persistent launch, whose cross-CTA
# counters, X^T and H's triangle then live in the static array; forced to the direct scoring,
# both entry points take two residual buffers and the second stream
CASES = {
    "tiny-512": lambda: synth.make_layer("tiny-512"),
    "ragged": lambda: synth.random_layer(11, 1000, 2048, 300, n_out=10),
    "long-calibration": lambda: synth.random_layer(12, 2048, 1024, 4096, n_out=10),
}


@pytest.fixture(params=["auto", "direct"])
def score_mode(request):
    awq.awq_set_score_mode(request.param)
    yield request.param
    awq.awq_set_score_mode("auto")


@pytest.mark.parametrize("which", sorted(CASES))
def test_static_search_matches_workspace_search_on_two_calls(which, score_mode):
    d = CASES[which]()
    W = torch.from_numpy(d["W"]).cuda()
    X = torch.from_numpy(d["X"]).cuda()
    N, K = W.shape
    T = X.shape[0]
    alphas = synth.alpha_grid(20)
    assert awq.awq_search_workspace_bytes(N, K, T, 20) <= awq.SEARCH_STATIC_SCRATCH_BYTES
    want = awq.search_scale(W, X, alphas)
    awq.awq_stream_status()
    for call in range(2):
        got = _outputs(len(alphas), K)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        awq.awq_search_scale_static(W, N, K, X, T, None, alphas, len(alphas), 128, False, *got)
        awq.awq_stream_status()
        if call == 1:   # the first call may load the library's device code; later ones allocate nothing
            assert torch.cuda.mem_get_info()[0] == free_before
        for name, u, v in zip(("err", "best", "s", "inv_s"), want, got):
            assert torch.equal(u, v), (which, score_mode, call, name)
        assert np.all(np.isfinite(got[0].cpu().numpy()))


def test_static_search_rejects_shapes_beyond_its_scratch():
    """A valid 8192 x 8192 layer (real buffers of that size): one residual buffer alone is
    128 MiB, beyond the static array, so the call is refused before anything is launched."""
    N = K = 8192
    T = 64
    W = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    X = torch.zeros((T, K), dtype=torch.float16, device="cuda")
    err, best, s, inv = _outputs(20, K)
    need = awq.awq_search_workspace_bytes(N, K, T, 20)
    assert need > awq.SEARCH_STATIC_SCRATCH_BYTES
    with pytest.raises(awq.AwqError) as ei:
        awq.awq_search_scale_static(W, N, K, X, T, None, synth.alpha_grid(20), 20, 128, False,
                                    err, best, s, inv)
    assert ei.value.name == "AWQ_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert torch.isnan(err).all() and int(best.item()) == -1   # nothing was launched
