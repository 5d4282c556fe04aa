"""GPU parity of the per-group clipping search and the clipped pack against the CPU oracle.

The clip ratio of a group is an integer decision taken on a floating-point criterion: the GPU
accumulates e(c) = sum_k h_k (W - w_hat)^2 in fp32, the oracle in fp64 from the GPU's channel
energy h. The GPU's ratio must be the oracle's first minimiser unless the oracle's errors of
the two ratios lie within the bound of the GPU's fp32 arithmetic (each d = W - w_hat off by at
most 2^-22 (|W| + |w_hat|), the sum over G terms by G 2^-24 relative); each such near-tie is
counted and printed. The packed codes, steps and zero points for the GPU's ratios are bit-exact
against the oracle's quantiser fed the same ratios.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from oracle import awq_ref as ref  # noqa: E402
from post_weight_quantization_stats_b300 import awq, build, synth  # noqa: E402
from tests.clip_bound import criterion_bound as _criterion_bound  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    awq.lib()
    torch.cuda.set_device(0)
    yield
    awq.awq_stream_status()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


def _check_clip(W16, X16, s, G, sym, bits, rows=None):
    ratios = ref.clip_ratio_grid(10)
    W, X = dev(W16), dev(X16)
    clip, energy = awq.clip_search(W, X, dev(s) if s is not None else None, ratios, G, sym,
                                   bits=bits)
    awq.awq_stream_status()
    h = host(energy).astype(np.float64)
    np.testing.assert_allclose(h, ref.channel_energy(X16), rtol=1e-5, atol=0)
    got = host(clip).T                                     # [N, K/G]
    assert np.all(np.isin(got, ratios))
    Wr = W16 if rows is None else W16[rows]
    gr = got if rows is None else got[rows]
    r = ref.clip_search(Wr, None, s, ratios, G, sym, bits, h=h)
    gi = np.searchsorted(-ratios, -gr)                     # index of each chosen ratio
    assert np.array_equal(ratios[gi], gr)
    mism = np.argwhere(gi != r["best"])
    near = 0
    if len(mism):
        bound = _criterion_bound(Wr, s, ratios, G, sym, bits, h)
        for n, g in mism:
            a, b = gi[n, g], r["best"][n, g]
            e = r["err"][:, n, g]
            assert e[a] - e[b] <= bound[a, n, g] + bound[b, n, g], (n, g, a, b, e)
            near += 1
    # packing with the GPU's ratios: bit-exact against the oracle quantiser fed them
    q, sc, z = awq.quantize_pack_clip(W, dev(s) if s is not None else None, clip, G, sym,
                                      bits=bits)
    awq.awq_stream_status()
    want = ref.quantize_pack(Wr, s, G, sym, bits, clip=gr)
    qh, sch, zh = host(q).view(np.uint32), host(sc), host(z)
    if rows is not None:
        qh, sch, zh = qh[rows], sch[:, rows], zh[:, rows]
    assert np.array_equal(qh, want["qweight"])
    assert np.array_equal(sch, want["scales"])
    if not sym:
        assert np.array_equal(zh, want["zeros"])
    clipped = float(np.mean(gi > 0))
    print(f"clip {Wr.shape} G={G} sym={sym} bits={bits}: {clipped:.1%} of groups clipped, "
          f"{near} near-ties of {gi.size}")
    return gi, r


CLIP_CASES = [(300, 1152, 200, 128, False, 4), (256, 512, 64, 64, True, 4),
              (1, 128, 8, 128, False, 4), (130, 256, 100, 32, False, 4),
              (200, 1024, 150, 128, False, 3), (64, 512, 96, 64, True, 3),
              (96, 256, 40, 32, True, 2), (160, 384, 50, 64, False, 2)]


@pytest.mark.parametrize("N,K,T,G,sym,bits", CLIP_CASES)
def test_clip_search_matches_oracle(N, K, T, G, sym, bits):
    d = synth.random_layer(N + K + T + G, N, K, T, n_out=max(1, K // 100))
    rng = np.random.Generator(np.random.PCG64(N * K))
    s = np.exp(rng.uniform(-0.5, 1.0, K)).astype(np.float32)
    _check_clip(d["W"], d["X"], s, G, sym, bits)
    _check_clip(d["W"], d["X"], None, G, sym, bits)


def test_clip_of_ones_is_the_plain_pack():
    d = synth.random_layer(77, 96, 512, 32)
    W = dev(d["W"])
    ones = torch.ones((512 // 128, 96), dtype=torch.float32, device="cuda")
    for sym in (False, True):
        a = awq.quantize_pack(W, None, 128, sym)
        b = awq.quantize_pack_clip(W, None, ones, 128, sym)
        awq.awq_stream_status()
        # symmetric packs write no zero points: compare codes and steps only
        for u, v in zip(a if not sym else a[:2], b if not sym else b[:2]):
            assert torch.equal(u, v)


@pytest.mark.slow
def test_clip_search_full_size_sampled_rows():
    """The benchmark layer (4096 x 4096, T = 8192) with the searched scale, in one launch over
    all rows: ratios and packed codes of 64 sampled rows against the oracle."""
    d = synth.make_layer("llama7b-attn-4096")
    W, X = dev(d["W"]), dev(d["X"])
    err, best, s, inv_s = awq.search_scale(W, X, synth.alpha_grid(20))
    awq.awq_stream_status()
    rows = np.sort(np.random.Generator(np.random.PCG64(3)).choice(4096, 64, replace=False))
    gi, r = _check_clip(d["W"], d["X"], host(s), 128, False, 4, rows=rows)
    # each sampled group's criterion at its ratio is never above its unclipped one
    e_at = np.take_along_axis(r["err"], gi[None], axis=0)[0]
    assert np.all(e_at <= r["err"][0] * (1 + 1e-5))


CLIP_WORKLOAD_LAYERS = [("llama7b-mlp", 0), ("llama7b-mlp", 2), ("llama70b-mlp", 0),
                        ("llama70b-mlp", 1)]


@pytest.mark.slow
@pytest.mark.parametrize("wl,i", CLIP_WORKLOAD_LAYERS)
def test_clip_search_workload_sampled_rows(wl, i):
    """The MLP workloads' layers at full size (K up to 28672, T = 8192 and 4096, the gated input
    of the down-projections), one launch over all rows with the scale of alpha = 0.5 from the
    GPU's statistic: ratios, energies and clipped packs of 64 sampled rows against the
    oracle."""
    d = synth.make_layer(wl, i)
    X = dev(d["X"])
    m = host(awq.calib_stats(X))
    s = ref.fl32(ref.scale_grid(m, [0.5]))[0].astype(np.float32)
    N = d["W"].shape[0]
    rows = np.sort(np.random.Generator(np.random.PCG64(N + i)).choice(N, 64, replace=False))
    del X
    _check_clip(d["W"], d["X"], s, 128, False, 4, rows=rows)
