"""GPU: folding 1/s into the previous operation, the block's elementwise operations, and AWQ on
a stack of Llama-style MLP blocks end to end, against the CPU oracle (staged: each stage of the
oracle is fed the GPU's inputs to that stage, so decisions are compared on equal terms)."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from oracle import awq_ref as ref  # noqa: E402
from oracle import block_ref as blk  # noqa: E402
from post_weight_quantization_stats_b300 import awq, block, build, synth  # noqa: E402


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


def _ulps16(a, b):
    """|a - b| in units of fp16 spacing at max(|a|, |b|) (normal range)."""
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    m = np.maximum(np.abs(a), np.abs(b))
    ulp = np.where(m >= 2.0 ** -14, 2.0 ** (np.floor(np.log2(np.maximum(m, 2.0 ** -14))) - 10),
                   2.0 ** -24)
    return np.abs(a - b) / ulp


@pytest.mark.parametrize("rows,cols,lda", [(300, 136, 136), (7, 64, 72), (4096, 1, 1),
                                           (33, 5, 7), (1, 8, 8)])
def test_scale_rows_bitexact(rows, cols, lda):
    rng = np.random.Generator(np.random.PCG64(rows * 3 + cols))
    full = (rng.standard_normal((rows, lda)) * 4).astype(np.float16)
    r = np.exp(rng.uniform(-3, 3, rows)).astype(np.float32)
    A = dev(full.reshape(-1))
    awq.awq_scale_rows(A, rows, cols, lda, dev(r))
    awq.awq_stream_status()
    got = host(A).reshape(rows, lda)
    assert np.array_equal(got[:, :cols], blk.scale_rows(full[:, :cols], r))
    assert np.array_equal(got[:, cols:], full[:, cols:])      # padding untouched


@pytest.mark.parametrize("T,D", [(77, 4096), (5, 8), (256, 512)])
def test_rmsnorm(T, D):
    rng = np.random.Generator(np.random.PCG64(T + D))
    X = (rng.standard_normal((T, D)) * 3).astype(np.float16)
    g = (1 + 0.3 * rng.standard_normal(D)).astype(np.float16)
    got = host(block.rmsnorm(dev(X), dev(g), 1e-6))
    assert np.max(_ulps16(got, blk.rmsnorm(X, g, 1e-6))) <= 1.0


def test_silu_mul():
    rng = np.random.Generator(np.random.PCG64(9))
    G = (rng.standard_normal(8000) * 4).astype(np.float16)
    U = (rng.standard_normal(8000) * 2).astype(np.float16)
    got = host(block.silu_mul(dev(G), dev(U)))
    assert np.max(_ulps16(got, blk.silu_mul(G, U))) <= 1.0


def _weights(seed, D, I):
    rng = np.random.Generator(np.random.PCG64(seed))
    return block.MLPWeights(
        gamma=dev((1 + 0.2 * rng.standard_normal(D)).astype(np.float16)),
        W_gate=dev(synth.draw_weight(rng, I, D, 0.03)),
        W_up=dev(synth.draw_weight(rng, I, D, 0.03)),
        W_down=dev(synth.draw_weight(rng, D, I, 0.03)))


def _check_alpha(err_gpu, best_gpu, r):
    """The GPU's choice equals the oracle's unless the oracle's own errors are a near-tie."""
    if best_gpu != r["best"]:
        e = r["err"]
        assert e[best_gpu] <= e[r["best"]] * (1 + 1e-4), (best_gpu, r["best"], e)
    np.testing.assert_allclose(err_gpu, r["err"], rtol=1e-3)


def test_awq_mlp_stack_end_to_end():
    """Two MLP blocks (D = 512, I = 1024, 512 calibration tokens with 1% outlier channels):
    per block, the alpha of gate/up and of down against the oracle's search on the same inputs,
    the folded norm weight and up rows bit-exact, the packs bit-exact, the quantised block's
    output within 2e-2 of max |oracle|; and the stack's output error below plain RTN's."""
    D, I, T, G = 512, 1024, 512, 128
    rng = np.random.Generator(np.random.PCG64(11))
    X16, _ = synth.draw_activations(rng, T, D, n_out=5, mult=20.0, student_t=False)
    blocks = [_weights(21, D, I), _weights(22, D, I)]
    alphas = synth.alpha_grid(20)
    X = dev(X16)
    q = block.quantize_stack(X, blocks, alphas, G)
    awq.awq_stream_status()
    x = X
    for w, qb in zip(blocks, q):
        fp = block.mlp_fp16(x, w)
        Wgu = np.concatenate([host(w.W_gate), host(w.W_up)], axis=0)
        r1 = ref.search_scale(Wgu, host(fp["xn"]), alphas, G)
        r2 = ref.search_scale(host(w.W_down), host(fp["h"]), alphas, G)
        _check_alpha(host(qb.err1).astype(np.float64), qb.best1, r1)
        _check_alpha(host(qb.err2).astype(np.float64), qb.best2, r2)
        s1, s2 = host(qb.s1), host(qb.s2)
        inv1 = (np.float32(1) / s1).astype(np.float32)
        inv2 = (np.float32(1) / s2).astype(np.float32)
        assert np.array_equal(host(qb.gamma), blk.scale_rows(host(w.gamma), inv1))
        Wu_f = blk.scale_rows(host(w.W_up), inv2)
        for got, W, s in ((qb.gate, host(w.W_gate), s1), (qb.up, Wu_f, s1),
                          (qb.down, host(w.W_down), s2)):
            want = ref.quantize_pack(W, s, G)
            assert np.array_equal(host(got[0]).view(np.uint32), want["qweight"])
            assert np.array_equal(host(got[1]), want["scales"])
            assert np.array_equal(host(got[2]), want["zeros"])
        out = block.mlp_quantized(x, qb)
        qd = {"gamma": host(qb.gamma),
              "gate": {"qweight": host(qb.gate[0]).view(np.uint32), "scales": host(qb.gate[1]),
                       "zeros": host(qb.gate[2])},
              "up": {"qweight": host(qb.up[0]).view(np.uint32), "scales": host(qb.up[1]),
                     "zeros": host(qb.up[2])},
              "down": {"qweight": host(qb.down[0]).view(np.uint32), "scales": host(qb.down[1]),
                       "zeros": host(qb.down[2])}}
        # each product checked on the GPU's own input to it
        want = blk.mlp_quantized(host(x), qd, G, xn=host(out["xn"]), h=host(out["h"]))
        for name in ("g", "u", "y"):
            a, b = host(out[name]).astype(np.float64), want[name].astype(np.float64)
            assert np.max(np.abs(a - b)) <= 2e-2 * np.max(np.abs(b)), name
        x = fp["y"]
    y_fp = x.float()
    y_awq = block.run_stack(X, q).float()
    q0 = block.quantize_stack(X, blocks, np.zeros(1, np.float32), G)
    y_rtn = block.run_stack(X, q0).float()
    awq.awq_stream_status()
    e_awq = torch.mean((y_awq - y_fp) ** 2).item()
    e_rtn = torch.mean((y_rtn - y_fp) ** 2).item()
    assert e_awq < e_rtn, (e_awq, e_rtn)


def test_stack_run_resumes_bit_identically(tmp_path):
    """Three linears through the resumable stack run on the GPU quantiser: stopped after the
    second, restarted, the results equal an uninterrupted run's bit for bit, and the first
    layer's alpha equals the oracle's search on the same statistic."""
    from post_weight_quantization_stats_b300 import stack

    def layers():
        out = []
        for i in range(3):
            d = synth.random_layer(40 + i, 256, 512, 300, n_out=5)
            out.append((i, f"l{i}", lambda d=d: (dev(d["W"]), dev(d["X"]))))
        return out

    alphas = synth.alpha_grid(20)
    q = stack.gpu_quantizer(alphas)
    clean = str(tmp_path / "clean")
    want = stack.quantize_layers(layers(), clean, q)

    class Stop(Exception):
        pass

    def stop(i):
        if i == 1:
            raise Stop()
    d = str(tmp_path / "run")
    with pytest.raises(Stop):
        stack.quantize_layers(layers(), d, q, on_layer=stop)
    got = stack.quantize_layers(layers(), d, q)
    assert sorted(got) == [0, 1, 2]
    for i in range(3):
        a, b = stack.load_layer(clean, want[i]), stack.load_layer(d, got[i])
        for k in a:
            assert np.array_equal(a[k], b[k]), (i, k)
    l0 = synth.random_layer(40, 256, 512, 300, n_out=5)
    r = ref.search_scale(l0["W"], l0["X"], alphas, m=stack.load_layer(d, got[0])["m"])
    b = int(stack.load_layer(d, got[0])["best"])
    assert b == r["best"] or r["err"][b] <= r["err"][r["best"]] * (1 + 1e-4)
