"""The clipping search's fp32 criterion, emulated on the CPU step by step as the GPU kernel forms
it, stays within the bound the GPU parity test allows (tests/clip_bound.py) of the oracle's fp64
error: w' = fl32(w s), r = fl32(w' - (code - zero) step16) rounded once, g = fl32(h / fl32(s^2)),
and the terms g r^2 summed in fp32 in the kernel's order (two chains of element pairs per
32-channel run, then the run's four partial sums, then the runs of a group). The codes are the
oracle's (the GPU's are bit-exact against them in the parity tests)."""

import numpy as np
import pytest

from oracle import awq_ref as ref
from post_weight_quantization_stats_b300 import synth
from tests.clip_bound import criterion_bound

f32 = np.float32


def _emulated_criterion(W16, s, ratios, G, sym, bits, h):
    N, K = W16.shape
    ng = K // G
    w = W16.astype(f32)
    sv = s.astype(f32) if s is not None else np.ones(K, f32)
    wp = (w * sv[None, :]).astype(f32)                                  # fl32(w s)
    g = (h.astype(f32) / (sv * sv).astype(f32)).astype(f32)            # fl32(h / fl32(s^2))
    out = np.zeros((len(ratios), N, ng))
    for j, c in enumerate(ratios):
        qd = ref.quantize_pack(W16, s, G, sym, bits, clip=np.full((N, ng), c, f32))
        codes = ref.unpack_nibbles(qd["qweight"]).astype(np.float64)
        zero = np.asarray(qd["zeros"], np.float64).T if not sym else np.full((N, ng), 8.0)
        step16 = np.asarray(qd["scales"], np.float16).astype(np.float64).T
        gk = np.arange(K) // G
        qz_step = (codes - zero[:, gk]) * step16[:, gk]                 # exact in fp32
        r = (wp.astype(np.float64) - qz_step).astype(f32)               # one rounding
        gr = (g[None, :] * r).astype(f32)
        term_x = lambda acc, k: (gr[:, k].astype(np.float64) * r[:, k] + acc).astype(f32)
        run = 32 if G >= 32 else G
        for gi in range(ng):
            runs = []
            for t in range(G // run):
                k0 = gi * G + t * run
                e = [[np.zeros(N, f32), np.zeros(N, f32)] for _ in range(2)]   # e[chain][x|y]
                for p in range(run // 2):
                    ch = p & 1
                    e[ch][0] = term_x(e[ch][0], k0 + 2 * p)
                    e[ch][1] = term_x(e[ch][1], k0 + 2 * p + 1)
                runs.append(((e[0][0] + e[0][1]).astype(f32) + (e[1][0] + e[1][1]).astype(f32))
                            .astype(f32))
            while len(runs) > 1:                                        # butterfly over the team
                half = len(runs) // 2
                runs = [(runs[i] + runs[i + half]).astype(f32) for i in range(half)]
            out[j, :, gi] = runs[0]
    return out


@pytest.mark.parametrize("G,sym,bits", [(128, False, 4), (64, True, 4), (32, False, 3),
                                        (128, False, 2)])
def test_fp32_criterion_within_the_gpu_tests_bound(G, sym, bits):
    d = synth.random_layer(G + bits, 24, 512, 96, n_out=5)
    rng = np.random.Generator(np.random.PCG64(G * bits))
    s = np.exp(rng.uniform(-0.5, 1.0, 512)).astype(np.float32)
    h = ref.channel_energy(d["X"])
    ratios = ref.clip_ratio_grid(10)
    exact = ref.clip_search(d["W"], None, s, ratios, G, sym, bits, h=h)["err"]
    got = _emulated_criterion(d["W"], s, ratios, G, sym, bits, h)
    bound = criterion_bound(d["W"], s, ratios, G, sym, bits, h)
    gap = np.abs(got - exact)
    assert np.all(gap <= bound), float(np.max(gap / np.maximum(bound, 1e-300)))
    # the bound is not vacuous: the emulated errors use a fair share of it somewhere
    assert np.max(gap / np.maximum(bound, 1e-300)) > 1e-3
