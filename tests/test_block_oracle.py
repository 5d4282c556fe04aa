"""The block oracle (fold of 1/s, RMSNorm, silu * up, the AWQ flow over an MLP block) against
closed forms and invariants ("AWQ Math", "The equivalent transform"; "AWQ > Benefits and
Practical Considerations": the scale folds into the previous layer)."""

import numpy as np
import pytest

from oracle import awq_ref as ref
from oracle import block_ref as blk


def _block(seed, D=64, I=128):
    """Weights whose magnitudes stay in fp16's normal range under scaling by 2^-2 .. 2^2."""
    rng = np.random.Generator(np.random.PCG64(seed))

    def w(n, k):
        a = rng.standard_normal((n, k))
        a = np.sign(a) * np.clip(np.abs(a), 2.0 ** -6, 8.0)
        return a.astype(np.float16)
    gamma = (1.0 + 0.25 * rng.standard_normal(D)).astype(np.float16)
    return gamma, w(I, D), w(I, D), w(D, I)


def _scaled_cols(W16, s):
    return (W16.astype(np.float64) * s[None, :]).astype(np.float16)


def test_fold_with_power_of_two_scales_is_exact():
    """With s_1 and s_2 powers of two every rounding commutes with the scaling, so the folded
    block (gamma / s_1; W_gate, W_up diag(s_1); rows of W_up / s_2; W_down diag(s_2)) gives the
    unfolded block's output bit for bit. Folding 1/s_2 into the wrong operation (gate's rows)
    does not, since silu is not linear."""
    gamma, Wg, Wu, Wd = _block(1)
    D, I = Wg.shape[1], Wg.shape[0]
    rng = np.random.Generator(np.random.PCG64(2))
    X = (rng.standard_normal((16, D)) * 2).astype(np.float16)
    s1 = 2.0 ** rng.integers(-2, 3, D)
    s2 = 2.0 ** rng.integers(-2, 3, I)
    want = blk.mlp_fp16(X, gamma, Wg, Wu, Wd)["y"]
    g_f = blk.scale_rows(gamma, (1.0 / s1).astype(np.float32))
    Wu_f = blk.scale_rows(Wu, (1.0 / s2).astype(np.float32))
    got = blk.mlp_fp16(X, g_f, _scaled_cols(Wg, s1), _scaled_cols(Wu_f, s1),
                       _scaled_cols(Wd, s2))["y"]
    assert np.array_equal(got, want)
    Wg_wrong = blk.scale_rows(Wg, (1.0 / s2).astype(np.float32))
    bad = blk.mlp_fp16(X, g_f, _scaled_cols(Wg_wrong, s1), _scaled_cols(Wu, s1),
                       _scaled_cols(Wd, s2))["y"]
    assert not np.array_equal(bad, want)


def test_scale_rows_rounding():
    """One fp32 multiply rounded to fp16: identity for 1, exact for powers of two, sign-odd,
    and fp16's round-to-nearest-even on an exact half-way product."""
    A = np.array([[1.0, -3.0, 0.5], [6.0, 2.0 ** -10, -7.0]], np.float16)
    assert np.array_equal(blk.scale_rows(A, np.ones(2, np.float32)), A)
    B = blk.scale_rows(A, np.array([0.25, 8.0], np.float32))
    assert np.array_equal(B.astype(np.float64), A.astype(np.float64) * np.array([[0.25], [8.0]]))
    assert np.array_equal(blk.scale_rows(-A, np.array([3.0, 5.0], np.float32)),
                          -blk.scale_rows(A, np.array([3.0, 5.0], np.float32)))
    # 2049 * 1 is exact in fp32 and half-way between fp16's 2048 and 2050: even wins
    C = np.array([[2049.0]], np.float32).astype(np.float16)   # already 2048 in fp16
    assert float(C[0, 0]) == 2048.0
    D = blk.scale_rows(np.array([[683.0]], np.float16), np.array([3.0], np.float32))
    assert float(D[0, 0]) == 2048.0                            # 2049 -> 2048 (ties to even)


def test_rmsnorm_closed_forms():
    """A constant row c normalises to sign(c) * gamma (eps = 0); rows of +-a likewise; scaling
    the input by 2 leaves the output unchanged."""
    D = 16
    gamma = np.linspace(0.5, 2.0, D).astype(np.float16)
    X = np.stack([np.full(D, 3.0), np.full(D, -0.75),
                  np.tile([2.5, -2.5], D // 2)]).astype(np.float16)
    Y = blk.rmsnorm(X, gamma, eps=0.0).astype(np.float64)
    g = gamma.astype(np.float64)
    assert np.array_equal(Y[0], g)
    assert np.array_equal(Y[1], -g)
    assert np.array_equal(Y[2], np.tile([1.0, -1.0], D // 2) * g)
    rng = np.random.Generator(np.random.PCG64(3))
    Z = rng.standard_normal((5, D)).astype(np.float16)
    assert np.array_equal(blk.rmsnorm(Z, gamma, 0.0), blk.rmsnorm((Z.astype(np.float64) * 2).astype(np.float16), gamma, 0.0))


def test_silu_identities():
    """silu(0) = 0, silu(g) - silu(-g) = g, silu -> g for large g and -> 0 for very negative g."""
    g = np.array([0.0, 0.5, 1.5, 3.0, 20.0, -20.0], np.float16)
    one = np.ones_like(g)
    s = blk.silu_mul(g, one).astype(np.float64)
    sn = blk.silu_mul(-g, one).astype(np.float64)
    assert s[0] == 0.0
    gg = g.astype(np.float64)
    assert np.all(np.abs((s - sn) - gg) <= 2 * np.abs(gg) * 2.0 ** -10 + 1e-7)
    assert s[4] == 20.0 and abs(s[5]) < 1e-6
    u = np.array([2.0, -1.0, 4.0, 0.5, 1.0, 1.0], np.float16)
    assert np.array_equal(blk.silu_mul(g, u)[:4].astype(np.float64) != 0, np.array([False, True, True, True]))


def test_alpha_zero_is_rtn():
    """With alpha = 0 only, s = 1: nothing is folded and the three packs are plain RTN."""
    gamma, Wg, Wu, Wd = _block(4, D=128, I=256)
    rng = np.random.Generator(np.random.PCG64(5))
    X = rng.standard_normal((32, 128)).astype(np.float16)
    q = blk.quantize_mlp(X, gamma, Wg, Wu, Wd, [0.0], group_size=64)
    assert np.array_equal(q["gamma"], gamma) and np.array_equal(q["Wu"], Wu)
    for name, W in (("gate", Wg), ("up", Wu), ("down", Wd)):
        r = ref.quantize_pack(W, None, 64)
        assert np.array_equal(q[name]["qweight"], r["qweight"])
        assert np.array_equal(q[name]["scales"], r["scales"])


def test_awq_block_beats_rtn_on_outlier_inputs():
    """On inputs with a few outsized channels, the searched scales give a smaller block output
    error than plain RTN (the search can only do as well or better per linear, since alpha = 0
    is on the grid)."""
    D, I, T = 128, 256, 64
    rng = np.random.Generator(np.random.PCG64(6))
    gamma = np.ones(D, np.float16)
    Wg, Wu = (rng.standard_normal((I, D)) * 0.05).astype(np.float16), (rng.standard_normal((I, D)) * 0.05).astype(np.float16)
    Wd = (rng.standard_normal((D, I)) * 0.05).astype(np.float16)
    X = rng.standard_normal((T, D))
    X[:, [3, 50, 97]] *= 30
    X = X.astype(np.float16)
    alphas = np.arange(10) / 10
    want = blk.mlp_fp16(X, gamma, Wg, Wu, Wd)["y"].astype(np.float64)
    q = blk.quantize_mlp(X, gamma, Wg, Wu, Wd, alphas, group_size=64)
    q0 = blk.quantize_mlp(X, gamma, Wg, Wu, Wd, [0.0], group_size=64)
    e_awq = np.mean((blk.mlp_quantized(X, q, 64)["y"].astype(np.float64) - want) ** 2)
    e_rtn = np.mean((blk.mlp_quantized(X, q0, 64)["y"].astype(np.float64) - want) ** 2)
    assert q["r1"]["best"] > 0 and e_awq < e_rtn, (q["r1"]["best"], e_awq, e_rtn)
