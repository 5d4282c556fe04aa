"""Pins that tie the CPU oracle to what the AWQ pages and plain mathematics fix.

Every ``pin_*`` takes the oracle module ``o`` and raises ``AssertionError`` when the oracle
disagrees with a closed form, an invariant, a worked example printed on the pages, or a
brute-force computation. The same functions run against deliberately broken copies of the
oracle (see ``test_oracle_mutations.py``) to show that a plausible mistake anywhere in it is
caught by at least one of them.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _ladder_group(levels, z0, e, G):
    """A group of G values (j - z0) * 2^-e cycling through ``levels`` (exact in fp16)."""
    vals = [(levels[i % len(levels)] - z0) * 2.0 ** (-e) for i in range(G)]
    return np.array(vals, dtype=np.float64)


# ------------------------------------------------------------------ calibration statistic

def pin_calib_stats_closed_form(o):
    """m_j = average |x_j| ("AWQ Math", "Saliency is an activation property")."""
    T, K = 6, 16
    c = (np.arange(K) - 7.5).astype(np.float16)            # exact halves
    sign = np.array([(-1) ** t for t in range(T)], dtype=np.float16)
    X = (sign[:, None] * c[None, :]).astype(np.float16)
    m = o.calib_stats(X)
    assert np.array_equal(m, np.abs(c.astype(np.float64))), m
    # a column holding 0, 1, ..., T-1 averages to (T - 1) / 2
    X2 = np.zeros((T, K), np.float16)
    X2[:, 3] = np.arange(T)
    assert o.calib_stats(X2)[3] == (T - 1) / 2
    # brute force (math.fsum over every element) on random data
    rng = np.random.Generator(np.random.PCG64(7))
    X3 = rng.standard_normal((9, 5)).astype(np.float16)
    ref = [math.fsum(abs(float(X3[t, j])) for t in range(9)) / 9 for j in range(5)]
    assert np.allclose(o.calib_stats(X3), ref, rtol=1e-15, atol=0)


# ------------------------------------------------------------------ scale parameterisation

def pin_scale_grid(o):
    """s_j = (s_X,j)^alpha; alpha = 0 gives every scale 1 ("AWQ Math", "Searching the scale")."""
    m = np.array([4.0, 0.25, 1.0, 9.0, 0.0])
    s = o.scale_grid(m, [0.0, 0.5, 1.0])
    assert np.array_equal(s[0], np.ones(5))
    assert np.allclose(s[1], [2.0, 0.5, 1.0, 3.0, math.sqrt(1e-6)], rtol=1e-15)
    assert np.allclose(s[2], [4.0, 0.25, 1.0, 9.0, 1e-6], rtol=1e-15)


# ------------------------------------------------------------------ quantiser

def pin_quant_ladder_asym(o):
    """A group spanning exactly 16 levels is reproduced exactly: step = range/15, z = -lo/step."""
    for G in (64, 128):
        for z0 in (0, 3, 7, 15):
            for e in (4, 7, 10):
                g = _ladder_group(list(range(16)), z0, e, G)
                W = np.stack([g, g[::-1]]).astype(np.float16)
                qd = o.quantize(W, None, G, False)
                assert np.all(qd["step32"] == np.float32(2.0 ** (-e))), (z0, e, qd["step32"])
                assert np.all(qd["zero"] == z0), (z0, qd["zero"])
                want = np.rint(W.astype(np.float64) * 2.0 ** e) + z0
                assert np.array_equal(qd["codes"].astype(np.float64), want)


def pin_quant_ladder_sym(o):
    """Symmetric: step = max|w| / 2^(N-1) ("AWQ Math", "Weight-only quantization")."""
    for G in (64, 128):
        for e in (3, 6, 9):
            g = _ladder_group(list(range(-8, 8)), 0, e, G)
            W = g[None, :].astype(np.float16)
            qd = o.quantize(W, None, G, True)
            assert np.all(qd["step32"] == np.float32(2.0 ** (-e)))
            assert np.array_equal(qd["codes"][0].astype(np.int64),
                                  np.rint(g * 2.0 ** e).astype(np.int64) + 8)
            assert np.all(qd["zero"] == 8)


def pin_quant_ties_to_even(o):
    """Exact half-way values round to the even level (round-half-to-even reading)."""
    e, G = 5, 128
    vals = [j * 2.0 ** -e for j in range(16)] + [(j + 0.5) * 2.0 ** -e for j in range(15)]
    g = np.array([vals[i % len(vals)] for i in range(G)])
    qd = o.quantize(g[None, :].astype(np.float16), None, G, False)
    assert qd["step32"][0, 0] == np.float32(2.0 ** -e) and qd["zero"][0, 0] == 0
    for i in range(G):
        v = vals[i % len(vals)] * 2.0 ** e
        want = v if v == int(v) else (math.floor(v) if math.floor(v) % 2 == 0 else math.ceil(v))
        assert qd["codes"][0, i] == want, (v, qd["codes"][0, i])


def _bound_cases():
    rng = np.random.Generator(np.random.PCG64(11))
    W = (rng.standard_normal((6, 256)) * 0.02).astype(np.float16)
    W[1, :128] = np.abs(W[1, :128]) + np.float16(0.01)     # group entirely > 0
    W[2, 128:] = -np.abs(W[2, 128:]) - np.float16(0.01)    # group entirely < 0
    W[3, :128] = 0                                          # all-zero group
    s = np.exp(rng.uniform(-1.5, 2.5, 256)).astype(np.float32)
    return W, s


def pin_quant_error_bound(o):
    """|w' - (q - z) step| <= step / 2 for every unclamped weight ("Weight-only quantization")."""
    W, s = _bound_cases()
    for sym in (False, True):
        for G in (64, 128):
            for ss in (None, s):
                qd = o.quantize(W, ss, G, sym)
                wp = qd["scaled"]
                g_of_k = np.arange(W.shape[1]) // G
                step = qd["step32"].astype(np.float64)[:, g_of_k]
                zero = qd["zero"].astype(np.float64)[:, g_of_k]
                rec = (qd["codes"] - zero) * step
                err = np.abs(wp - rec)
                ok = ~qd["clamped"]
                assert np.all(err[ok] <= step[ok] / 2 * (1 + 2.0 ** -20)), (sym, G)
                assert qd["codes"].max() <= 15 and qd["zero"].max() <= 15
                if sym:
                    # only the top of the range (w'/step > 7.5) is ever clamped
                    assert np.all(wp[qd["clamped"]] > 7.4 * step[qd["clamped"]])
                else:
                    # with the range widened to hold 0, a clamp is at most one step away
                    assert np.all(err <= step * (1 + 2.0 ** -20))
                # an exact zero weight reconstructs exactly (asymmetric: the level q = z)
                zmask = wp == 0.0
                assert np.all(rec[zmask] == 0.0)
                # the all-zero group (row 3, first 128 channels) stores step 1 and codes = z
                gz = 0 if G == 128 else slice(0, 2)
                assert np.all(qd["step32"][3, gz] == 1.0) and np.all(qd["step16"][3, gz] == 1.0)
                assert np.all(qd["codes"][3, :128] == qd["zero"][3, 0])


def pin_quant_nearest_level(o):
    """Brute force: the chosen code is a nearest of the 16 representable levels."""
    W, s = _bound_cases()
    for sym in (False, True):
        qd = o.quantize(W, s, 128, sym)
        wp = qd["scaled"]
        g_of_k = np.arange(W.shape[1]) // 128
        step = qd["step32"].astype(np.float64)[:, g_of_k]
        zero = qd["zero"].astype(np.float64)[:, g_of_k]
        levels = (np.arange(16)[None, None, :] - zero[:, :, None]) * step[:, :, None]
        dist = np.abs(wp[:, :, None] - levels)
        best = dist.min(axis=2)
        chosen = np.take_along_axis(dist, qd["codes"][:, :, None].astype(np.int64), 2)[:, :, 0]
        assert np.all(chosen <= best + step * 2.0 ** -22), sym


def pin_quant_bit_widths(o):
    """N = 3 and N = 2 ("Weight-only quantization": D = max|w| / 2^(N-1) for N bits): exact
    ladders of 2^N levels give their own indices as codes; the symmetric step is max|w| / 4 and
    max|w| / 2, the top level clamps to 2^(N-1) - 1; every unclamped weight is within D/2; the
    chosen code is a nearest of the 2^N representable levels; N = 4 is the default."""
    G = 64
    for bits in (3, 2):
        n = 2 ** bits
        d = 2.0 ** -5
        for shift in (0, n // 2 - 1):                  # zero point 0 and mid-range
            g = np.array([((i % n) - shift) * d for i in range(G)])
            qd = o.quantize(g[None, :].astype(np.float16), None, G, False, bits)
            assert qd["step32"][0, 0] == np.float32(d) and qd["zero"][0, 0] == shift
            assert np.array_equal(qd["codes"][0], np.arange(G) % n)
        h = n // 2
        g = np.array([((i % (n + 1)) - h) * d for i in range(G)])   # -h .. +h steps
        qd = o.quantize(g[None, :].astype(np.float16), None, G, True, bits)
        assert qd["step32"][0, 0] == np.float32(h * d / h) and qd["zero"][0, 0] == 8
        q = np.minimum((np.arange(G) % (n + 1)) - h, h - 1)
        assert np.array_equal(qd["codes"][0].astype(int), q + 8)
        assert np.array_equal(qd["clamped"][0], (np.arange(G) % (n + 1)) == n)
        W, s = _bound_cases()
        for sym in (False, True):
            qd = o.quantize(W, s, 128, sym, bits)
            wp = qd["scaled"]
            g_of_k = np.arange(W.shape[1]) // 128
            step = qd["step32"].astype(np.float64)[:, g_of_k]
            zero = qd["zero"].astype(np.float64)[:, g_of_k]
            c = qd["codes"].astype(np.int64)
            lo_c, hi_c = (8 - h, 7 + h) if sym else (0, n - 1)
            assert c.min() >= lo_c and c.max() <= hi_c
            ok = ~qd["clamped"]
            err = np.abs(wp - (c - zero) * step)
            assert np.all(err[ok] <= step[ok] / 2 * (1 + 2.0 ** -20)), (bits, sym)
            levels = (np.arange(lo_c, hi_c + 1)[None, None, :] - zero[:, :, None]) * step[:, :, None]
            dist = np.abs(wp[:, :, None] - levels)
            chosen = np.take_along_axis(dist, (c - lo_c)[:, :, None], 2)[:, :, 0]
            assert np.all(chosen <= dist.min(axis=2) + step * 2.0 ** -22), (bits, sym)
    W, s = _bound_cases()
    for sym in (False, True):
        a, b = o.quantize(W, s, 64, sym), o.quantize(W, s, 64, sym, 4)
        assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["step32"], b["step32"])


def pin_quant_equivariance(o):
    """A power-of-two scale of the whole weight scales the step and leaves codes unchanged."""
    W, _ = _bound_cases()
    W = W[[0, 1, 2, 4, 5]]                      # no all-zero group (its step is fixed at 1)
    base = o.quantize(W, None, 128, False)
    for k in (-3, -1, 2, 5):
        s = np.full(W.shape[1], 2.0 ** k, np.float32)
        qd = o.quantize(W, s, 128, False)
        assert np.array_equal(qd["codes"], base["codes"]) and np.array_equal(qd["zero"], base["zero"])
        assert np.array_equal(qd["step32"], (base["step32"] * np.float32(2.0 ** k)))


def pin_pack_order(o):
    """Nibble i of word w holds channel 8w + i (literal words)."""
    codes = (np.arange(32) % 16).astype(np.uint8)[None, :]
    qw = o.pack_nibbles(codes)
    assert qw.dtype == np.uint32
    assert list(qw[0]) == [0x76543210, 0xFEDCBA98, 0x76543210, 0xFEDCBA98]
    rng = np.random.Generator(np.random.PCG64(3))
    c = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    assert np.array_equal(o.unpack_nibbles(o.pack_nibbles(c)), c)


def pin_dequant_closed_form(o):
    """w_hat = (q - z) * step / s, with per-group steps/zeros in [K/G, N] layout."""
    N, K, G = 3, 256, 128
    codes = np.zeros((N, K), np.uint8)
    codes[:, :G] = 9
    codes[:, G:] = 2
    scales = np.array([[0.5, 0.25, 2.0], [1.0, 4.0, 0.125]], np.float16)   # [K/G, N]
    zeros = np.array([[8, 7, 9], [0, 3, 2]], np.uint8)
    s = np.linspace(0.5, 2.0, K).astype(np.float32)
    w = o.dequantize(o.pack_nibbles(codes), scales, zeros, G, s=s)
    for n in range(N):
        for k in (0, 5, 127, 128, 200, 255):
            g = k // G
            want = (int(codes[n, k]) - int(zeros[g, n])) * float(scales[g, n]) / float(s[k])
            assert w[n, k] == want, (n, k, w[n, k], want)
    w2 = o.dequantize(o.pack_nibbles(codes), scales, zeros, G, inv_s=1.0 / s)
    assert np.allclose(w2, w, rtol=1e-6)


# ------------------------------------------------------------------ transform & error model

def pin_transform_exact(o):
    """y = W' x' with W' = W diag(s), x' = diag(s)^-1 x, exactly ("The equivalent transform")."""
    rng = np.random.Generator(np.random.PCG64(5))
    W = (rng.standard_normal((16, 64)) * 0.02).astype(np.float16)
    X = rng.standard_normal((8, 64)).astype(np.float16)
    s = (2.0 ** rng.integers(-4, 5, 64)).astype(np.float32)
    Wp = o.scaled_weight(W, s)
    Xp = X.astype(np.float64) / s.astype(np.float64)[None, :]
    assert np.array_equal(o.layer_output(Xp, Wp), o.layer_output(X, W))
    s2 = np.exp(rng.uniform(-1, 1, 64))
    Wp2 = W.astype(np.float64) * s2[None, :]
    y2 = o.layer_output(X.astype(np.float64) / s2[None, :], Wp2)
    y = o.layer_output(X, W)
    assert np.max(np.abs(y2 - y)) <= 1e-12 * np.max(np.abs(y))


def pin_worked_example(o):
    """"AWQ Math", "A worked numeric example": group max 1.0, N=4 -> step 0.125; the salient
    channel's expected output error 0.3125 -> 0.15625 at s=2; a large s inflates the step."""
    fx = _golden("worked_example.json")
    G = 128
    rng = np.random.Generator(np.random.PCG64(fx["seed"]))
    g = np.zeros(G)
    g[0] = fx["group_max"]
    g[1:] = rng.uniform(-0.9, 0.9, G - 1)
    g[5] = fx["salient_w"]
    qd = o.quantize(g[None, :].astype(np.float16), None, G, True)
    assert float(qd["step32"][0, 0]) == fx["delta"]
    # scaling the salient channel by 2 keeps the group max, so the step stays 0.125
    s = np.ones(G, np.float32)
    s[5] = fx["s"]
    qd2 = o.quantize(g[None, :].astype(np.float16), s, G, True)
    assert float(qd2["step32"][0, 0]) == fx["delta_after_scaling"]
    # pushing s so far that w*s exceeds the group max raises the step for the whole group
    s[5] = fx["large_s"]
    qd3 = o.quantize(g[None, :].astype(np.float16), s, G, True)
    big = float(np.float32(float(np.float16(fx["salient_w"])) * fx["large_s"])) / 8
    assert float(qd3["step32"][0, 0]) == big > fx["delta"]
    # expected output error of the salient channel, averaged over its rounding fraction
    n = fx["mc_samples"]
    # salient weights drawn over a whole number of steps, below 7.5 steps after scaling by s
    # (no clamp), so the rounding fraction is uniform and its mean is exactly 0.25
    w = rng.uniform(0.0, 3 * fx["delta"], n)
    Wm = np.zeros((n, G))
    Wm[:, 0] = fx["group_max"]
    Wm[:, 5] = w
    xabs = fx["x_abs"]
    Wm16 = Wm.astype(np.float16)
    for scale, want in ((1.0, fx["err_before"]), (fx["s"], fx["err_after"])):
        ss = np.ones(G, np.float32)
        ss[5] = scale
        qp = o.quantize_pack(Wm16, ss, G, True)
        w_hat = o.dequantize(qp["qweight"], qp["scales"], qp["zeros"], G, s=ss)
        err = np.abs(w_hat[:, 5] - Wm16[:, 5].astype(np.float64)) * xabs
        sd = err.std() / math.sqrt(n)
        assert abs(err.mean() - want) < 5 * sd + 1e-3 * want, (scale, err.mean(), want)


def pin_round_error_mean(o):
    """RoundErr in [0, 0.5] with E[RoundErr] ~ 0.25 ("Why scaling shrinks the error")."""
    fx = _golden("round_error.json")
    rng = np.random.Generator(np.random.PCG64(fx["seed"]))
    n, G = fx["groups"], 128
    W = rng.uniform(-1, 1, (n, G)).astype(np.float16)
    qd = o.quantize(W, None, G, True)
    frac = np.abs(qd["scaled"] / qd["step32"].astype(np.float64) - (qd["codes"].astype(np.float64) - 8))
    frac = frac[~qd["clamped"]]
    assert frac.max() <= fx["round_err_max"] * (1 + 2.0 ** -20)
    sd = frac.std() / math.sqrt(frac.size)
    assert abs(frac.mean() - fx["round_err_mean"]) < 5 * sd, frac.mean()


# ------------------------------------------------------------------ scoring & search

def pin_score_closed_form(o):
    """E = mean over outputs of (W x - w_hat x)^2: zero for exact codes, closed form for one
    perturbed weight, and equal to a brute-force triple loop."""
    G = 64
    g = _ladder_group(list(range(16)), 4, 6, G)
    W = np.stack([g, np.roll(g, 3)]).astype(np.float16)       # exactly representable
    rng = np.random.Generator(np.random.PCG64(9))
    X = rng.standard_normal((5, G)).astype(np.float16)
    qp = o.quantize_pack(W, None, G, False)
    assert o.error_of_codes(X, W, qp["qweight"], qp["scales"], qp["zeros"], np.ones(G, np.float32), G) == 0.0
    # one weight perturbed by d: E = d^2 sum_t x_tk^2 / (T N)
    W_hat = W.astype(np.float64).copy()
    d, k = 0.0625, 17
    W_hat[1, k] += d
    want = d * d * float(np.sum(X[:, k].astype(np.float64) ** 2)) / (X.shape[0] * W.shape[0])
    assert abs(o.output_mse(X, W, W_hat) - want) <= 1e-15 * want + 1e-300
    # brute-force triple loop on a tiny random layer
    W2 = (rng.standard_normal((3, G)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, G)).astype(np.float32)
    qp2 = o.quantize_pack(W2, s, G, False)
    w_hat = o.dequantize(qp2["qweight"], qp2["scales"], qp2["zeros"], G, s=s)
    tot = 0.0
    for t in range(X.shape[0]):
        for n in range(W2.shape[0]):
            acc = 0.0
            for kk in range(G):
                acc += float(X[t, kk]) * (float(W2[n, kk]) - float(w_hat[n, kk]))
            tot += acc * acc
    brute = tot / (X.shape[0] * W2.shape[0])
    got = o.error_of_codes(X, W2, qp2["qweight"], qp2["scales"], qp2["zeros"], s, G)
    assert abs(got - brute) <= 1e-9 * brute


def pin_search(o):
    """alpha = 0 is plain RTN; the winner is never worse than RTN; exact ties go to the smallest
    alpha; with outlier channels the search moves away from alpha = 0."""
    rng = np.random.Generator(np.random.PCG64(21))
    N, K, T, G = 8, 256, 32, 128
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    X = rng.standard_normal((T, K)).astype(np.float32)
    X[:, [10, 77, 200]] *= 20
    X = X.astype(np.float16)
    alphas = (np.arange(20) / 20).astype(np.float32)
    r = o.search_scale(W, X, alphas, G)
    rtn = o.quantize_pack(W, None, G, False)
    q0 = o.quantize_pack(W, r["s_grid"][0], G, False)
    assert np.array_equal(r["s_grid"][0], np.ones(K, np.float32))
    assert np.array_equal(q0["qweight"], rtn["qweight"]) and np.array_equal(q0["scales"], rtn["scales"])
    e_rtn = o.error_of_codes(X, W, rtn["qweight"], rtn["scales"], rtn["zeros"], np.ones(K, np.float32), G)
    assert r["err"][0] == e_rtn
    assert r["err"][r["best"]] <= r["err"][0]
    assert r["best"] == int(np.flatnonzero(r["err"] == r["err"].min())[0])
    assert r["best"] > 0, r["err"]
    # every |x| equal to 1 makes every scale 1, every alpha ties, and alpha_0 must win
    Xt = np.where(rng.random((T, K)) < 0.5, -1.0, 1.0).astype(np.float16)
    rt = o.search_scale(W, Xt, alphas, G)
    assert np.all(rt["err"] == rt["err"][0]) and rt["best"] == 0


# ------------------------------------------------------------------ W4A16 matmul

def pin_residual(o):
    """D = W - Q(W diag(s)) diag(s)^-1, the weight error one candidate is scored by ("Searching
    the scale"): on a group with lo = -7/16 and hi = 1/2 (step 1/16, zero point 7) the half-way
    weights (0.5, 1.5, 2.5, -0.5, -1.5) / 16 round to even and leave +-1/32 with the matching
    sign, while the on-grid weights leave 0; symmetric, 1/2 clamps to 7 steps and leaves 1/16.
    Scaling by powers of two commutes with it; |D| <= |W| everywhere (so 2^p D fits fp16)."""
    G = 128
    W = np.zeros((1, G), np.float16)
    W[0, :7] = np.array([-7.0, 8.0, 0.5, 1.5, 2.5, -0.5, -1.5]) / 16
    W[0, 7:23] = (np.arange(16) - 7) / 16.0
    one = np.ones(G, np.float32)
    D = o.residual(W, one, G, False)
    assert np.array_equal(D[0, :7] * 32, [0, 0, 1, -1, 1, -1, 1])
    assert np.all(D[0, 7:] == 0)
    Ds = o.residual(W, one, G, True)
    assert np.array_equal(Ds[0, :7] * 32, [0, 2, 1, -1, 1, -1, 1])
    two = np.where(np.arange(G) % 3 == 0, 4.0, 0.5).astype(np.float32)
    # per-channel powers of two move each weight's quotient, not D's definition: w_hat * s is
    # the same level grid for W' = W s, so D s is the residual of W' with s = 1
    Wp = (W.astype(np.float64) * two).astype(np.float16)
    assert np.array_equal(o.residual(W, two, G, False) * two, o.residual(Wp, one, G, False))
    Wb, sb = _bound_cases()
    for sym in (False, True):
        for gs in (64, 128):
            for bits in (4, 3, 2):        # at every code width (the GPU's 2^p scale relies on it)
                Db = o.residual(Wb, sb, gs, sym, bits)
                assert np.all(np.abs(Db) <= np.abs(Wb.astype(np.float64)) * (1 + 2.0 ** -20))
    assert o.residual_exponent(W) == 14          # max|W| = 1/2 < 2^0
    assert o.residual_exponent(np.array([[1.0, -0.25]], np.float16)) == 13
    assert o.residual_exponent(np.array([[-65504.0]], np.float16)) == -2
    assert o.residual_exponent(np.zeros((2, 8), np.float16)) == 0


def pin_gemm_closed_form(o):
    """Dequant-fused matmul: codes z+1 with step 1 give w_hat = 1, so Y is the row sums of X
    (times inv_s when given) ("Benefits ...": unpack, group scale, zero point, inverse scale)."""
    M, N, K, G = 3, 5, 256, 128
    rng = np.random.Generator(np.random.PCG64(13))
    X = rng.standard_normal((M, K)).astype(np.float16)
    zeros = rng.integers(0, 15, (K // G, N)).astype(np.uint8)
    codes = np.zeros((N, K), np.uint8)
    for n in range(N):
        for g in range(K // G):
            codes[n, g * G:(g + 1) * G] = zeros[g, n] + 1
    scales = np.ones((K // G, N), np.float16)
    qw = o.pack_nibbles(codes)
    Y = o.w4a16_gemm(X, qw, scales, zeros, G)
    assert Y.shape == (M, N)
    rows = X.astype(np.float64).sum(axis=1)
    assert np.allclose(Y, rows[:, None], rtol=1e-15, atol=1e-12)
    inv_s = rng.uniform(0.5, 2, K).astype(np.float32)
    Y2 = o.w4a16_gemm(X, qw, scales, zeros, G, inv_s=inv_s)
    want = X.astype(np.float64) @ inv_s.astype(np.float64)
    assert np.allclose(Y2, want[:, None], rtol=1e-14, atol=1e-12)
    # distinct per-output steps: column n is (n + 1) times the row sum
    scales_n = np.tile(np.arange(1, N + 1, dtype=np.float16), (K // G, 1))
    Y3 = o.w4a16_gemm(X, qw, scales_n, zeros, G)
    assert np.allclose(Y3, rows[:, None] * np.arange(1, N + 1)[None, :], rtol=1e-14, atol=1e-12)
    r, c = np.array([0, 2, 1]), np.array([4, 0, 3])
    assert np.allclose(o.w4a16_gemm_entries(X, qw, scales, zeros, r, c, G, inv_s), Y2[r, c], rtol=1e-14)


def pin_memory_footprint(o):
    """The packed format is ~4x smaller than fp16 ("Benefits ...": 7B 14 -> 4 GB, 13B 26 -> 7
    GB, 70B 140 -> 40 GB)."""
    fx = _golden("memory_footprint.json")
    for row in fx["models"]:
        p = row["params"]
        fp16_gb = 2 * p / 1e9
        # a square-ish stand-in layer with the model's parameter count
        q_gb = o.packed_bytes(p // 4096, 4096, 128) / 1e9
        assert abs(fp16_gb - row["fp16_gb"]) <= 0.1 * row["fp16_gb"]
        assert abs(q_gb - row["int4_gb"]) <= fx["tolerance_rel"] * row["int4_gb"], (row, q_gb)
        assert 3.7 < fp16_gb / q_gb < 4.0


# ------------------------------------------------------------------ per-group clipping

def pin_channel_energy(o):
    """h_k = sum_t x_tk^2: X[t, k] = (t + 1) (k + 1) gives (k + 1)^2 T (T + 1)(2T + 1) / 6."""
    T, K = 9, 6
    X = (np.arange(1, T + 1)[:, None] * np.arange(1, K + 1)[None, :]).astype(np.float64)
    want = (np.arange(1, K + 1) ** 2) * T * (T + 1) * (2 * T + 1) / 6
    assert np.array_equal(o.channel_energy(X), want)


def pin_clip(o):
    """Clipping (a reading; the pages print no clipping step): a ratio of one is the plain
    quantiser; a ratio c bounds the group's magnitudes by b = fl32(c max|w'|) (asymmetric range
    min(hi, b), max(lo, -b); symmetric max|w'| -> b), the weights beyond take the end codes and
    the rest stay within half the (smaller) step; the search clips deep (to the grid's last
    ratio) a group whose one large weight sits on a channel with little calibration energy and
    at most lightly (c >= 0.9) when that channel carries the energy, and with no energy at all
    every ratio ties and the first (1.0) wins."""
    rng = np.random.Generator(np.random.PCG64(33))
    N, K, G = 3, 256, 128
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    grid = o.clip_ratio_grid(10)
    assert np.array_equal(grid, np.float32([1, .95, .9, .85, .8, .75, .7, .65, .6, .55]))
    ones = np.ones((N, K // G), np.float32)
    for sym in (False, True):
        a, b = o.quantize_pack(W, None, G, sym), o.quantize_pack(W, None, G, sym, clip=ones)
        for key in ("qweight", "scales", "zeros"):
            assert np.array_equal(a[key], b[key])
    # range ends and the half-step bound under a clip of 0.5 (asymmetric)
    c = np.full((N, K // G), 0.5, np.float32)
    q = o.quantize(W, None, G, False, clip=c)
    grp = q["scaled"].reshape(N, K // G, G)
    b = o.fl32(np.abs(grp).max(axis=2) * 0.5).astype(np.float64)
    hi = np.minimum(np.maximum(grp.max(axis=2), 0), b)
    lo = np.maximum(np.minimum(grp.min(axis=2), 0), -b)
    assert np.all((hi == b) | (lo == -b))         # the larger end is cut to the bound
    step = q["step32"].astype(np.float64)
    assert np.array_equal(step, o.fl32(o.fl32(hi - lo) / 15).astype(np.float64))
    codes = q["codes"].reshape(N, K // G, G).astype(np.float64)
    w_hat = (codes - q["zero"][:, :, None]) * step[:, :, None]
    clamped = q["clamped"].reshape(N, K // G, G)
    free = ~clamped
    assert np.all(np.abs(grp - w_hat)[free] <= step[:, :, None].repeat(G, 2)[free] / 2 * (1 + 2.0 ** -20))
    above, below = grp > hi[:, :, None] + step[:, :, None], grp < lo[:, :, None] - step[:, :, None]
    assert above.any() and below.any()
    assert np.all(codes[above] == 15) and np.all(clamped[above])
    assert np.all(codes[below] == 0) and np.all(clamped[below])
    # the energy decides: one large weight on channel 5 of group 0 of row 0
    W2 = (rng.uniform(-0.1, 0.1, (1, G))).astype(np.float16)
    W2[0, 5] = 1.0
    X = rng.standard_normal((64, G)).astype(np.float16)
    for h5, deep in ((1e-4, True), (1e4, False)):
        h = np.ones(G)
        h[5] = h5
        r = o.clip_search(W2, X, None, grid, G, h=h)
        c = grid[r["best"][0, 0]]
        assert (c == grid[-1]) if deep else (c >= 0.9), (h5, r["err"][:, 0, 0])
        assert r["err"][r["best"][0, 0], 0, 0] <= r["err"][0, 0, 0]
        assert r["clip"].shape == (1, 1) and r["clip"][0, 0] == grid[r["best"][0, 0]]
    rz = o.clip_search(W, X[:, :1].repeat(K, 1), None, grid, G, h=np.zeros(K))
    assert np.all(rz["best"] == 0) and np.all(rz["clip"] == 1.0)
    # e(c) is the energy-weighted squared weight error of the group (a brute-force sum)
    h = rng.uniform(0.5, 2.0, K)
    r = o.clip_search(W, None, None, grid[:3], G, h=h)
    for j, cj in enumerate(grid[:3]):
        qd = o.quantize_pack(W, None, G, False, clip=np.full((N, K // G), cj, np.float32))
        wh = o.dequantize(qd["qweight"], qd["scales"], qd["zeros"], G)
        for n in range(N):
            for g in range(K // G):
                e = 0.0
                for k in range(g * G, (g + 1) * G):
                    d = float(W[n, k]) - wh[n, k]
                    e += h[k] * d * d
                assert abs(e - r["err"][j, n, g]) <= 1e-12 * max(e, 1e-30)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
