"""Plain, slow CPU oracle for the AWQ per-linear-layer step (test infrastructure only).

This module is the definition the CUDA path is checked against. It is test infrastructure:
only the test suite, the package entry point's smoke check and the benchmark's CPU-baseline
leg may import it. The product path never calls it and shares no code with it.

Everything is float64 numpy unless a step decides an integer (a quantisation code, a zero
point, the chosen alpha). Those decisions are taken in the kernel's precision, fp32, written
here as an fp64 operation followed by a round-to-nearest-even to fp32. For one +, -, * or / of
fp32 operands that equals the IEEE fp32 result, since fp64 carries more than 2*24+2 bits.

Sources (titles and sections of the pages this follows):

* "AWQ Math", section "Saliency is an activation property, not a weight property": the
  per-input-channel statistic, the average |x_j| over the calibration set.
* "AWQ Math", section "The equivalent transform": W' = W diag(s), x' = diag(s)^-1 x, y = W' x'.
* "AWQ Math", section "Searching the scale": s_j = (s_X,j)^alpha with alpha in [0, 1];
  alpha* = argmin ||W x - Q(W diag(s)) diag(s)^-1 x|| measured as the mean-squared error of the
  layer output over the calibration set; alpha = 0 is plain quantisation.
* "AWQ Math", section "Weight-only quantization and where it breaks": Q(w) = D round(w / D),
  D = max|w| / 2^(N-1), rounding error at most D/2 (the symmetric variant).
* "AWQ Math", section "Shapes, granularity, and complexity", and "AWQ > Benefits and Practical
  Considerations": per-group (128 input channels) step and zero point; storage is the 4-bit
  integers plus per-group scales and zero points.
* "AWQ > Benefits and Practical Considerations": the inference kernel unpacks 4-bit integers,
  applies the group scale and zero point and, optionally, the per-channel inverse scale.

Readings where the pages are silent (each is listed in the design notes):

* Asymmetric quantiser (the pages name a step and a zero point but print no formula): the
  group range is widened to include 0, D = (hi - lo) / (2^4 - 1), z = clamp(rint(-lo / D)),
  q = clamp(rint(w / D) + z, 0, 15); D = 1 for an all-zero group.
* Bit width N (the pages' D = max|w| / 2^(N-1) is written for any N; 4 is the default, 3 and 2
  are the narrower variants): asymmetric codes 0..2^N - 1, symmetric q in [-2^(N-1), 2^(N-1) - 1];
  codes of every width are stored in 4-bit nibbles (no denser packing), so the matmul reads them
  unchanged.
* Symmetric quantiser: the printed D = max|w| / 8 with codes clamped to [-8, 7] (4 bits hold
  16 levels); stored as q + 8 with an implicit zero point of 8.
* rint is round-half-to-even; the stored step is fp16 (round to nearest even); codes are
  decided from the fp32 step, the dequantised weight uses the stored fp16 step.
* alpha grid alpha_i = i / n for i < n (0 included, 1 excluded); s_j = max(m_j, 1e-6)^alpha;
  no normalisation of s; ties in the argmin go to the smallest alpha.
* The error is the mean over all T x C_out outputs of the squared difference between the
  exact output of the fp16 inputs and the output of the dequantised weights.
* Per-group clipping (the pages print no clipping step; "AWQ Math", "CPU-SLM implications and
  common pitfalls" only warns to watch the group size): each group's magnitudes are bounded by
  c max|w'| for a ratio c from a grid (1, 0.95, ..., 0.55), and each group takes the first ratio
  minimising its own output error on the calibration set with the cross-channel terms dropped,
  sum_k h_k (W - w_hat)^2 with h_k = sum_t x_tk^2.

Packed format: nibble i (bits 4i..4i+3) of ``qweight[n, w]`` is the code of input channel
``k = 8 w + i``; ``scales[g, n]`` (fp16) and ``zeros[g, n]`` (uint8) are per group g of
``group_size`` input channels.
"""

from __future__ import annotations

import numpy as np

EPS = 1e-6        # floor on the statistic before the power (dead channels)
BITS = (2, 3, 4)  # code widths N; codes of every width are stored in 4-bit nibbles
SYM_ZERO = 8      # implicit zero point of the stored symmetric codes (q + 8), for every width


def fl32(a) -> np.ndarray:
    """Round an fp64 value (array) to the nearest fp32, ties to even."""
    return np.asarray(a, dtype=np.float64).astype(np.float32)


# ----------------------------------------------------------------------------------------
# Calibration statistic ("AWQ Math", "Saliency is an activation property ...")
# ----------------------------------------------------------------------------------------

def calib_stats(X: np.ndarray) -> np.ndarray:
    """m_j = (1/T) sum_t |X[t, j]|, the average activation magnitude of input channel j."""
    X64 = np.asarray(X, dtype=np.float64)
    T = X64.shape[0]
    total = np.zeros(X64.shape[1], dtype=np.float64)
    for t in range(T):
        total += np.abs(X64[t])
    return total / T


# ----------------------------------------------------------------------------------------
# Scale parameterisation ("AWQ Math", "Searching the scale")
# ----------------------------------------------------------------------------------------

def scale_grid(m: np.ndarray, alphas, eps: float = EPS) -> np.ndarray:
    """s[i, j] = max(m_j, eps) ** alpha_i, in fp64. Row i is the scale vector of alpha_i."""
    base = np.maximum(np.asarray(m, dtype=np.float64), eps)
    a = np.asarray(alphas, dtype=np.float64)
    return base[None, :] ** a[:, None]


# ----------------------------------------------------------------------------------------
# Group-wise INT4 quantiser of W diag(s) ("Weight-only quantization ...", "Shapes ...")
# ----------------------------------------------------------------------------------------

def scaled_weight(W: np.ndarray, s) -> np.ndarray:
    """w'[n, k] = fl32(W[n, k] * s_k): the transform W' = W diag(s) in the kernel's fp32."""
    W64 = np.asarray(W, dtype=np.float64)
    if s is None:
        return fl32(W64)
    s32 = np.asarray(s, dtype=np.float32).astype(np.float64)
    return fl32(W64 * s32[None, :])


def quantize(W: np.ndarray, s=None, group_size: int = 128, symmetric: bool = False,
             bits: int = 4, clip=None) -> dict:
    """Quantise W diag(s) group-wise to ``bits``-wide codes (N in "Weight-only quantization").

    ``clip`` (optional, [N, K/G] fp32 ratios in (0, 1]) bounds each group's magnitudes before
    the step is taken: with b = fl32(c max|w'|), the asymmetric ends (already widened to hold 0)
    become min(hi, b) and max(lo, -b), the symmetric max|w'| becomes b; weights outside the
    bounded range take the end codes through the usual clamp. ``clip`` of all ones is the plain
    quantiser.

    Returns ``codes`` [N, K] (stored nibble values), ``step32`` [N, K/G] (fp32 step the codes
    were decided with), ``step16`` [N, K/G] (stored fp16 step), ``zero`` [N, K/G] (uint8; 8 in
    symmetric mode) and ``clamped`` [N, K] (True where a clamp changed the code).
    """
    if bits not in BITS:
        raise ValueError("bits must be 2, 3 or 4")
    qmax = 2 ** bits - 1              # asymmetric levels 0 .. qmax
    half = 2 ** (bits - 1)            # symmetric: step = max|w'| / 2^(N-1), q in [-half, half-1]
    wp = scaled_weight(W, s).astype(np.float64)          # exact fp32 values held in fp64
    N, K = wp.shape
    if K % group_size:
        raise ValueError("K must be a multiple of the group size")
    grp = wp.reshape(N, K // group_size, group_size)
    c = None if clip is None else np.asarray(clip, dtype=np.float32).astype(np.float64)
    bound = None if c is None else fl32(np.max(np.abs(grp), axis=2) * c).astype(np.float64)
    if symmetric:
        amax = np.max(np.abs(grp), axis=2)
        if c is not None:
            amax = bound
        step = fl32(amax / half).astype(np.float64)
        step[step == 0.0] = 1.0
        r = np.rint(fl32(grp / step[:, :, None]).astype(np.float64))
        q = np.clip(r, -half, half - 1)
        zero = np.full((N, K // group_size), SYM_ZERO, dtype=np.uint8)
        codes = (q + SYM_ZERO).astype(np.uint8)
        clamped = q != r
    else:
        hi = np.maximum(np.max(grp, axis=2), 0.0)
        lo = np.minimum(np.min(grp, axis=2), 0.0)
        if c is not None:
            hi = np.minimum(hi, bound)
            lo = np.maximum(lo, -bound)
        rng_ = fl32(hi - lo).astype(np.float64)
        step = fl32(rng_ / qmax).astype(np.float64)
        step[step == 0.0] = 1.0
        z = np.clip(np.rint(fl32(-lo / step).astype(np.float64)), 0, qmax)
        r = np.rint(fl32(grp / step[:, :, None]).astype(np.float64)) + z[:, :, None]
        q = np.clip(r, 0, qmax)
        zero = z.astype(np.uint8)
        codes = q.astype(np.uint8)
        clamped = q != r
    step32 = step.astype(np.float32)
    return {
        "codes": codes.reshape(N, K),
        "step32": step32,
        "step16": step32.astype(np.float16),
        "zero": zero,
        "clamped": clamped.reshape(N, K),
        "scaled": wp,
    }


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[N, K] codes 0..15 -> [N, K/8] uint32; nibble i of word w holds channel 8w + i."""
    c = np.asarray(codes, dtype=np.uint64)
    N, K = c.shape
    c = c.reshape(N, K // 8, 8)
    out = np.zeros((N, K // 8), dtype=np.uint64)
    for i in range(8):
        out |= c[:, :, i] << np.uint64(4 * i)
    return out.astype(np.uint32)


def unpack_nibbles(qweight: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`: [N, K/8] uint32 -> [N, K] uint8."""
    qw = np.asarray(qweight, dtype=np.uint32)
    N, W = qw.shape
    out = np.zeros((N, W, 8), dtype=np.uint8)
    for i in range(8):
        out[:, :, i] = (qw >> np.uint32(4 * i)) & np.uint32(0xF)
    return out.reshape(N, W * 8)


def quantize_pack(W: np.ndarray, s=None, group_size: int = 128,
                  symmetric: bool = False, bits: int = 4, clip=None) -> dict:
    """The stored form: ``qweight`` [N, K/8] uint32, ``scales`` [K/G, N] fp16,
    ``zeros`` [K/G, N] uint8 (all 8 in symmetric mode), plus the :func:`quantize` details.
    ``clip`` as in :func:`quantize`, [N, K/G]."""
    qd = quantize(W, s, group_size, symmetric, bits, clip)
    qd["qweight"] = pack_nibbles(qd["codes"])
    qd["scales"] = np.ascontiguousarray(qd["step16"].T)
    qd["zeros"] = np.ascontiguousarray(qd["zero"].T)
    return qd


def dequantize(qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
               group_size: int = 128, inv_s=None, s=None) -> np.ndarray:
    """w_hat[n, k] = (q[n, k] - z[g, n]) * step16[g, n], then times inv_s_k or divided by s_k.

    This is Q(W diag(s)) diag(s)^-1 in fp64 from the stored fields.
    """
    codes = unpack_nibbles(qweight).astype(np.float64)
    N, K = codes.shape
    step = np.asarray(scales, dtype=np.float16).astype(np.float64).T      # [N, K/G]
    zero = np.asarray(zeros, dtype=np.float64).T                          # [N, K/G]
    g_of_k = np.arange(K) // group_size
    w_hat = (codes - zero[:, g_of_k]) * step[:, g_of_k]
    if s is not None:
        w_hat = w_hat / np.asarray(s, dtype=np.float32).astype(np.float64)[None, :]
    if inv_s is not None:
        w_hat = w_hat * np.asarray(inv_s, dtype=np.float32).astype(np.float64)[None, :]
    return w_hat


# ----------------------------------------------------------------------------------------
# Output error and the alpha search ("AWQ Math", "Searching the scale")
# ----------------------------------------------------------------------------------------

def layer_output(X: np.ndarray, W) -> np.ndarray:
    """y = W x for every calibration token: [T, C_out] = X [T, K] @ W^T, in fp64."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def output_mse(X: np.ndarray, W: np.ndarray, W_hat: np.ndarray) -> float:
    """Mean over all tokens and outputs of (W x - W_hat x)^2."""
    y = layer_output(X, W)
    y_hat = layer_output(X, W_hat)
    return float(np.mean((y - y_hat) ** 2))


def search_scale(W: np.ndarray, X: np.ndarray, alphas, group_size: int = 128,
                 symmetric: bool = False, m=None, s_grid=None, eps: float = EPS,
                 bits: int = 4) -> dict:
    """The alpha search of one linear layer.

    For each alpha_i: s = max(m, eps)^alpha_i (rounded to fp32, the kernel's precision), codes of
    W diag(s), w_hat = Q(W diag(s)) diag(s)^-1, error E_i = mean (W x - w_hat x)^2 over the
    calibration tokens. alpha* is the first minimiser. ``m`` and ``s_grid`` (fp32 [n_alpha, K])
    may be supplied to evaluate the quantiser on another implementation's statistic/scales.
    """
    if m is None:
        m = calib_stats(X)
    if s_grid is None:
        s_grid = fl32(scale_grid(m, alphas, eps))
    s_grid = np.asarray(s_grid, dtype=np.float32)
    y = layer_output(X, W)
    err = np.zeros(len(s_grid), dtype=np.float64)
    for i, s in enumerate(s_grid):
        qd = quantize_pack(W, s, group_size, symmetric, bits)
        w_hat = dequantize(qd["qweight"], qd["scales"], qd["zeros"], group_size, s=s)
        err[i] = float(np.mean((y - layer_output(X, w_hat)) ** 2))
    best = int(np.argmin(err))           # numpy returns the first minimiser
    return {"err": err, "best": best, "s": s_grid[best].copy(), "m": np.asarray(m),
            "s_grid": s_grid}


def error_of_codes(X: np.ndarray, W: np.ndarray, qweight, scales, zeros, s,
                   group_size: int = 128) -> float:
    """E for codes produced elsewhere (staged parity): mean (W x - Q diag(s)^-1 x)^2."""
    w_hat = dequantize(qweight, scales, zeros, group_size, s=s)
    return output_mse(X, W, w_hat)


def residual(W: np.ndarray, s, group_size: int = 128, symmetric: bool = False,
             bits: int = 4) -> np.ndarray:
    """D = W - Q(W diag(s)) diag(s)^-1 in fp64: the weight error of one candidate, whose product
    with the calibration inputs is that candidate's output error, since
    W x - Q(W diag(s)) diag(s)^-1 x = D x ("AWQ Math", "Searching the scale")."""
    qd = quantize_pack(W, s, group_size, symmetric, bits)
    w_hat = dequantize(qd["qweight"], qd["scales"], qd["zeros"], group_size, s=s)
    return np.asarray(W, dtype=np.float64) - w_hat


def residual_exponent(W: np.ndarray) -> int:
    """p with max|W| < 2^(14 - p) <= 2 max|W| (0 for an all-zero W): the power-of-two factor the
    GPU applies to D before rounding it to fp16, which keeps every |2^p D| below 2^14 because
    |D| <= |W| element by element."""
    mx = float(np.max(np.abs(np.asarray(W, dtype=np.float64)))) if np.size(W) else 0.0
    if mx == 0.0:
        return 0
    _, e = np.frexp(mx)            # mx = f 2^e, f in [0.5, 1)
    return 14 - int(e)


# ----------------------------------------------------------------------------------------
# Per-group clipping search (a reading: the pages print no clipping step; see the notes)
# ----------------------------------------------------------------------------------------

def clip_ratio_grid(n: int = 10) -> np.ndarray:
    """Clip ratios c_j = 1 - j/20 for j < n (1, 0.95, ..., 0.55 for n = 10) as fp32."""
    return (1.0 - np.arange(n, dtype=np.float64) / 20.0).astype(np.float32)


def channel_energy(X: np.ndarray) -> np.ndarray:
    """h_k = sum_t X[t, k]^2 in fp64: the calibration energy of input channel k, the weight a
    weight error on that channel carries in the layer's output error (the diagonal of X^T X)."""
    X64 = np.asarray(X, dtype=np.float64)
    h = np.zeros(X64.shape[1], dtype=np.float64)
    for t in range(X64.shape[0]):
        h += X64[t] * X64[t]
    return h


def clip_search(W: np.ndarray, X: np.ndarray, s, ratios, group_size: int = 128,
                symmetric: bool = False, bits: int = 4, h=None) -> dict:
    """Each group's clip ratio: for every ratio c of ``ratios`` the group is quantised with its
    range shrunk by c (:func:`quantize`), and its error e(c) = sum_k h_k (W[n, k] - w_hat[n, k])^2
    over the group's channels k is the group's output error on the calibration set with the
    cross-channel terms dropped (h = :func:`channel_energy`, w_hat = Q(W diag(s)) diag(s)^-1 as in
    the search). The first minimiser wins, so with ratios[0] = 1 a group is clipped only when
    that strictly lowers its error.

    Returns ``best`` [N, K/G] (index into ratios), ``clip`` [K/G, N] fp32 (the chosen ratios,
    stored like the steps) and ``err`` [n_ratio, N, K/G] (fp64)."""
    W64 = np.asarray(W, dtype=np.float64)
    N, K = W64.shape
    ng = K // group_size
    if h is None:
        h = channel_energy(X)
    h = np.asarray(h, dtype=np.float64)
    r = np.asarray(ratios, dtype=np.float32)
    err = np.zeros((len(r), N, ng), dtype=np.float64)
    for j, c in enumerate(r):
        clip = np.full((N, ng), c, dtype=np.float32)
        qd = quantize_pack(W, s, group_size, symmetric, bits, clip=clip)
        d = W64 - dequantize(qd["qweight"], qd["scales"], qd["zeros"], group_size, s=s)
        err[j] = (d * d * h[None, :]).reshape(N, ng, group_size).sum(axis=2)
    best = np.argmin(err, axis=0)                   # numpy returns the first minimiser
    return {"best": best, "clip": np.ascontiguousarray(r[best].T), "err": err}


# ----------------------------------------------------------------------------------------
# W4A16 dequant-fused matmul ("AWQ > Benefits and Practical Considerations")
# ----------------------------------------------------------------------------------------

def w4a16_gemm(X: np.ndarray, qweight, scales, zeros, group_size: int = 128,
               inv_s=None) -> np.ndarray:
    """Y [M, N] = X [M, K] @ (dequant(Q) diag(inv_s))^T in fp64 (inv_s None: folded away)."""
    w_hat = dequantize(qweight, scales, zeros, group_size, inv_s=inv_s)
    return np.asarray(X, dtype=np.float64) @ w_hat.T


def w4a16_gemm_entries(X: np.ndarray, qweight, scales, zeros, rows, cols,
                       group_size: int = 128, inv_s=None) -> np.ndarray:
    """Y[rows[i], cols[i]] one by one (sampled checks of a large product)."""
    X64 = np.asarray(X, dtype=np.float64)
    cols = np.asarray(cols)
    w_hat = dequantize(np.asarray(qweight)[cols], np.asarray(scales)[:, cols],
                       np.asarray(zeros)[:, cols], group_size, inv_s=inv_s)
    return np.einsum("ik,ik->i", X64[np.asarray(rows)], w_hat)


def packed_bytes(n: int, k: int, group_size: int = 128) -> int:
    """Stored bytes of one layer: 4-bit codes + fp16 step + uint8 zero per group."""
    return n * k // 2 + 3 * n * (k // group_size)
