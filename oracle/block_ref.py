"""Plain CPU oracle for folding 1/s into the previous operation and for an AWQ-quantised
Llama-style MLP block run end to end (test infrastructure only: the test suite may import it,
the product path never does).

Sources (titles and sections of the pages this follows):

* "AWQ Math", section "The equivalent transform": y = W x = (W diag(s)) (diag(s)^-1 x), so the
  1/s factor can move into whatever produces x.
* "AWQ > Benefits and Practical Considerations": the per-channel scale folds into the previous
  layer (a norm or a linear), and the quantised layer then runs on the folded input.
* "AWQ Math", section "Searching the scale": each linear's alpha is searched on its own
  calibration input, which for a layer inside a block is the output of the layers before it.

Readings (listed in the design notes):

* The block is RMSNorm -> gate and up (one search: the two linears share their input and s)
  -> silu(gate) * up -> down. The down projection's calibration input is the fp16 block's own
  silu(gate) * up on the calibration tokens (activations propagated through the unquantised
  block, as the search of each linear assumes the original model's input).
* 1/s of gate/up folds into the RMSNorm weight; 1/s of down folds into the rows of W_up
  (scaling up's output channel k scales h_k, since silu(gate) does not depend on up).
* The fold is one fp32 multiply of the fp16 value by the fp32 inverse scale, rounded to fp16.
* RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma; silu(g) = g / (1 + exp(-g)); both rounded
  to fp16 once at the end (fp64 here, fp32 on the GPU: tolerance-checked, not bit-exact).
"""

from __future__ import annotations

import numpy as np

from . import awq_ref as ref


def scale_rows(A16: np.ndarray, row_scale) -> np.ndarray:
    """A'[r, c] = fp16(fl32(A[r, c] * row_scale[r])): the fold of 1/s into the rows that
    produce input channel r ("AWQ Math", "The equivalent transform")."""
    A64 = np.asarray(A16, dtype=np.float16).astype(np.float64)
    r = np.asarray(row_scale, dtype=np.float32).astype(np.float64)
    shape = (-1,) + (1,) * (A64.ndim - 1)
    return ref.fl32(A64 * r.reshape(shape)).astype(np.float16)


def rmsnorm(X16: np.ndarray, gamma16: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """fp16(x / sqrt(mean_j x_j^2 + eps) * gamma), per token, in fp64."""
    X = np.asarray(X16, dtype=np.float16).astype(np.float64)
    g = np.asarray(gamma16, dtype=np.float16).astype(np.float64)
    r = 1.0 / np.sqrt(np.mean(X * X, axis=1, keepdims=True) + float(np.float32(eps)))
    return (X * r * g[None, :]).astype(np.float16)


def silu_mul(G16: np.ndarray, U16: np.ndarray) -> np.ndarray:
    """fp16(silu(g) * u), silu(g) = g / (1 + e^-g), in fp64."""
    G = np.asarray(G16, dtype=np.float16).astype(np.float64)
    U = np.asarray(U16, dtype=np.float16).astype(np.float64)
    return (G / (1.0 + np.exp(-G)) * U).astype(np.float16)


def linear16(X16: np.ndarray, W: np.ndarray) -> np.ndarray:
    """fp16 output of a linear layer: fp16(X @ W^T) with the product in fp64."""
    return (np.asarray(X16, dtype=np.float16).astype(np.float64)
            @ np.asarray(W, dtype=np.float64).T).astype(np.float16)


def mlp_fp16(X16, gamma16, Wg, Wu, Wd, eps: float = 1e-6) -> dict:
    """The unquantised block with fp16 activations between operations."""
    xn = rmsnorm(X16, gamma16, eps)
    g = linear16(xn, Wg)
    u = linear16(xn, Wu)
    h = silu_mul(g, u)
    return {"xn": xn, "g": g, "u": u, "h": h, "y": linear16(h, Wd)}


def quantize_mlp(X16, gamma16, Wg, Wu, Wd, alphas, group_size: int = 128,
                 eps: float = 1e-6, xn=None, h=None) -> dict:
    """AWQ on the block: alpha search for gate/up (stacked, shared input and s) on the normed
    calibration input, for down on the propagated silu(gate) * up; fold both inverse scales
    into the previous operations; quantise the three weights with their s. ``xn`` and ``h``
    may be supplied (another implementation's intermediates) for staged parity."""
    fp = mlp_fp16(X16, gamma16, Wg, Wu, Wd, eps)
    xn = fp["xn"] if xn is None else xn
    h = fp["h"] if h is None else h
    Wgu = np.concatenate([np.asarray(Wg), np.asarray(Wu)], axis=0)
    r1 = ref.search_scale(Wgu, xn, alphas, group_size)
    r2 = ref.search_scale(Wd, h, alphas, group_size)
    s1, s2 = r1["s"], r2["s"]
    inv1 = (np.float32(1) / s1).astype(np.float32)
    inv2 = (np.float32(1) / s2).astype(np.float32)
    gamma_f = scale_rows(gamma16, inv1)
    Wu_f = scale_rows(Wu, inv2)
    return {"r1": r1, "r2": r2, "s1": s1, "s2": s2, "gamma": gamma_f, "Wu": Wu_f,
            "gate": ref.quantize_pack(Wg, s1, group_size),
            "up": ref.quantize_pack(Wu_f, s1, group_size),
            "down": ref.quantize_pack(Wd, s2, group_size)}


def mlp_quantized(X16, q: dict, group_size: int = 128, eps: float = 1e-6, xn=None,
                  g=None, u=None, h=None) -> dict:
    """The quantised block on folded inputs (inv_s = NULL everywhere), fp16 between operations;
    intermediates may be supplied for staged comparison."""
    def lin(x, pk):
        w = ref.dequantize(pk["qweight"], pk["scales"], pk["zeros"], group_size)
        return (np.asarray(x, dtype=np.float16).astype(np.float64) @ w.T).astype(np.float16)
    xn = rmsnorm(X16, q["gamma"], eps) if xn is None else xn
    g = lin(xn, q["gate"]) if g is None else g
    u = lin(xn, q["up"]) if u is None else u
    h = silu_mul(g, u) if h is None else h
    return {"xn": xn, "g": g, "u": u, "h": h, "y": lin(h, q["down"])}
