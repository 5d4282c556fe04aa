"""The fp32 error bound of the GPU clipping criterion, shared by the GPU parity test and its
CPU check (test code: the oracle supplies the exact quantities)."""

import numpy as np

from oracle import awq_ref as ref


def criterion_bound(W16, s, ratios, G, sym, bits, h):
    """[n_ratio, N, K/G] bound on |e_gpu - e_exact| for the GPU's fp32 criterion: each d = W - w_hat
    off by at most delta = 2^-22 (|W| + |w_hat|), the sum over G terms off by G 2^-24 relative;
    e_exact is the oracle's fp64 error with the same energies h."""
    W = W16.astype(np.float64)
    N, K = W.shape
    out = np.zeros((len(ratios), N, K // G))
    for j, c in enumerate(ratios):
        qd = ref.quantize_pack(W16, s, G, sym, bits, clip=np.full((N, K // G), c, np.float32))
        w_hat = ref.dequantize(qd["qweight"], qd["scales"], qd["zeros"], G, s=s)
        d = np.abs(W - w_hat)
        delta = 2.0 ** -22 * (np.abs(W) + np.abs(w_hat))
        e = (h[None, :] * d * d).reshape(N, K // G, G).sum(axis=2)
        out[j] = (h[None, :] * (2 * d * delta + delta * delta)).reshape(N, K // G, G).sum(axis=2) \
            + G * 2.0 ** -24 * e
    return out
