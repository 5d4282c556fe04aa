"""AWQ on a Llama-style MLP block, end to end, through libawq's entry points.

The block is RMSNorm -> gate and up -> silu(gate) * up -> down. Quantising it follows
"AWQ Math", "Searching the scale" and "The equivalent transform", with the fold of the
"AWQ > Benefits and Practical Considerations" page:

1. x_n = rmsnorm(x, gamma) on the calibration tokens (awq_rmsnorm).
2. One alpha search for gate and up together (they share their input and therefore s):
   awq_search_scale on the stacked [W_gate; W_up].
3. The down projection's calibration input is propagated through the unquantised block:
   h = silu(x_n W_gate^T) * (x_n W_up^T) (the two dense fp16 products are plain cuBLAS GEMMs
   through torch; silu * up is awq_silu_mul), then a second search on W_down.
4. Fold: gamma *= 1/s_1 (awq_scale_rows on the norm weight) and the rows of W_up *= 1/s_2, so
   the folded block emits x_n / s_1 into gate/up and h / s_2 into down.
5. Pack gate and up with s_1 and down with s_2 (awq_quantize_pack); the quantised block runs
   the three W4A16 products with inv_s = NULL.

A stack of blocks is quantised one block at a time, each on the output of the unquantised
blocks before it. Every step of the AWQ path runs in the library's CUDA kernels; torch holds the
buffers and does the two dense fp16 GEMMs of step 3.
"""

from __future__ import annotations

from dataclasses import dataclass

from . import awq


@dataclass
class MLPWeights:
    """fp16 CUDA tensors: gamma [D], W_gate and W_up [I, D], W_down [D, I]."""
    gamma: object
    W_gate: object
    W_up: object
    W_down: object


@dataclass
class QuantMLP:
    """The folded, packed block and what the searches chose."""
    gamma: object            # folded norm weight [D] fp16
    gate: tuple              # (qweight, scales, zeros) of W_gate diag(s_1)
    up: tuple                # of diag(1/s_2) W_up diag(s_1)
    down: tuple              # of W_down diag(s_2)
    s1: object
    s2: object
    best1: int
    best2: int
    err1: object
    err2: object
    group_size: int


def _empty(torch, shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def rmsnorm(X, gamma, eps=1e-6):
    import torch
    T, D = X.shape
    Y = _empty(torch, (T, D), torch.float16, X)
    awq.awq_rmsnorm(X, T, D, gamma, eps, Y)
    return Y


def silu_mul(G, U):
    import torch
    H = _empty(torch, G.shape, torch.float16, G)
    awq.awq_silu_mul(G, U, G.numel(), H)
    return H


def _dense(X, W):
    """fp16 X @ W^T with fp32 accumulation (a plain cuBLAS GEMM)."""
    import torch
    old = torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction
    torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = False
    try:
        return torch.matmul(X, W.t())
    finally:
        torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = old


def mlp_fp16(X, w: MLPWeights, eps=1e-6) -> dict:
    """The unquantised block (fp16 activations between operations)."""
    xn = rmsnorm(X, w.gamma, eps)
    g = _dense(xn, w.W_gate)
    u = _dense(xn, w.W_up)
    h = silu_mul(g, u)
    return {"xn": xn, "g": g, "u": u, "h": h, "y": _dense(h, w.W_down)}


def quantize_mlp(X_calib, w: MLPWeights, alphas, group_size=128, eps=1e-6) -> QuantMLP:
    """Steps 1-5 above for one block on its calibration input X_calib [T, D] fp16."""
    import torch
    fp = mlp_fp16(X_calib, w, eps)
    W_gu = torch.cat([w.W_gate, w.W_up], dim=0).contiguous()
    err1, best1, s1, inv1 = awq.search_scale(W_gu, fp["xn"], alphas, group_size)
    err2, best2, s2, inv2 = awq.search_scale(w.W_down, fp["h"], alphas, group_size)
    gamma_f = w.gamma.clone()
    awq.awq_scale_rows(gamma_f, gamma_f.numel(), 1, 1, inv1)
    W_up_f = w.W_up.clone()
    awq.awq_scale_rows(W_up_f, W_up_f.shape[0], W_up_f.shape[1], W_up_f.shape[1], inv2)
    return QuantMLP(gamma=gamma_f,
                    gate=awq.quantize_pack(w.W_gate, s1, group_size),
                    up=awq.quantize_pack(W_up_f, s1, group_size),
                    down=awq.quantize_pack(w.W_down, s2, group_size),
                    s1=s1, s2=s2, best1=int(best1.item()), best2=int(best2.item()),
                    err1=err1, err2=err2, group_size=group_size)


def mlp_quantized(X, q: QuantMLP, eps=1e-6) -> dict:
    """The quantised block: folded norm, three W4A16 products with inv_s = NULL."""
    G = q.group_size
    xn = rmsnorm(X, q.gamma, eps)
    g = awq.w4a16_gemm(xn, *q.gate, None, G)
    u = awq.w4a16_gemm(xn, *q.up, None, G)
    h = silu_mul(g, u)
    return {"xn": xn, "g": g, "u": u, "h": h, "y": awq.w4a16_gemm(h, *q.down, None, G)}


def quantize_stack(X_calib, blocks, alphas, group_size=128, eps=1e-6) -> list:
    """Quantise a stack of blocks (y_l = MLP_l(x_l), x_{l+1} = y_l), each block on the output
    of the unquantised blocks before it."""
    out = []
    x = X_calib
    for w in blocks:
        out.append(quantize_mlp(x, w, alphas, group_size, eps))
        x = mlp_fp16(x, w, eps)["y"]
    return out


def run_stack(X, qblocks, eps=1e-6):
    """Output of the quantised stack."""
    x = X
    for q in qblocks:
        x = mlp_quantized(x, q, eps)["y"]
    return x
