"""Thin Python binding of libawq (``include/awq.h``): argument marshalling only.

The ``awq_*`` functions mirror the C entry points one to one; pointer arguments accept an
integer address or a CUDA ``torch.Tensor`` (its ``data_ptr()``), ``stream`` accepts a
``torch.cuda.Stream``, a raw handle or ``None`` (torch's current stream). A non-zero status
raises :class:`AwqError`. The convenience wrappers at the bottom only allocate outputs with
torch and call the same entry points; every step of the computation runs in the library's CUDA
kernels. There is no fallback: without the built library or a B300 the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libawq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "awq.h")

STATUS = {
    0: "AWQ_OK", 1: "AWQ_ERR_INVALID_ARG", 2: "AWQ_ERR_UNSUPPORTED_SHAPE",
    3: "AWQ_ERR_MISALIGNED", 4: "AWQ_ERR_WORKSPACE", 5: "AWQ_ERR_CUDA", 6: "AWQ_ERR_TIMEOUT",
    7: "AWQ_ERR_NO_DEVICE",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class AwqError(RuntimeError):
    """A libawq call returned a non-zero awq_status_t."""

    def __init__(self, fn: str, status: int):
        self.status = int(status)
        self.name = STATUS.get(int(status), f"status {status}")
        super().__init__(f"{fn}: {self.name}")


class QCfg(ctypes.Structure):
    _fields_ = [("group_size", ctypes.c_int32), ("symmetric", ctypes.c_int32),
                ("bits", ctypes.c_int32)]


_c_void_p, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t

_SIGNATURES = {
    "awq_calib_stats": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p]),
    "awq_search_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, QCfg]),
    "awq_search_scale": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _i64, _c_void_p,
                                        _c_void_p, _i32, QCfg, _c_void_p, _sz, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "awq_search_scale_static": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _i64,
                                               _c_void_p, _c_void_p, _i32, QCfg, _c_void_p,
                                               _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "awq_quantize_pack": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, QCfg, _c_void_p,
                                         _c_void_p, _c_void_p, _c_void_p]),
    "awq_quant_residual": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, QCfg,
                                          _c_void_p, _c_void_p, _c_void_p]),
    "awq_clip_search": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _i64, _c_void_p,
                                       _c_void_p, _i32, QCfg, _c_void_p, _c_void_p, _c_void_p]),
    "awq_quantize_pack_clip": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, QCfg,
                                              _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "awq_w4a16_gemm": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p,
                                      _c_void_p, _c_void_p, QCfg, _c_void_p, _c_void_p]),
    "awq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "awq_stream_status": (ctypes.c_int, [_c_void_p]),
    "awq_launch_count": (ctypes.c_uint64, []),
    "awq_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "awq_set_score_mode": (ctypes.c_int, [ctypes.c_int]),
    "awq_scale_rows": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p]),
    "awq_rmsnorm": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, ctypes.c_float, _c_void_p,
                                   _c_void_p]),
    "awq_silu_mul": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "awq_profile_begin": (ctypes.c_int, []),
    "awq_profile_end": (ctypes.c_int, [_c_void_p, _c_void_p]),
}

KERNELS = ("calib_stats", "scale_grid", "absmax", "residual", "score", "finalize",
           "quantize_pack", "gemv", "gemm_tc", "gram_prep", "gram", "score_gram", "gram_search",
           "scale_rows", "rmsnorm", "silu_mul", "clip_search")
SCORE_MODES = {"auto": 0, "direct": 1, "gram": 2, "gram_launches": 3}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libawq.so from the package directory (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m post_weight_quantization_stats_b300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list:
    """Names of every function the C header declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(awq_[a-z0-9_]+)\s*\(", text)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s):
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _cfg(group_size=128, symmetric=False, bits=4) -> QCfg:
    return QCfg(int(group_size), 1 if symmetric else 0, int(bits))


def _check(fn, status):
    if status != 0:
        raise AwqError(fn, status)


# ----------------------------------------------------------------------------- C entry points

def awq_calib_stats(X, T, K, ldx, mean_abs, stream=None):
    _check("awq_calib_stats", lib().awq_calib_stats(_ptr(X), T, K, ldx, _ptr(mean_abs),
                                                    _stream(stream)))


def awq_search_workspace_bytes(N, K, T, n_alpha, group_size=128, symmetric=False, bits=4) -> int:
    return int(lib().awq_search_workspace_bytes(N, K, T, n_alpha,
                                                _cfg(group_size, symmetric, bits)))


def awq_search_scale(W, N, K, X, T, mean_abs, alphas, n_alpha, group_size, symmetric, workspace,
                     ws_bytes, err_out, best_idx, s_out, inv_s_out, stream=None, bits=4):
    arr = (ctypes.c_float * int(n_alpha))(*[float(a) for a in alphas])
    _check("awq_search_scale", lib().awq_search_scale(
        _ptr(W), N, K, _ptr(X), T, _ptr(mean_abs), ctypes.cast(arr, ctypes.c_void_p), n_alpha,
        _cfg(group_size, symmetric, bits), _ptr(workspace), ws_bytes, _ptr(err_out), _ptr(best_idx),
        _ptr(s_out), _ptr(inv_s_out), _stream(stream)))


def awq_search_scale_static(W, N, K, X, T, mean_abs, alphas, n_alpha, group_size, symmetric,
                            err_out, best_idx, s_out, inv_s_out, stream=None, bits=4):
    """The alpha search with the library's static scratch array instead of a workspace, for
    callers that cannot allocate device memory (see include/awq.h). Allocates nothing."""
    arr = (ctypes.c_float * int(n_alpha))(*[float(a) for a in alphas])
    _check("awq_search_scale_static", lib().awq_search_scale_static(
        _ptr(W), N, K, _ptr(X), T, _ptr(mean_abs), ctypes.cast(arr, ctypes.c_void_p), n_alpha,
        _cfg(group_size, symmetric, bits), _ptr(err_out), _ptr(best_idx), _ptr(s_out),
        _ptr(inv_s_out), _stream(stream)))


def _header_scratch_bytes() -> int:
    """AWQ_SEARCH_STATIC_SCRATCH_BYTES as the C header defines it (``(a u * b u * ...)``)."""
    m = re.search(r"#define\s+AWQ_SEARCH_STATIC_SCRATCH_BYTES\s+\(([^)]*)\)", open(HEADER).read())
    if m is None:
        raise RuntimeError("AWQ_SEARCH_STATIC_SCRATCH_BYTES is not defined in include/awq.h")
    n = 1
    for f in m.group(1).split("*"):
        n *= int(f.strip().rstrip("uUlL"))
    return n


SEARCH_STATIC_SCRATCH_BYTES = _header_scratch_bytes()


def awq_quantize_pack(W, N, K, s, group_size, symmetric, qweight, scales, zeros, stream=None,
                      bits=4):
    _check("awq_quantize_pack", lib().awq_quantize_pack(
        _ptr(W), N, K, _ptr(s), _cfg(group_size, symmetric, bits), _ptr(qweight), _ptr(scales),
        _ptr(zeros), _stream(stream)))


def awq_clip_search(W, N, K, X, T, s, ratios, n_ratio, group_size, symmetric, energy, clip_out,
                    stream=None, bits=4):
    arr = (ctypes.c_float * int(n_ratio))(*[float(r) for r in ratios])
    _check("awq_clip_search", lib().awq_clip_search(
        _ptr(W), N, K, _ptr(X), T, _ptr(s), ctypes.cast(arr, ctypes.c_void_p), n_ratio,
        _cfg(group_size, symmetric, bits), _ptr(energy), _ptr(clip_out), _stream(stream)))


def awq_quantize_pack_clip(W, N, K, s, clip, group_size, symmetric, qweight, scales, zeros,
                           stream=None, bits=4):
    _check("awq_quantize_pack_clip", lib().awq_quantize_pack_clip(
        _ptr(W), N, K, _ptr(s), _ptr(clip), _cfg(group_size, symmetric, bits), _ptr(qweight),
        _ptr(scales), _ptr(zeros), _stream(stream)))


def awq_quant_residual(W, N, K, s, inv_s, group_size, symmetric, absmax_bits, D, stream=None,
                       bits=4):
    _check("awq_quant_residual", lib().awq_quant_residual(
        _ptr(W), N, K, _ptr(s), _ptr(inv_s), _cfg(group_size, symmetric, bits), _ptr(absmax_bits),
        _ptr(D), _stream(stream)))


def awq_w4a16_gemm(X, M, N, K, qweight, scales, zeros, inv_s, group_size, symmetric, Y,
                   stream=None, bits=4):
    _check("awq_w4a16_gemm", lib().awq_w4a16_gemm(
        _ptr(X), M, N, K, _ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(inv_s),
        _cfg(group_size, symmetric, bits), _ptr(Y), _stream(stream)))


def awq_scale_rows(A, rows, cols, lda, row_scale, stream=None):
    _check("awq_scale_rows", lib().awq_scale_rows(_ptr(A), rows, cols, lda, _ptr(row_scale),
                                                  _stream(stream)))


def awq_rmsnorm(X, T, D, gamma, eps, Y, stream=None):
    _check("awq_rmsnorm", lib().awq_rmsnorm(_ptr(X), T, D, _ptr(gamma), float(eps), _ptr(Y),
                                            _stream(stream)))


def awq_silu_mul(G, U, n, H, stream=None):
    _check("awq_silu_mul", lib().awq_silu_mul(_ptr(G), _ptr(U), n, _ptr(H), _stream(stream)))


def awq_status_string(status: int) -> str:
    return lib().awq_status_string(int(status)).decode()


def awq_stream_status(stream=None):
    _check("awq_stream_status", lib().awq_stream_status(_stream(stream)))


def awq_launch_count() -> int:
    return int(lib().awq_launch_count())


def awq_set_wait_limit_ns(limit_ns: int) -> int:
    return int(lib().awq_set_wait_limit_ns(int(limit_ns)))


def awq_set_score_mode(mode):
    """Process-wide choice of how the search scores candidates: "auto", "direct", "gram" or
    "gram_launches"."""
    _check("awq_set_score_mode", lib().awq_set_score_mode(SCORE_MODES.get(mode, mode)))


def awq_profile_begin():
    _check("awq_profile_begin", lib().awq_profile_begin())


def awq_profile_end() -> dict:
    """{kernel name: (launches, total ms)} of the launches since awq_profile_begin."""
    n = len(KERNELS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_uint64 * n)()
    _check("awq_profile_end", lib().awq_profile_end(ctypes.cast(ms, ctypes.c_void_p),
                                                    ctypes.cast(cnt, ctypes.c_void_p)))
    return {k: (int(cnt[i]), float(ms[i])) for i, k in enumerate(KERNELS) if cnt[i]}


# ----------------------------------------------------------------------------- tensor helpers

def calib_stats(X, stream=None):
    """m [K] fp32 = mean |X| over rows of a CUDA fp16 [T, K] tensor."""
    import torch
    T, K = X.shape
    m = torch.empty(K, dtype=torch.float32, device=X.device)
    awq_calib_stats(X, T, K, X.stride(0), m, stream)
    return m


def quantize_pack(W, s=None, group_size=128, symmetric=False, stream=None, bits=4):
    """(qweight [N, K/8] int32, scales [K/G, N] fp16, zeros [K/G, N] uint8) of W diag(s), with
    ``bits``-wide codes in the 4-bit nibbles."""
    import torch
    N, K = W.shape
    q = torch.empty((N, K // 8), dtype=torch.int32, device=W.device)
    sc = torch.empty((K // group_size, N), dtype=torch.float16, device=W.device)
    z = torch.empty((K // group_size, N), dtype=torch.uint8, device=W.device)
    awq_quantize_pack(W, N, K, s, group_size, symmetric, q, sc, z, stream, bits)
    return q, sc, z


def clip_search(W, X, s=None, ratios=None, group_size=128, symmetric=False, stream=None, bits=4):
    """(clip [K/G, N] fp32, energy [K] fp32): each group's clip ratio (awq_clip_search); ratios
    default to 1 - j/20 for j < 10."""
    import torch
    N, K = W.shape
    T = X.shape[0]
    if ratios is None:
        ratios = [1.0 - j / 20.0 for j in range(10)]
    energy = torch.empty(K, dtype=torch.float32, device=W.device)
    clip = torch.empty((K // group_size, N), dtype=torch.float32, device=W.device)
    awq_clip_search(W, N, K, X, T, s, ratios, len(ratios), group_size, symmetric, energy, clip,
                    stream, bits)
    return clip, energy


def quantize_pack_clip(W, s, clip, group_size=128, symmetric=False, stream=None, bits=4):
    """quantize_pack with each group's magnitudes bounded by clip [K/G, N] (see awq.h)."""
    import torch
    N, K = W.shape
    q = torch.empty((N, K // 8), dtype=torch.int32, device=W.device)
    sc = torch.empty((K // group_size, N), dtype=torch.float16, device=W.device)
    z = torch.empty((K // group_size, N), dtype=torch.uint8, device=W.device)
    awq_quantize_pack_clip(W, N, K, s, clip, group_size, symmetric, q, sc, z, stream, bits)
    return q, sc, z


def quant_residual(W, s, inv_s, group_size=128, symmetric=False, stream=None, bits=4):
    """(D [N, K] fp16, absmax_bits [1] int32): D = 2^p (W - Q(W diag(s)) diag(s)^-1), p from
    max|W| whose fp32 bits absmax_bits holds (see awq_quant_residual)."""
    import torch
    N, K = W.shape
    D = torch.empty((N, K), dtype=torch.float16, device=W.device)
    mx = torch.empty(1, dtype=torch.int32, device=W.device)
    awq_quant_residual(W, N, K, s, inv_s, group_size, symmetric, mx, D, stream, bits)
    return D, mx


def search_scale(W, X, alphas, group_size=128, symmetric=False, mean_abs=None, workspace=None,
                 stream=None, bits=4):
    """The alpha search: returns (err [n] fp32, best_idx [1] int32, s [K], inv_s [K])."""
    import torch
    N, K = W.shape
    T = X.shape[0]
    n = len(alphas)
    ws_bytes = awq_search_workspace_bytes(N, K, T, n, group_size, symmetric, bits)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=W.device)
    err = torch.empty(n, dtype=torch.float32, device=W.device)
    best = torch.empty(1, dtype=torch.int32, device=W.device)
    s = torch.empty(K, dtype=torch.float32, device=W.device)
    inv_s = torch.empty(K, dtype=torch.float32, device=W.device)
    awq_search_scale(W, N, K, X, T, mean_abs, alphas, n, group_size, symmetric, workspace,
                     workspace.numel(), err, best, s, inv_s, stream, bits)
    return err, best, s, inv_s


def w4a16_gemm(X, qweight, scales, zeros, inv_s=None, group_size=128, symmetric=False,
               stream=None):
    """Y [M, N] fp16 = X [M, K] (dequant(Q) diag(inv_s))^T."""
    import torch
    M, K = X.shape
    N = qweight.shape[0]
    Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    awq_w4a16_gemm(X, M, N, K, qweight, scales, zeros, inv_s, group_size, symmetric, Y, stream)
    return Y
