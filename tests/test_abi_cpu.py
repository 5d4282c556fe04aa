"""The C-ABI library without a GPU: it builds, loads, exports every function the header
declares, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import subprocess

import pytest

from post_weight_quantization_stats_b300 import awq, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return awq.lib()


def test_header_declares_the_boundary():
    names = awq.header_functions()
    for fn in ("awq_calib_stats", "awq_search_scale", "awq_quantize_pack", "awq_w4a16_gemm",
               "awq_search_workspace_bytes", "awq_status_string", "awq_stream_status"):
        assert fn in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", awq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for fn in awq.header_functions():
        assert fn in exported, fn
        assert hasattr(L, fn)


def test_status_strings(L):
    for code, name in awq.STATUS.items():
        assert awq.awq_status_string(code) == name


def test_workspace_bytes(L):
    awq.awq_set_score_mode("direct")
    try:
        n = awq.awq_search_workspace_bytes(4096, 4096, 8192, 20)
    finally:
        awq.awq_set_score_mode("auto")
    assert n >= 2 * 4096 * 4096 * 2      # two fp16 residual buffers (overlapped schedule)
    assert n < 2 * 4096 * 4096 * 2 + (4 << 20)
    assert awq.awq_search_workspace_bytes(4096, 4100, 8192, 20) == 0   # K % G
    assert awq.awq_search_workspace_bytes(4096, 4096, 8192, 65) == 0   # too many alphas
    assert awq.awq_search_workspace_bytes(4096, 4096, 8192, 20, group_size=96) == 0


def test_score_mode_and_gram_workspace(L):
    """AUTO scores through H = X^T X where that takes fewer tensor-core steps: for the
    4096 x 4096 layer with 8192 tokens the workspace then adds X^T [K, T], the fp16 triangle of
    H [K, K] and the column sums [T / 64, K]; with 512 tokens the direct product is cheaper."""
    N = K = 4096
    T = 8192
    direct = 2 * N * K * 2
    gram_extra = K * T * 2 + K * K * 2 + (T // 64) * K * 4
    n = awq.awq_search_workspace_bytes(N, K, T, 20)
    assert direct + gram_extra <= n < direct + gram_extra + (4 << 20)
    small_t = awq.awq_search_workspace_bytes(N, K, 512, 20)
    assert direct <= small_t < direct + (4 << 20)
    awq.awq_set_score_mode("gram")
    try:
        forced = awq.awq_search_workspace_bytes(N, K, 512, 20)
        assert direct + K * 512 * 2 + K * K * 2 <= forced < direct + K * 512 * 2 + K * K * 2 + (4 << 20)
        # T = 1 pads to 64 tokens
        assert awq.awq_search_workspace_bytes(128, 64, 1, 2, group_size=64) >= 2 * 64 * 64 * 2
    finally:
        awq.awq_set_score_mode("auto")
    with pytest.raises(awq.AwqError):
        awq.awq_set_score_mode(4)
    # GRAM needs K % 64 == 0: forced on K = 800 (G = 32) it is refused before any launch
    A = 1 << 20
    alphas = (ctypes.c_float * 2)(0.0, 0.5)
    cfg = awq.QCfg(32, 0)
    awq.awq_set_score_mode("gram")
    try:
        assert awq.awq_search_workspace_bytes(64, 800, 256, 2, group_size=32) == 0
        assert L.awq_search_scale(A, 64, 800, A, 256, None, ctypes.cast(alphas, ctypes.c_void_p),
                                  2, cfg, A, 1 << 30, A, A, None, None, None) == \
            awq.STATUS_CODE["AWQ_ERR_UNSUPPORTED_SHAPE"]
    finally:
        awq.awq_set_score_mode("auto")
    assert awq.awq_search_workspace_bytes(64, 800, 256, 2, group_size=32) > 0
    assert awq.awq_search_workspace_bytes(N, K, T, 20) == n


def _code(L, fn, *args):
    return getattr(L, fn)(*args)


def test_host_validation_rejects_without_cuda(L):
    cfg = awq.QCfg(128, 0)
    A = 1 << 20   # a fake, 16-byte aligned address: never dereferenced (rejected first)
    S = awq.STATUS_CODE
    # NULL pointers / sizes
    assert _code(L, "awq_calib_stats", None, 8, 128, 128, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert _code(L, "awq_calib_stats", A, 0, 128, 128, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert _code(L, "awq_calib_stats", A, 8, 128, 100, A, None) == S["AWQ_ERR_UNSUPPORTED_SHAPE"]
    assert _code(L, "awq_calib_stats", A + 2, 8, 128, 128, A, None) == S["AWQ_ERR_MISALIGNED"]
    assert _code(L, "awq_quantize_pack", A, 16, 100, None, cfg, A, A, A, None) == \
        S["AWQ_ERR_UNSUPPORTED_SHAPE"]
    assert _code(L, "awq_quantize_pack", A, 16, 256, None, awq.QCfg(48, 0), A, A, A, None) == \
        S["AWQ_ERR_INVALID_ARG"]
    for bad_bits in (1, 5, 8, -1):                        # code widths: 0 (= 4), 2, 3, 4
        assert _code(L, "awq_quantize_pack", A, 16, 256, None, awq.QCfg(128, 0, bad_bits), A, A,
                     A, None) == S["AWQ_ERR_INVALID_ARG"]
        assert awq.lib().awq_search_workspace_bytes(16, 256, 8, 2, awq.QCfg(128, 0, bad_bits)) == 0
    assert _code(L, "awq_quantize_pack", A, 16, 256, None, cfg, A, A, None, None) == \
        S["AWQ_ERR_INVALID_ARG"]                          # asymmetric needs zeros
    assert _code(L, "awq_quantize_pack", A, 16, 256, A + 4, cfg, A, A, A, None) == \
        S["AWQ_ERR_MISALIGNED"]
    assert _code(L, "awq_w4a16_gemm", A, 0, 16, 256, A, A, A, None, cfg, A, None) == \
        S["AWQ_ERR_INVALID_ARG"]
    assert _code(L, "awq_w4a16_gemm", A, 4, 16, 256, A, A, A, None, cfg, A + 8, None) == \
        S["AWQ_ERR_MISALIGNED"]
    assert _code(L, "awq_quant_residual", A, 16, 256, None, A, cfg, A, A, None) == \
        S["AWQ_ERR_INVALID_ARG"]                          # s is required
    assert _code(L, "awq_quant_residual", A, 16, 256, A, A, cfg, None, A, None) == \
        S["AWQ_ERR_INVALID_ARG"]                          # so is the max|W| word
    assert _code(L, "awq_quant_residual", A, 16, 100, A, A, cfg, A, A, None) == \
        S["AWQ_ERR_UNSUPPORTED_SHAPE"]
    assert _code(L, "awq_quant_residual", A, 16, 256, A, A + 4, cfg, A, A, None) == \
        S["AWQ_ERR_MISALIGNED"]
    assert _code(L, "awq_quant_residual", A, 16, 256, A, A, cfg, A + 2, A, None) == \
        S["AWQ_ERR_MISALIGNED"]
    alphas = (ctypes.c_float * 2)(0.0, 0.5)
    ap = ctypes.cast(alphas, ctypes.c_void_p)
    awq.awq_set_score_mode("direct")   # the direct schedules' sizes (AUTO may ask for more)
    try:
        ws = awq.awq_search_workspace_bytes(16, 256, 8, 2)
    finally:
        awq.awq_set_score_mode("auto")
    ws_min = ws - (16 * 256 * 2 + 255) // 256 * 256    # one residual buffer instead of two
    assert _code(L, "awq_search_scale", A, 16, 256, A, 8, None, ap, 2, cfg, A, ws_min, A, A,
                 None, None, None) == S["AWQ_ERR_NO_DEVICE"]    # accepted: only the device check fails
    assert _code(L, "awq_search_scale", A, 16, 256, A, 8, None, ap, 2, cfg, A, ws_min - 1, A, A,
                 None, None, None) == S["AWQ_ERR_WORKSPACE"]
    assert _code(L, "awq_search_scale", A, 16, 256, A, 8, None, ap, 0, cfg, A, ws, A, A,
                 None, None, None) == S["AWQ_ERR_INVALID_ARG"]
    assert _code(L, "awq_search_scale", A, 16, 256, A, 8, None, None, 2, cfg, A, ws, A, A,
                 None, None, None) == S["AWQ_ERR_INVALID_ARG"]


def test_valid_call_without_a_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = awq.QCfg(128, 0)
    A = 1 << 20
    assert _code(L, "awq_quantize_pack", A, 16, 256, None, cfg, A, A, A, None) == \
        awq.STATUS_CODE["AWQ_ERR_NO_DEVICE"]
    assert _code(L, "awq_quant_residual", A, 16, 256, A, A, cfg, A, A, None) == \
        awq.STATUS_CODE["AWQ_ERR_NO_DEVICE"]
    for bits in (2, 3, 4):                                # accepted: only the device check fails
        assert _code(L, "awq_quantize_pack", A, 16, 256, None, awq.QCfg(128, 1, bits), A, A, A,
                     None) == awq.STATUS_CODE["AWQ_ERR_NO_DEVICE"]


def test_launch_counter_starts_without_launches(L):
    assert awq.awq_launch_count() >= 0
    old = awq.awq_set_wait_limit_ns(123)
    assert awq.awq_set_wait_limit_ns(old) == 123


def test_static_search_checks_arguments_before_its_size(L):
    """awq_search_scale_static makes awq_search_scale's argument checks first: for a layer too
    large for its static array, a NULL pointer, a misaligned pointer or T K beyond 2^31 gets the
    same error as from the workspace entry point; only valid inputs are refused for their size
    (AWQ_ERR_WORKSPACE). All of it before any CUDA call."""
    cfg = awq.QCfg(128, 0)
    A = 1 << 20
    S = awq.STATUS_CODE
    alphas = (ctypes.c_float * 2)(0.0, 0.5)
    ap = ctypes.cast(alphas, ctypes.c_void_p)
    N = K = 8192
    T = 64
    assert awq.awq_search_workspace_bytes(N, K, T, 2) > awq.SEARCH_STATIC_SCRATCH_BYTES

    def static(W=A, X=A, T=T, alphas=ap, n_alpha=2, err=A, best=A, s=None, inv=None, cfg=cfg):
        return L.awq_search_scale_static(W, N, K, X, T, None, alphas, n_alpha, cfg, err, best, s,
                                         inv, None)

    def workspace(W=A, X=A, T=T, alphas=ap, n_alpha=2, err=A, best=A, s=None, inv=None, cfg=cfg):
        return L.awq_search_scale(W, N, K, X, T, None, alphas, n_alpha, cfg, A, 1 << 40, err,
                                  best, s, inv, None)

    for kw, want in (({"W": None}, "AWQ_ERR_INVALID_ARG"), ({"best": None}, "AWQ_ERR_INVALID_ARG"),
                     ({"alphas": None}, "AWQ_ERR_INVALID_ARG"), ({"n_alpha": 0}, "AWQ_ERR_INVALID_ARG"),
                     ({"cfg": awq.QCfg(96, 0)}, "AWQ_ERR_INVALID_ARG"),
                     ({"X": A + 2}, "AWQ_ERR_MISALIGNED"), ({"s": A + 4}, "AWQ_ERR_MISALIGNED"),
                     ({"T": 1 << 19}, "AWQ_ERR_UNSUPPORTED_SHAPE")):
        assert static(**kw) == S[want], kw
        assert workspace(**kw) == S[want], kw
    assert static() == S["AWQ_ERR_WORKSPACE"]
    # a shape the array holds passes every host check and stops only at the device lookup
    import torch
    if not torch.cuda.is_available():
        assert L.awq_search_scale_static(A, 16, 256, A, 8, None, ap, 2, cfg, A, A, None, None,
                                         None) == S["AWQ_ERR_NO_DEVICE"]


def test_clip_calls_reject_bad_arguments_on_the_host(L):
    """awq_clip_search and awq_quantize_pack_clip: ratio counts and values, NULL outputs, sizes
    and alignment are checked before any CUDA call."""
    cfg = awq.QCfg(128, 0)
    A = 1 << 20
    S = awq.STATUS_CODE

    def ratios(*v):
        arr = (ctypes.c_float * len(v))(*v)
        return ctypes.cast(arr, ctypes.c_void_p), arr

    good, keep1 = ratios(1.0, 0.9)
    zero, keep2 = ratios(1.0, 0.0)
    big, keep3 = ratios(1.0, 1.5)
    call = L.awq_clip_search
    assert call(A, 16, 256, A, 8, None, good, 0, cfg, A, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert call(A, 16, 256, A, 8, None, good, 33, cfg, A, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert call(A, 16, 256, A, 8, None, zero, 2, cfg, A, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert call(A, 16, 256, A, 8, None, big, 2, cfg, A, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert call(A, 16, 256, A, 8, None, good, 2, cfg, None, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert call(A, 16, 256, A, 8, None, good, 2, cfg, A, None, None) == S["AWQ_ERR_INVALID_ARG"]
    assert call(A, 16, 100, A, 8, None, good, 2, cfg, A, A, None) == S["AWQ_ERR_UNSUPPORTED_SHAPE"]
    assert call(A, 16, 256, A + 2, 8, None, good, 2, cfg, A, A, None) == S["AWQ_ERR_MISALIGNED"]
    assert call(A, 16, 256, A, 8, None, good, 2, cfg, A + 4, A, None) == S["AWQ_ERR_MISALIGNED"]
    pack = L.awq_quantize_pack_clip
    assert pack(A, 16, 256, None, None, cfg, A, A, A, None) == S["AWQ_ERR_INVALID_ARG"]
    assert pack(A, 16, 256, None, A + 2, cfg, A, A, A, None) == S["AWQ_ERR_MISALIGNED"]
    import torch
    if not torch.cuda.is_available():
        assert call(A, 16, 256, A, 8, None, good, 2, cfg, A, A, None) == S["AWQ_ERR_NO_DEVICE"]
        assert pack(A, 16, 256, None, A, cfg, A, A, A, None) == S["AWQ_ERR_NO_DEVICE"]
