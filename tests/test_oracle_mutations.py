"""Plant plausible mistakes in copies of the oracle (on the CPU) and check the pins catch each.

Each mutation is a textual edit of ``oracle/awq_ref.py`` executed as a throw-away module; the
real oracle is never modified. A mutation counts as caught when any pin raises (a wrong value
or a shape error alike).
"""

import os
import types

import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "awq_ref.py")

MUTATIONS = {
    "range divisor 16 instead of 15": ("rng_ / qmax", "rng_ / (qmax + 1)"),
    "zero point sign flipped": ("np.rint(fl32(-lo / step)", "np.rint(fl32(lo / step)"),
    "zero point added with wrong sign": ("grp / step[:, :, None]).astype(np.float64)) + z",
                                         "grp / step[:, :, None]).astype(np.float64)) - z"),
    "floor instead of round": ("r = np.rint(fl32(grp", "r = np.floor(fl32(grp"),
    "range not widened to hold 0": ("hi = np.maximum(np.max(grp, axis=2), 0.0)",
                                    "hi = np.max(grp, axis=2)"),
    "symmetric divisor 7": ("fl32(amax / half)", "fl32(amax / (half - 1))"),
    "symmetric clamp [-7, 7]": ("np.clip(r, -half, half - 1)", "np.clip(r, -half + 1, half - 1)"),
    "scaled weight divides by s": ("fl32(W64 * s32[None, :])", "fl32(W64 / s32[None, :])"),
    "dequant multiplies by s": ("w_hat = w_hat / np.asarray(s", "w_hat = w_hat * np.asarray(s"),
    "dequant adds the zero point": ("(codes - zero[:, g_of_k])", "(codes + zero[:, g_of_k])"),
    "dequant uses the fp32 step": ("step = np.asarray(scales, dtype=np.float16)",
                                   "step = np.asarray(scales, dtype=np.float32) * 1.001"),
    "wrong group index": ("g_of_k = np.arange(K) // group_size",
                          "g_of_k = np.arange(K) % (K // group_size)"),
    "nibble order reversed in pack": ("<< np.uint64(4 * i)", "<< np.uint64(4 * (7 - i))"),
    "residual adds the dequantised weight": ("np.asarray(W, dtype=np.float64) - w_hat",
                                             "np.asarray(W, dtype=np.float64) + w_hat"),
    "residual exponent off by one": ("return 14 - int(e)", "return 15 - int(e)"),
    "asymmetric levels fixed at 16": ("qmax = 2 ** bits - 1", "qmax = 15"),
    "symmetric half-range fixed at 8": ("half = 2 ** (bits - 1)", "half = 8"),
    "statistic drops the absolute value": ("total += np.abs(X64[t])", "total += X64[t]"),
    "statistic divides by T - 1": ("return total / T", "return total / (T - 1)"),
    "statistic uses the max": ("total += np.abs(X64[t])",
                               "total = np.maximum(total, np.abs(X64[t]) * T)"),
    "scale exponent 1 - alpha": ("base[None, :] ** a[:, None]",
                                 "base[None, :] ** (1.0 - a[:, None])"),
    "no floor on the statistic": ("np.maximum(np.asarray(m, dtype=np.float64), eps)",
                                  "np.asarray(m, dtype=np.float64)"),
    "error is a sum, not a mean": ("return float(np.mean((y - y_hat) ** 2))",
                                   "return float(np.sum((y - y_hat) ** 2))"),
    "search error is a sum": ("err[i] = float(np.mean((y - layer_output(X, w_hat)) ** 2))",
                              "err[i] = float(np.sum((y - layer_output(X, w_hat)) ** 2))"),
    "search compares against the quantised scaled weight": (
        "err[i] = float(np.mean((y - layer_output(X, w_hat)) ** 2))",
        "err[i] = float(np.mean((y - layer_output(X, w_hat * s[None, :])) ** 2))"),
    "argmin picks the last minimiser": ("best = int(np.argmin(err))",
                                        "best = int(len(err) - 1 - np.argmin(err[::-1]))"),
    "gemm applies inv_s as a divide": (
        "w_hat = w_hat * np.asarray(inv_s, dtype=np.float32)",
        "w_hat = w_hat / np.asarray(inv_s, dtype=np.float32)"),
    "gemm output columns reversed": ("return np.asarray(X, dtype=np.float64) @ w_hat.T",
                                    "return (np.asarray(X, dtype=np.float64) @ w_hat.T)[:, ::-1]"),
    "packed bytes miss the zero points": ("return n * k // 2 + 3 * n * (k // group_size)",
                                          "return n * k // 2"),
    "packed bytes count a byte per code": ("return n * k // 2 + 3 * n * (k // group_size)",
                                           "return n * k + 3 * n * (k // group_size)"),
    "all-zero group keeps step 0": ("        step[step == 0.0] = 1.0\n        z = np.clip",
                                    "        z = np.clip"),
    "clip bound divides by the ratio": ("np.max(np.abs(grp), axis=2) * c)",
                                        "np.max(np.abs(grp), axis=2) / c)"),
    "clip bound left at the low end only": ("            hi = np.minimum(hi, bound)\n", ""),
    "clip error not weighted by the energy": ("err[j] = (d * d * h[None, :])",
                                              "err[j] = (d * d * h.mean())"),
    "clip error on |d| instead of d squared": ("err[j] = (d * d * h[None, :])",
                                               "err[j] = (np.abs(d) * h[None, :])"),
    "energy sums |x|": ("h += X64[t] * X64[t]", "h += np.abs(X64[t])"),
    "clip picks the last minimiser": ("best = np.argmin(err, axis=0)",
                                      "best = len(r) - 1 - np.argmin(err[::-1], axis=0)"),
}


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("awq_ref_mutant")
    with __import__("warnings").catch_warnings():
        __import__("warnings").simplefilter("ignore")
        exec(compile(src.replace(old, new), "awq_ref_mutant.py", "exec"), mod.__dict__)
    return mod


def _caught(mod):
    import warnings
    for pin in oracle_pins.ALL_PINS:
        try:
            with warnings.catch_warnings():
                warnings.simplefilter("ignore")
                pin(mod)
        except Exception:   # noqa: BLE001 - an assertion or a shape error both count
            return pin.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    old, new = MUTATIONS[name]
    assert _caught(_mutant(old, new)) is not None, f"no pin caught: {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _caught(_mutant("", "")) is None
