"""Seeded synthetic inputs for the AWQ per-linear-layer step.

This module is shared by the CUDA path's callers (tests, bench) and by the oracle's tests. It
holds none of the method's arithmetic: no activation statistic, no scale, no quantizer, no
error. It only draws random weights and calibration activations shaped like the workloads the
AWQ pages talk about, so that both sides can be fed byte-identical inputs.

Recipe (what each draw stands in for):

* Weights ``W [C_out, C_in]`` are i.i.d. normal with a per-workload sigma, rounded to fp16
  (AWQ Math page, "Shapes, granularity, and complexity": W is ``[C_out, C_in]``).
* Calibration activations ``X [T, C_in]`` are i.i.d. standard normal, rounded to fp16, with a
  small seeded set of "outlier" input channels scaled up. The AWQ Math page ("Saliency is an
  activation property") puts the salient fraction at roughly 0.1%-1% of channels; the
  Benefits page puts the calibration set at 128-512 samples. Where the outlier recipe asks for
  heavy tails, the outlier channels are Student-t (nu=3) draws.
* The MLP down-projection's calibration input in the Llama-7B MLP and the 7B-like stack is the
  gated activation of the generated ``X``: ``fp16(silu(X W_gate^T) * (X W_up^T))`` with fp32
  accumulation on the host. That is the model's forward pass, not part of AWQ. The Llama-70B
  layers both take plain draws with 1% outlier channels (no gating), as that workload states.

No public dataset or trained checkpoint is used or needed: these draws stand in for the
"calibration data" and model weights the pages talk about.

Seeds: ``numpy.random.PCG64(1000 * workload_id + layer_index)``.
"""

from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """One linear layer's synthetic problem: W [n, k] and calibration X [t, k]."""

    name: str
    n: int              # C_out
    k: int              # C_in
    t: int              # calibration tokens
    sigma: float        # weight standard deviation
    outlier_frac: float  # fraction of input channels that are outliers (rounded, >= 1)
    outlier_mult: float  # multiplier applied to outlier channels
    outlier_student_t: bool = False  # outlier channels drawn from Student-t (nu=3)
    outlier_count: int | None = None  # explicit outlier channel count (overrides frac)
    gated: bool = False  # MLP down-projection: input = fp16(silu(gate) * up) of the block's X


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named workload: an id (for seeding), its layers and the GEMM batch sizes it sweeps."""

    wid: int
    name: str
    layers: tuple
    gemm_m: tuple
    group_size: int = 128
    n_alpha: int = 20
    description: str = ""


WORKLOADS = {
    "tiny-512": Workload(
        1, "tiny-512",
        (LayerSpec("linear", 512, 512, 64, 0.02, 0.0, 20.0, False, 5),),
        (1, 16),
        description="single linear K=512 -> N=512, T=64, 5 outlier channels x20, G=128",
    ),
    "llama7b-attn-4096": Workload(
        2, "llama7b-attn-4096",
        (LayerSpec("attn_proj", 4096, 4096, 8192, 0.02, 0.005, 10.0, True, 20),),
        (1, 4, 16, 128),
        description="Llama-7B-shaped attention projection K=N=4096, T=8192, 0.5% Student-t "
                    "(nu=3) outlier channels x10, G=128",
    ),
    "llama7b-mlp": Workload(
        3, "llama7b-mlp",
        (LayerSpec("gate_proj", 11008, 4096, 8192, 0.02, 0.005, 10.0, True, 20),
         LayerSpec("up_proj", 11008, 4096, 8192, 0.02, 0.005, 10.0, True, 20),
         LayerSpec("down_proj", 4096, 11008, 8192, 0.02, 0.0, 1.0, False, 0, gated=True)),
        (1, 2, 4, 8, 16, 32),
        description="Llama-7B-shaped MLP gate/up 4096->11008 and down 11008->4096, T=8192; "
                    "down-proj input = fp16(silu(gate) * up) of the generated X",
    ),
    "llama70b-mlp": Workload(
        4, "llama70b-mlp",
        (LayerSpec("up_proj", 28672, 8192, 4096, 0.01, 0.01, 20.0, False),
         LayerSpec("down_proj", 8192, 28672, 4096, 0.01, 0.01, 20.0, False)),
        (1, 8, 64, 256, 1024),
        description="Llama-70B-shaped layers 8192->28672 and 28672->8192, T=4096, 1% outlier "
                    "channels x20, G=128",
    ),
    "llama7b-stack": Workload(
        5, "llama7b-stack",
        tuple(
            LayerSpec(f"l{i}.{p}", n, k, 2048, 0.02, 0.01, 20.0, False, gated=(p == "down"))
            for i in range(32)
            for p, n, k in (("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096),
                            ("o", 4096, 4096), ("gate", 11008, 4096), ("up", 11008, 4096),
                            ("down", 4096, 11008))
        ),
        tuple(range(1, 65)),
        description="7B-like decoder stack: 32 x {q,k,v,o 4096^2, gate/up 4096->11008, "
                    "down 11008->4096}, T=2048 per layer, 1% outlier channels x20",
    ),
}


def rng_for(wid: int, layer_index: int) -> np.random.Generator:
    """The generator every draw of one layer comes from."""
    return np.random.Generator(np.random.PCG64(1000 * wid + layer_index))


def _n_outliers(spec: LayerSpec) -> int:
    if spec.outlier_count is not None:
        return int(spec.outlier_count)
    if spec.outlier_frac <= 0.0:
        return 0
    return max(1, int(round(spec.outlier_frac * spec.k)))


def draw_weight(rng: np.random.Generator, n: int, k: int, sigma: float) -> np.ndarray:
    """W [n, k] ~ N(0, sigma), rounded to fp16."""
    w = rng.standard_normal((n, k), dtype=np.float32)
    w *= np.float32(sigma)
    return w.astype(np.float16)


def draw_activations(rng: np.random.Generator, t: int, k: int, n_out: int, mult: float,
                     student_t: bool) -> tuple:
    """X [t, k] ~ N(0,1) fp16 with ``n_out`` seeded outlier channels scaled by ``mult``.

    Returns ``(X, outlier_channels)``.
    """
    x = rng.standard_normal((t, k), dtype=np.float32)
    idx = np.sort(rng.choice(k, size=n_out, replace=False)) if n_out else np.zeros(0, np.int64)
    if n_out:
        if student_t:
            cols = rng.standard_t(3.0, size=(t, n_out)).astype(np.float32)
        else:
            cols = x[:, idx]
        x[:, idx] = cols * np.float32(mult)
    return x.astype(np.float16), idx


def gated_activation(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray) -> np.ndarray:
    """fp16(silu(X W_gate^T) * (X W_up^T)) with fp32 accumulation (the model's MLP forward)."""
    import torch  # CPU matmul only; this is input preparation, not the method

    xt = torch.from_numpy(x.astype(np.float32))
    g = xt @ torch.from_numpy(w_gate.astype(np.float32)).T
    u = xt @ torch.from_numpy(w_up.astype(np.float32)).T
    h = torch.nn.functional.silu(g) * u
    return h.to(torch.float16).numpy()


def _gate_up_indices(wl: Workload, layer_index: int) -> tuple:
    """Layer indices of the gate and up projections feeding a down projection."""
    if wl.name == "llama7b-stack":
        base = layer_index - (layer_index % 7)
        return base + 4, base + 5
    base = layer_index - (layer_index % len(wl.layers))
    return base + 0, base + 1


def make_layer(workload, layer_index: int = 0, t: int | None = None,
               n: int | None = None) -> dict:
    """Draw one layer of a workload: ``{"W", "X", "outliers", "spec"}``.

    ``t`` and ``n`` optionally keep only the leading calibration tokens / output rows of the
    same draws (bounded samples of a full-size layer).
    """
    wl = WORKLOADS[workload] if isinstance(workload, str) else workload
    spec = wl.layers[layer_index % len(wl.layers)]
    rng = rng_for(wl.wid, layer_index)
    w = draw_weight(rng, spec.n, spec.k, spec.sigma)
    if spec.gated:
        gate_i, up_i = _gate_up_indices(wl, layer_index)
        g = make_layer(wl, gate_i, t=t)
        up_spec = wl.layers[up_i % len(wl.layers)]
        w_up = draw_weight(rng_for(wl.wid, up_i), up_spec.n, up_spec.k, up_spec.sigma)
        x = gated_activation(g["X"], g["W"], w_up)
        outl = np.zeros(0, np.int64)
    else:
        x, outl = draw_activations(rng, spec.t, spec.k, _n_outliers(spec), spec.outlier_mult,
                                   spec.outlier_student_t)
    if t is not None:
        x = x[: int(t)]
    if n is not None:
        w = w[: int(n)]
    return {"W": np.ascontiguousarray(w), "X": np.ascontiguousarray(x), "outliers": outl,
            "spec": spec}


def random_layer(seed: int, n: int, k: int, t: int, sigma: float = 0.02, n_out: int = 0,
                 mult: float = 20.0, student_t: bool = False) -> dict:
    """An ad-hoc layer of any shape (parity tests, edge cases), same recipe as the workloads."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = draw_weight(rng, n, k, sigma)
    x, outl = draw_activations(rng, t, k, n_out, mult, student_t)
    return {"W": w, "X": x, "outliers": outl}


def alpha_grid(n_alpha: int = 20) -> np.ndarray:
    """The search grid alpha_i = i / n_alpha, i = 0..n_alpha-1, as fp32 (0 in, 1 out)."""
    return (np.arange(n_alpha, dtype=np.float64) / n_alpha).astype(np.float32)


def clip_ratios(n_ratio: int = 10) -> np.ndarray:
    """The clipping grid c_j = 1 - j/20, j = 0..n_ratio-1, as fp32 (1 keeps the full range)."""
    return (1.0 - np.arange(n_ratio, dtype=np.float64) / 20.0).astype(np.float32)


def stack_bytes(workload: str = "llama7b-stack", group_size: int = 128) -> int:
    """Packed bytes (codes + fp16 scale + uint8 zero) of every layer of a workload."""
    wl = WORKLOADS[workload]
    total = 0
    for s in wl.layers:
        total += s.n * s.k // 2 + 3 * s.n * (s.k // group_size)
    return total


__all__ = ["LayerSpec", "Workload", "WORKLOADS", "make_layer", "random_layer", "alpha_grid",
           "rng_for", "draw_weight", "draw_activations", "gated_activation", "stack_bytes"]

