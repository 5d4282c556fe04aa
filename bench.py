#!/usr/bin/env python
"""Benchmark of the AWQ per-linear-layer step on one B300 (or N, one independent layer each).

One step = the whole hot path over one synthetic layer shaped like a Llama-7B attention
projection (K = N = 4096, T = 8192 calibration tokens, 20 alphas, group 128):
  calibration statistic -> alpha search (scale grid, per-alpha residual + tcgen05 scoring,
  argmin) -> final quantise/pack -> W4A16 matmul at M = 1, 4, 16, 128.
Inputs are resident in HBM when the timed region starts; L2 is flushed (256 MB write) between
steps, outside the per-step CUDA events. The headline is layers/s; the JSON line also carries the
roofline of the dominant kernel (the scoring GEMM), per-kernel live timings, a W4A16 sweep
(CUDA-graph replays over weight sets larger than L2, on this layer and the Llama-70B MLP shapes)
with its decode (HBM) and M=1024 (tensor) rooflines, one decode step through all 224 linears of
the synthetic 7B stack, the end-to-end number through host buffers, the CPU oracle baseline and
the SM clocks seen during the timed region (NVML, every ~10 ms).

``--impl reference`` times the CPU oracle instead (bounded samples of the same layer).
Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under torchrun, every rank
runs its own layer (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from post_weight_quantization_stats_b300 import synth  # noqa: E402

METRIC = "W4A16 GEMV/GEMM HBM TB/s & TFLOP/s vs roofline; AWQ search layers/sec"
UNIT = "layers/s"
WORKLOAD = "llama7b-attn-4096"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-hbm-sweep", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the search at the 7B-MLP, 70B-MLP and 224-linear stack workloads")
    ap.add_argument("--case", default=None,
                    help="run one kernel family on a small case and exit (for profiler "
                         "captures): 'search' (statistic, alpha search and pack of the "
                         "workload's layer, 3 times), 'clip' (one layer step, then the clipping search "
                         "and clipped pack 5 times) or 'w4a16:N:K:M' (4 launches of one shape)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------ host helpers

def dist_env():
    """(rank, local_rank, world) from the torchrun environment (defaults: single process)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def layer_units(wl_name):
    """Layers one step processes and their shapes (every rank runs one layer of the workload)."""
    wl = synth.WORKLOADS[wl_name]
    spec = wl.layers[0]
    return wl, spec


def source_digest(sources):
    """sha256 prefix of the kernel's source files (under the package's csrc/), concatenated in
    the given order; None if one is missing."""
    import hashlib
    h = hashlib.sha256()
    for name in sources:
        src = os.path.join(ROOT, "post_weight_quantization_stats_b300", "csrc", name)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_md, sources):
    """DRAM bytes per launch from a committed ncu summary, or None when any source the kernel
    is built from has changed since the counters were taken (the digest no longer matches)."""
    if profile_md is None:
        return None
    path = os.path.join(ROOT, "profiles", profile_md)
    sha = source_digest(sources)
    if sha is None or not os.path.exists(path):
        return None
    text = open(path).read()
    want, traffic = None, None
    for line in text.splitlines():
        if line.startswith("source_sha256_16:"):
            want = line.split(":", 1)[1].strip()
        if line.startswith("| traffic_bytes_per_launch |"):
            traffic = int(line.split("|")[2].strip())
    return traffic if want == sha else None


def layer_for_rank(wl_name, rank):
    """The layer rank ``rank`` processes: rank 0 gets the workload's first layer; every other
    rank an independent draw of the same shape (its own seed), so N ranks do N layers."""
    wl = synth.WORKLOADS[wl_name]
    if rank == 0:
        return synth.make_layer(wl_name, 0)
    if len(wl.layers) > 1:
        return synth.make_layer(wl_name, rank % len(wl.layers))
    own = synth.Workload(wl.wid * 100 + rank, wl.name, wl.layers, wl.gemm_m)
    return synth.make_layer(own, 0)


def algorithmic(spec, G, n_alpha, gemm_m):
    """Algorithmic bytes/flops per launch of each kernel for one layer (N, K, T)."""
    N, K, T = spec.n, spec.k, spec.t
    packed = N * K // 2 + 3 * N * (K // G)
    return {
        "calib_stats": {"bytes": 2 * T * K + 4 * K},
        "absmax": {"bytes": 2 * N * K},
        "residual": {"bytes": 2 * N * K + 8 * K + 2 * N * K},
        "score": {"flops": 2 * T * N * K},
        # Gram schedule: X^T and column sums (read X, write X^T), H's lower triangle (T K (K+1)
        # flops), then per alpha sum_n d_n^T H' d_n: K (K+1) / 2 multiply-adds and a K-long dot
        # per output
        "gram_prep": {"bytes": 2 * T * K + 2 * ((T + 63) // 64 * 64) * K + 4 * ((T + 63) // 64) * K,
                      "launches": 2},   # transpose + column-sum maximum, bytes for both
        "gram": {"flops": T * K * (K + 1)},
        "score_gram": {"flops": N * K * (K + 3)},
        # the persistent launch: H's triangle and every alpha's score
        "gram_search": {"flops": T * K * (K + 1) + n_alpha * N * K * (K + 3)},
        "quantize_pack": {"bytes": 2 * N * K + 4 * K + packed},
        "gemv": {m: {"bytes": packed + 2 * m * K + 2 * m * N + 4 * K, "flops": 2 * m * N * K}
                 for m in gemm_m},
        "packed_bytes": packed,
    }


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None
        self.path = None

    def start(self):
        if self.bus_id:
            probe = subprocess.run(["nvidia-smi", "-i", self.bus_id, "--query-gpu=index",
                                    "--format=csv,noheader"], capture_output=True, text=True)
            if probe.returncode != 0:
                self.bus_id = None
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        return summarize_clocks(rows)


class NvmlClockSampler:
    """SM clock, max clock, power and clock-event reasons read through NVML every ~10 ms on a
    background thread (many samples even for a timed region of a few hundred ms). Produces the
    same rows as ClockSampler; raises if NVML is unavailable."""

    # NVML clock-event reason bits (nvml.h): sw power cap, hw slowdown, sw / hw thermal slowdown
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    NVML_CLOCK_SM = 1

    def __init__(self, bus_id=None, period_s=0.01):
        import ctypes
        self.ct = ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")   # the driver's NVML (read-only queries)
        self.nv = nv
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        rc = -1
        if bus_id:
            rc = nv.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(h))
        if rc != 0 and nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML device handle")
        self.h = h
        self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.rows = []
        self._stop = None
        self._thread = None

    def _query(self):
        ct, nv = self.ct, self.nv
        sm, mx, pw, r = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if (nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(sm)) or
                nv.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(mx)) or
                nv.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw)) or
                self.reasons_fn(self.h, ct.byref(r))):
            return None
        return sm.value, mx.value, pw.value / 1000.0, r.value

    def _loop(self):
        while not self._stop.is_set():
            q = self._query()
            if q is not None:
                sm, mx, pw, r = q
                act = ["Active" if r & self.BITS[k] else "Not Active"
                       for k in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                 "sw_power_cap")]
                self.rows.append(["0", str(sm), str(mx), f"{pw:.1f}", hex(r)] + act)
            self._stop.wait(self.period)

    def start(self):
        import threading
        if self._query() is None:
            raise RuntimeError("NVML queries failed")
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=5)
        out = summarize_clocks(self.rows)
        out["source"] = "nvml"
        return out


class _FallbackSampler(ClockSampler):
    """The nvidia-smi sampler, recording why NVML could not be used."""

    def __init__(self, bus_id, reason):
        super().__init__(bus_id)
        self.reason = reason

    def stop(self):
        out = super().stop()
        out["source"] = "nvidia-smi"
        out["nvml_error"] = self.reason
        return out


def clock_sampler(bus_id):
    """NVML sampler when NVML works, else the nvidia-smi one."""
    try:
        return NvmlClockSampler(bus_id).start()
    except Exception as e:  # noqa: BLE001
        return _FallbackSampler(bus_id, f"{type(e).__name__}: {e}"[:200]).start()


def summarize_clocks(rows):
    """Median SM clock, max clock and every throttle reason seen Active in the samples."""
    def num(x):
        try:
            return float(x)
        except ValueError:
            return None

    sm = [num(r[1]) for r in rows if num(r[1]) is not None]
    mx = [num(r[2]) for r in rows if num(r[2]) is not None]
    reasons = set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for r in rows:
        for name, val in zip(names, r[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(value, world):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------ CPU oracle

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001
        pass
    return os.cpu_count() or 1


def oracle_layer_seconds(layer, alphas, gemm_m, G, n_rows, m_cache=None):
    """Time the oracle on the first ``n_rows`` output rows of the layer (full T and K) and
    extrapolate linearly in rows to the whole layer. Returns (seconds per layer, detail)."""
    from oracle import awq_ref as ref

    W, X = layer["W"], layer["X"]
    N = W.shape[0]
    t0 = time.perf_counter()
    m = ref.calib_stats(X) if m_cache is None else m_cache
    t_stats = time.perf_counter() - t0
    Ws = W[:n_rows]
    t1 = time.perf_counter()
    r = ref.search_scale(Ws, X, alphas, G, m=m)
    qd = ref.quantize_pack(Ws, r["s"], G)
    inv = (np.float32(1) / r["s"]).astype(np.float32)
    for M in gemm_m:
        ref.w4a16_gemm(X[:M], qd["qweight"], qd["scales"], qd["zeros"], G, inv_s=inv)
    t_rows = time.perf_counter() - t1
    stats_time = t_stats if m_cache is None else 0.0
    per_layer = stats_time + t_rows * (N / n_rows)
    return per_layer, {"t_stats": t_stats, "t_rows": t_rows, "n_rows": n_rows, "m": m}


def choose_rows(layer, alphas, gemm_m, G, budget_s):
    """Output-row count whose oracle time fits ``budget_s`` (probe with 16 rows, scale)."""
    N = layer["W"].shape[0]
    probe = min(16, N)
    _, d = oracle_layer_seconds(layer, alphas, gemm_m, G, probe)
    per_row = max(d["t_rows"] / probe, 1e-6)
    rows = int(max(probe, min(N, budget_s / per_row)))
    return rows, d["m"]


def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo), or None."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def oracle_single_thread(layer, s, G, budget_s=2.0):
    """The oracle's statistic and quantise-pack on one thread (BLAS limited to one thread; the
    numpy element-wise work is single-threaded anyway), on leading samples of the layer's X and
    W: GB/s of the algorithmic bytes (2 T K for the statistic; 2 N K + 4 K + packed bytes for
    the pack)."""
    import contextlib

    from oracle import awq_ref as ref
    try:
        from threadpoolctl import threadpool_limits
        one_thread = threadpool_limits(1)
    except Exception:  # noqa: BLE001
        one_thread = contextlib.nullcontext()
    with one_thread:
        X, W = layer["X"], layer["W"]
        K = X.shape[1]
        t_rows = max(1, min(X.shape[0], int(2 ** 22 // K)))
        t0 = time.perf_counter()
        ref.calib_stats(X[:t_rows])
        t_stats = time.perf_counter() - t0
        n_rows = max(1, min(W.shape[0], int(2 ** 20 // K)))
        t0 = time.perf_counter()
        ref.quantize_pack(W[:n_rows], s, G)
        t_pack = time.perf_counter() - t0
    pack_bytes = 2 * n_rows * K + 4 * K + n_rows * K // 2 + 3 * n_rows * (K // G)
    return {"threads": 1,
            "calib_stats_gbs": round(2 * t_rows * K / t_stats / 1e9, 4),
            "quantize_pack_gbs": round(pack_bytes / t_pack / 1e9, 4),
            "sample": f"statistic over the first {t_rows} tokens, pack of the first {n_rows} "
                      f"output rows (K={K})"}


def cpu_baseline(layer, alphas, gemm_m, G, budget_s=12.0):
    rows, m = choose_rows(layer, alphas, gemm_m, G, budget_s)
    sec, d = oracle_layer_seconds(layer, alphas, gemm_m, G, rows)
    N, K = layer["W"].shape
    T = layer["X"].shape[0]
    from oracle import awq_ref as ref
    s = ref.fl32(ref.scale_grid(m, [0.5]))[0].astype(np.float32)
    return {"value": 1.0 / sec, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"oracle (fp64 numpy) on {rows} of {N} output rows of the {N}x{K} layer "
                      f"with all T={T} calibration tokens and {len(alphas)} alphas plus the "
                      f"M={list(gemm_m)} matmuls; statistic over the full X; time extrapolated "
                      f"linearly in rows to the whole layer",
            "seconds_per_layer": sec, "sample_seconds": d["t_stats"] + d["t_rows"],
            "single_thread": oracle_single_thread(layer, s, G)}


def run_reference(args):
    """The oracle as the reference arm. Each step times the statistic over the whole X and the
    search, pack and matmuls of a bounded slice of output rows; ``ms_per_step`` is that measured
    time, and ``value`` the layers/s of the whole layer extrapolated linearly in rows from it
    (``extrapolated_ms_per_layer``), since one oracle layer takes minutes."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    wl, spec = layer_units(args.workload)
    layer = synth.make_layer(args.workload, 0)
    alphas = synth.alpha_grid(wl.n_alpha)
    G = wl.group_size
    total_steps = args.steps + args.warmup
    budget = max(1.0, min(8.0, 150.0 / max(total_steps, 1)))
    rows, _ = choose_rows(layer, alphas, wl.gemm_m, G, budget)
    step_s, layer_s = [], []
    for i in range(total_steps):
        t0 = time.perf_counter()
        sec, _ = oracle_layer_seconds(layer, alphas, wl.gemm_m, G, rows)
        if i >= args.warmup:
            step_s.append(time.perf_counter() - t0)
            layer_s.append(sec)
    mean_step = sum(step_s) / len(step_s)
    mean_layer = sum(layer_s) / len(layer_s)
    value = 1.0 / mean_layer
    sample = (f"each step: oracle (fp64 numpy) statistic over the full X, then the search of "
              f"{len(alphas)} alphas, the pack and the M={list(wl.gemm_m)} matmuls on {rows} of "
              f"{spec.n} output rows of the {spec.n}x{spec.k} layer with all T={spec.t} tokens; "
              f"ms_per_step is the measured step time, value the whole layer extrapolated "
              f"linearly in rows (extrapolated_ms_per_layer)")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_step * 1e3,
        "extrapolated_ms_per_layer": mean_layer * 1e3, "rows_per_step": rows,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "N": spec.n, "K": spec.k, "T": spec.t,
                   "group_size": G, "n_alpha": len(alphas), "gemm_m": list(wl.gemm_m)},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ GPU arm

class LayerStep:
    """Device buffers and the enqueue of one full layer step through the C ABI."""

    def __init__(self, awq, torch, layer, wl, dev):
        self.awq, self.torch = awq, torch
        W16, X16 = layer["W"], layer["X"]
        self.N, self.K = W16.shape
        self.T = X16.shape[0]
        self.G = wl.group_size
        self.alphas = synth.alpha_grid(wl.n_alpha)
        self.gemm_m = tuple(wl.gemm_m)
        self.W = torch.from_numpy(W16).to(dev)
        self.X = torch.from_numpy(X16).to(dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.m = torch.empty(self.K, **f32)
        self.err = torch.empty(len(self.alphas), **f32)
        self.best = torch.empty(1, dtype=torch.int32, device=dev)
        self.s = torch.empty(self.K, **f32)
        self.inv_s = torch.empty(self.K, **f32)
        self.ws_bytes = awq.awq_search_workspace_bytes(self.N, self.K, self.T, len(self.alphas),
                                                       self.G)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.q = torch.empty((self.N, self.K // 8), dtype=torch.int32, device=dev)
        self.sc = torch.empty((self.K // self.G, self.N), dtype=torch.float16, device=dev)
        self.z = torch.empty((self.K // self.G, self.N), dtype=torch.uint8, device=dev)
        self.ym = {M: torch.empty((M, self.N), dtype=torch.float16, device=dev)
                   for M in self.gemm_m}
        self.stream = torch.cuda.current_stream()

    def enqueue(self):
        a, st = self.awq, self.stream
        a.awq_calib_stats(self.X, self.T, self.K, self.K, self.m, st)
        a.awq_search_scale(self.W, self.N, self.K, self.X, self.T, self.m, self.alphas,
                           len(self.alphas), self.G, False, self.ws, self.ws_bytes, self.err,
                           self.best, self.s, self.inv_s, st)
        a.awq_quantize_pack(self.W, self.N, self.K, self.s, self.G, False, self.q, self.sc,
                            self.z, st)
        for M in self.gemm_m:
            # the first M calibration rows serve as the batch (a contiguous prefix of X)
            a.awq_w4a16_gemm(self.X, M, self.N, self.K, self.q, self.sc, self.z, self.inv_s,
                             self.G, False, self.ym[M], st)

    def outputs(self):
        return [self.err, self.best, self.s, self.inv_s, self.q, self.sc, self.z] + \
            [self.ym[M] for M in self.gemm_m]


def w4a16_kernel_name(M, K, G):
    """Which W4A16 kernel the library runs for M tokens and K input channels: the CUDA-core
    GEMV up to 4 tokens where its K parts fit its 15 consumer warps, the grouped tensor-core
    kernel up to 16 tokens (G >= 64), the dequant tensor-core kernel otherwise."""
    ipl = 4 if M == 1 else (2 if M == 2 else 1)
    if M <= 4 and -(-(K // 32) // (32 * ipl)) <= 15:
        return "gemv"
    return "grouped_tc" if M <= 16 and G >= 64 else "dequant_tc"


def w4a16_graph_time(awq, torch, N, K, G, M, sets, inv, reps_outer=3):
    """Per-launch time (us) of awq_w4a16_gemm at [M, K] x [N, K]^T, from a CUDA graph that walks
    rotating weight sets (more bytes than L2, so each launch streams its weights from HBM):
    events around whole graph replays, no host work inside the timed region."""
    X = torch.randn((M, K), device="cuda").half()
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for q, sc, z in sets:   # non-captured first launches (kernel attributes, module load)
        awq.awq_w4a16_gemm(X, M, N, K, q, sc, z, inv, G, False, Y)
    awq.awq_stream_status()
    per_graph = max(len(sets), 24 // max(1, len(sets)) * len(sets))
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(per_graph):
                q, sc, z = sets[i % len(sets)]
                awq.awq_w4a16_gemm(X, M, N, K, q, sc, z, inv, G, False, Y, stream)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps_outer):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    awq.awq_stream_status()
    return e0.elapsed_time(e1) * 1e3 / (reps_outer * per_graph)


def w4a16_sweep(awq, torch, shapes, ms, G, peaks):
    """W4A16 throughput per (shape, M): HBM GB/s of the algorithmic bytes (packed weights +
    metadata + activations + outputs + inv_s) and TFLOP/s, each against the measured peaks.
    ``ms`` is one list of M for every shape, or a list of lists (one per shape)."""
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20)
    gen = torch.Generator(device="cuda").manual_seed(7)
    out = []
    per_shape = ms if ms and isinstance(ms[0], (list, tuple)) else [ms] * len(shapes)
    for (N, K), ms in zip(shapes, per_shape):
        packed = N * K // 2 + 3 * N * (K // G)
        copies = int(max(2, -(-2 * l2 // packed)))
        sets = [(torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), dtype=torch.int32,
                               device="cuda", generator=gen),
                 (torch.rand((K // G, N), device="cuda", generator=gen) * 0.01 + 1e-3).half(),
                 torch.randint(0, 16, (K // G, N), dtype=torch.uint8, device="cuda",
                               generator=gen))
                for _ in range(copies)]
        inv = torch.rand(K, device="cuda", generator=gen) + 0.5
        for M in ms:
            us = w4a16_graph_time(awq, torch, N, K, G, M, sets, inv)
            byts = packed + 2 * M * K + 2 * M * N + 4 * K
            gbs = byts / (us * 1e-6) / 1e9
            tfl = 2 * M * N * K / (us * 1e-6) / 1e12
            out.append({"N": N, "K": K, "M": M,
                        "kernel": w4a16_kernel_name(M, K, G),
                        "us": round(us, 3), "GB/s": round(gbs, 1),
                        "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                        "TFLOP/s": round(tfl, 2),
                        "frac_tensor": round(tfl / peaks["bf16_tflops"], 4),
                        "weight_sets": copies, "timing": "CUDA graph replay, L2-cold weights"})
        del sets
        torch.cuda.empty_cache()
    return out


def stack_shapes(fuse_shared_input=False):
    """(N, K) of each launch of one decode step through the 7B stack: its 224 linears, or with
    the linears that read the same input concatenated along N (q/k/v as one 12288 x 4096
    matrix, gate/up as one 22016 x 4096), as serving stacks store them: 128 launches over the
    same weights."""
    wl = synth.WORKLOADS["llama7b-stack"]
    if not fuse_shared_input:
        return [(spec.n, spec.k) for spec in wl.layers]
    out = []
    for i in range(0, len(wl.layers), 7):
        q, k, v, o, gate, up, down = wl.layers[i:i + 7]
        out += [(q.n + k.n + v.n, q.k), (o.n, o.k), (gate.n + up.n, gate.k), (down.n, down.k)]
    return out


def stack_decode(awq, torch, peaks, G=128, ms=(1,), reps=5, fuse_shared_input=False):
    """Decode steps (M tokens) through all 224 linears of the synthetic 7B stack (see
    stack_shapes), each step captured in one CUDA graph: weight bytes streamed per step against
    the HBM peak, one entry per M. The packed weights are drawn once (3.4 GB at G = 128, more
    than L2 many times over)."""
    shapes = stack_shapes(fuse_shared_input)
    gen = torch.Generator(device="cuda").manual_seed(11)
    weights = []
    for N, K in shapes:
        weights.append((N, K,
                        torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), dtype=torch.int32,
                                      device="cuda", generator=gen),
                        (torch.rand((K // G, N), device="cuda", generator=gen) * 0.01 + 1e-3).half(),
                        torch.randint(0, 16, (K // G, N), dtype=torch.uint8, device="cuda",
                                      generator=gen),
                        torch.rand(K, device="cuda", generator=gen) + 0.5))
    out = []
    for M in ms:
        layers = []
        total = 0
        for N, K, q, sc, z, inv in weights:
            layers.append((N, K, q, sc, z, torch.randn((M, K), device="cuda", generator=gen).half(),
                           torch.empty((M, N), dtype=torch.float16, device="cuda"), inv))
            total += N * K // 2 + 3 * N * (K // G) + 2 * M * K + 2 * M * N + 4 * K
        for N, K, q, sc, z, X, Y, inv in layers[:7]:
            awq.awq_w4a16_gemm(X, M, N, K, q, sc, z, inv, G, False, Y)
        awq.awq_stream_status()
        stream = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for N, K, q, sc, z, X, Y, inv in layers:
                    awq.awq_w4a16_gemm(X, M, N, K, q, sc, z, inv, G, False, Y, stream)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        awq.awq_stream_status()
        t_ms = e0.elapsed_time(e1) / reps
        gbs = total / (t_ms * 1e-3) / 1e9
        out.append({"linears": 224, "launches": len(shapes), "M": M, "group_size": G,
                    "ms_per_token_step": round(t_ms, 4),
                    "tokens_per_s": round(M / (t_ms * 1e-3), 1), "bytes_per_step": total,
                    "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                    "roofline_ms": round(total / (peaks["hbm_gbs"] * 1e9) * 1e3, 4)})
        del graph, layers
    del weights
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------------ larger workloads
#
# The search at the other workloads' shapes (Llama-7B MLP, Llama-70B MLP, the 224-linear 7B-like
# stack) and the W4A16 sweeps at their batch sizes. Inputs are drawn on the GPU by the same recipe
# as synth.py (normal weights of the workload's sigma, normal activations with its outlier
# channels, the gated down-projection input where the workload has one), seeded, so that
# full-size layers need no host generation; the oracle comparisons at these shapes are in the
# GPU tests, on synth.py's host draws.

def gpu_layer(torch, spec, seed, gate=None):
    """W [n, k] and X [t, k] fp16 on the device for one LayerSpec. ``gate`` = (X, W_gate, W_up)
    of the block gives the gated down-projection input fp16(silu(X W_gate^T) * (X W_up^T))."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    W = (torch.randn((spec.n, spec.k), device="cuda", generator=g) * spec.sigma).half()
    if gate is not None:
        Xg, Wg, Wu = gate
        xf = Xg.float()
        h = torch.nn.functional.silu(xf @ Wg.float().T) * (xf @ Wu.float().T)
        return W, h.half()
    X = torch.randn((spec.t, spec.k), device="cuda", generator=g)
    n_out = synth._n_outliers(spec)
    if n_out:
        idx = torch.randperm(spec.k, device="cuda", generator=g)[:n_out]
        if spec.outlier_student_t:
            torch.manual_seed(seed)
            st = torch.distributions.StudentT(torch.tensor(3.0, device="cuda"))
            X[:, idx] = st.sample((spec.t, n_out)) * spec.outlier_mult
        else:
            X[:, idx] *= spec.outlier_mult
    return W, X.half()


class SearchBuffers:
    """Outputs and workspace of the per-layer step (statistic, search, pack) for one shape."""

    def __init__(self, awq, torch, N, K, T, n_alpha, G, sym):
        f32 = dict(dtype=torch.float32, device="cuda")
        self.m = torch.empty(K, **f32)
        self.err = torch.empty(n_alpha, **f32)
        self.best = torch.empty(1, dtype=torch.int32, device="cuda")
        self.s = torch.empty(K, **f32)
        self.inv = torch.empty(K, **f32)
        self.ws_bytes = awq.awq_search_workspace_bytes(N, K, T, n_alpha, G, sym)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.q = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
        self.sc = torch.empty((K // G, N), dtype=torch.float16, device="cuda")
        self.z = torch.empty((K // G, N), dtype=torch.uint8, device="cuda")

    def outputs(self):
        return [self.err, self.best, self.s, self.q, self.sc, self.z]


def enqueue_layer(awq, W, X, alphas, G, sym, b, stream=None):
    """Statistic, search and pack of one layer through the C ABI."""
    N, K = W.shape
    T = X.shape[0]
    awq.awq_calib_stats(X, T, K, K, b.m, stream)
    awq.awq_search_scale(W, N, K, X, T, b.m, alphas, len(alphas), G, sym, b.ws, b.ws_bytes,
                         b.err, b.best, b.s, b.inv, stream)
    awq.awq_quantize_pack(W, N, K, b.s, G, sym, b.q, b.sc, b.z, stream)


def search_flops(N, K, T, n_alpha, sched):
    """Flops of the search's scoring per layer: the direct form's n 2 T N K (the forward pass
    per grid point), and what the schedule that ran computes (Gram: H's triangle once and
    N K (K + 3) per candidate)."""
    direct = n_alpha * 2 * T * N * K
    if sched == "gram":
        return direct, T * K * (K + 1) + n_alpha * N * K * (K + 3)
    return direct, direct


def schedule_of(prof):
    return "gram" if ("gram_search" in prof or "score_gram" in prof) else "direct"


def search_workloads(awq, torch, peaks, reps=3):
    """Statistic + search + pack of the Llama-7B MLP (T = 8192) and Llama-70B MLP (T = 4096)
    layers at full size: ms per layer (mean of ``reps`` after one warm-up, L2 flushed between
    repetitions), layers/s, the schedule AUTO took and the search's roofline: the direct form's
    flops at the measured bf16 peak against the measured time, and the dominant scoring kernel's
    achieved TFLOP/s."""
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")
    out = []
    for wl_name in ("llama7b-mlp", "llama70b-mlp"):
        wl = synth.WORKLOADS[wl_name]
        alphas = synth.alpha_grid(wl.n_alpha)
        G = wl.group_size
        gate = None
        for li, spec in enumerate(wl.layers):
            if wl_name == "llama7b-mlp" and spec.name == "up_proj":
                continue                      # same shape as gate_proj
            if spec.gated:
                W, X = gpu_layer(torch, spec, 1000 * wl.wid + li, gate=gate)
            else:
                W, X = gpu_layer(torch, spec, 1000 * wl.wid + li)
            if wl_name == "llama7b-mlp" and spec.name == "gate_proj":
                Wu, _ = gpu_layer(torch, wl.layers[1], 1000 * wl.wid + 1)
                gate = (X, W, Wu)
            N, K = W.shape
            T = X.shape[0]
            b = SearchBuffers(awq, torch, N, K, T, len(alphas), G, False)
            enqueue_layer(awq, W, X, alphas, G, False, b)
            awq.awq_stream_status()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            awq.awq_profile_begin()
            for i in range(reps):
                flush.zero_()
                ev[i][0].record()
                enqueue_layer(awq, W, X, alphas, G, False, b)
                ev[i][1].record()
            torch.cuda.synchronize()
            prof = awq.awq_profile_end()
            awq.awq_stream_status()
            ms = sum(a.elapsed_time(c) for a, c in ev) / reps
            sched = schedule_of(prof)
            direct, run_flops = search_flops(N, K, T, len(alphas), sched)
            key = "gram_search" if sched == "gram" else "score"
            n_k, ms_k = prof.get(key, (0, 0.0))
            kern_tflops = None
            if n_k:
                per = ms_k / n_k * 1e-3
                kern_tflops = (run_flops if sched == "gram" else run_flops / len(alphas)) / per / 1e12
            roof_s = direct / (peaks["bf16_tflops"] * 1e12)
            out.append({
                "workload": wl_name, "layer": spec.name, "N": N, "K": K, "T": T, "schedule": sched,
                "ms": round(ms, 3), "layers_per_s": round(1e3 / ms, 2),
                "direct_form_tflop": round(direct / 1e12, 3),
                "roofline_ms": round(roof_s * 1e3, 3), "frac_of_roofline": round(roof_s * 1e3 / ms, 4),
                "scoring_kernel": key, "scoring_kernel_tflops": round(kern_tflops, 1) if kern_tflops else None,
                "scoring_kernel_frac": round(kern_tflops / peaks["bf16_tflops"], 4) if kern_tflops else None,
                "kernels_ms": {k: round(v[1] / reps, 3) for k, v in prof.items()},
                "timing": f"statistic + search + pack, mean of {reps} after a warm-up, L2 flushed"})
            del b, W, X
            torch.cuda.empty_cache()
        gate = None
    return out


# fp32 lane operations one clip-ratio evaluation of one weight needs at the least: the code
# (one fma into the rounding domain, clamp low, clamp high, remove the offset), the dequantised
# value (times the step, times 1/s), the difference, and the energy-weighted square (mul, fma)
CLIP_OPS_PER_EVAL = 9


def clip_timing(awq, torch, step, ratios, reps=10):
    """Per-group clipping on the benchmark layer after its scale search: the channel energy
    (a calib_stats launch), the ratio search and the clipped pack, timed per kernel over reps
    passes with L2 flushed before each. The search kernel is bound by fp32 issue: its peak is
    the SM count x 128 fp32 lanes x the SM clock, in lane operations per second."""
    a, st = awq, step.stream
    dev = step.W.device
    n_r = len(ratios)
    energy = torch.empty(step.K, dtype=torch.float32, device=dev)
    clip = torch.empty((step.K // step.G, step.N), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)

    def once():
        a.awq_clip_search(step.W, step.N, step.K, step.X, step.T, step.s, ratios, n_r, step.G,
                          False, energy, clip, st)
        a.awq_quantize_pack_clip(step.W, step.N, step.K, step.s, clip, step.G, False, step.q,
                                 step.sc, step.z, st)

    for _ in range(3):
        once()
    a.awq_stream_status()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    torch.cuda.synchronize()
    a.awq_profile_begin()
    for e0, e1 in ev:
        flush.zero_()
        e0.record()
        once()
        e1.record()
    torch.cuda.synchronize()
    prof = a.awq_profile_end()
    a.awq_stream_status()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / reps
    per = {k: round(v[1] * 1e3 / v[0], 3) for k, v in prof.items()}
    evals = step.N * step.K * n_r
    props = torch.cuda.get_device_properties(dev)
    peak = props.multi_processor_count * 128 * 2032e6
    us = per.get("clip_search")
    achieved = evals * CLIP_OPS_PER_EVAL / (us * 1e-6) if us else None
    return {
        "layer": f"{step.N}x{step.K}, T={step.T}, G={step.G}, asymmetric, searched scale",
        "n_ratio": n_r, "ms_per_layer": round(ms, 4), "kernels_us": per,
        "roofline": {"bound": "alu", "kernel": "clip_search_kernel",
                     "achieved": round(achieved / 1e12, 2) if achieved else None,
                     "peak": round(peak / 1e12, 2), "unit": "T fp32 lane-ops/s",
                     "frac": round(achieved / peak, 4) if achieved else None,
                     "ops_per_eval": CLIP_OPS_PER_EVAL, "evals_per_launch": evals},
        "timing": "energy + ratio search + clipped pack per pass, CUDA events, L2 flushed "
                  "(256 MB write) before each pass",
    }


def stack_layers(torch):
    """The 224 linears of the synthetic 7B-like stack on the device (W and its calibration X;
    the down-projections take the gated input of their block's gate and up projections)."""
    wl = synth.WORKLOADS["llama7b-stack"]
    layers = []
    block = {}
    for li, spec in enumerate(wl.layers):
        if spec.gated:
            W, X = gpu_layer(torch, spec, 1000 * wl.wid + li, gate=(block["gate"][1], block["gate"][0],
                                                                       block["up"][0]))
        else:
            W, X = gpu_layer(torch, spec, 1000 * wl.wid + li)
        kind = spec.name.split(".")[1]
        block[kind] = (W, X)
        if kind == "down":
            block = {}
        layers.append((spec, W, X))
    return wl, layers


def stack_search(awq, torch, peaks, variants=((128, False), (64, False), (128, True)), reps=1):
    """AWQ over all 224 linears of the stack (statistic + search + pack per layer, one layer
    after another on one stream, inputs resident): seconds per stack for each (group size,
    symmetric) variant, layers/s overall and per shape, against the roofline of the direct-form
    search flops at the measured bf16 peak."""
    wl, layers = stack_layers(torch)
    alphas = synth.alpha_grid(wl.n_alpha)
    out = {"linears": len(layers), "T": layers[0][0].t, "variants": []}
    direct_total = sum(search_flops(W.shape[0], W.shape[1], X.shape[0], len(alphas), "direct")[0]
                       for _, W, X in layers)
    for G, sym in variants:
        bufs = {}
        for _, W, X in layers:
            key = (W.shape[0], W.shape[1])
            if key not in bufs:
                bufs[key] = SearchBuffers(awq, torch, W.shape[0], W.shape[1], X.shape[0],
                                          len(alphas), G, sym)
        for _, W, X in layers:                                   # warm-up pass
            enqueue_layer(awq, W, X, alphas, G, sym, bufs[(W.shape[0], W.shape[1])])
        awq.awq_stream_status()
        per_shape = {}
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in layers]
        awq.awq_profile_begin()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(reps):
            e0.record()
            for i, (_, W, X) in enumerate(layers):
                ev[i][0].record()
                enqueue_layer(awq, W, X, alphas, G, sym, bufs[(W.shape[0], W.shape[1])])
                ev[i][1].record()
            e1.record()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
            for i, (_, W, _x) in enumerate(layers):
                per_shape.setdefault(f"{W.shape[0]}x{W.shape[1]}", []).append(ev[i][0].elapsed_time(ev[i][1]))
        prof = awq.awq_profile_end()
        awq.awq_stream_status()
        sec = tot / reps / 1e3
        roof = direct_total / (peaks["bf16_tflops"] * 1e12)
        sched = schedule_of(prof)
        n_k, ms_k = prof.get("score", (0, 0.0))
        score_flops = sum(search_flops(W.shape[0], W.shape[1], X.shape[0], len(alphas), "direct")[0]
                          for _, W, X in layers) * reps
        out["variants"].append({
            "group_size": G, "symmetric": sym, "seconds_per_stack": round(sec, 4),
            "layers_per_s": round(len(layers) / sec, 1), "schedule": sched,
            "roofline_s": round(roof, 4), "frac_of_roofline": round(roof / sec, 4),
            "per_shape_ms": {k: round(sum(v) / len(v), 3) for k, v in per_shape.items()},
            "scoring_kernel_tflops": round(score_flops / (ms_k * 1e-3) / 1e12, 1) if n_k else None,
            "kernels_ms": {k: round(v[1] / reps, 2) for k, v in prof.items()}})
        del bufs
        torch.cuda.empty_cache()
    out["direct_form_tflop"] = round(direct_total / 1e12, 1)
    out["timing"] = ("one pass over all linears after a warm-up pass, layers one after another "
                     "on one stream, inputs resident in HBM (13 GB of weights, 4.7 GB of "
                     "calibration activations)")
    return out, wl, layers


def stack_search_e2e(awq, torch, layers, alphas, G=128):
    """The stack pass through the C ABI from pinned host buffers: every layer's W and X are
    uploaded and its results (errors, alpha index, scales, packed codes, steps, zero points)
    read back inside the timed region. Two device buffer sets per shape alternate, with the
    copies on their own streams (one per direction), as a layer-by-layer pipeline would run.
    The host side holds one pinned W and X per shape (their values do not change the time)."""
    host = {}
    for _, W, X in layers:
        key = (W.shape[0], W.shape[1])
        if key not in host:
            host[key] = (W.cpu().pin_memory(), X.cpu().pin_memory())
    dev = {}
    for key, (Wh, Xh) in host.items():
        dev[key] = [(torch.empty_like(Wh, device="cuda"), torch.empty_like(Xh, device="cuda"),
                     SearchBuffers(awq, torch, key[0], key[1], Xh.shape[0], len(alphas), G, False))
                    for _ in range(2)]
    outs = {key: [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in d[2].outputs()]
                  for d in dv] for key, dv in dev.items()}
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    state = {key: {"uploaded": [torch.cuda.Event(), torch.cuda.Event()],
                   "computed": [torch.cuda.Event(), torch.cuda.Event()],
                   "read": [torch.cuda.Event(), torch.cuda.Event()], "used": [False, False],
                   "next": 0} for key in dev}
    h2d = d2h = 0

    def one(key):
        nonlocal h2d, d2h
        st = state[key]
        k = st["next"]
        st["next"] ^= 1
        Wd, Xd, b = dev[key][k]
        Wh, Xh = host[key]
        with torch.cuda.stream(up):
            if st["used"][k]:
                up.wait_event(st["computed"][k])
            Wd.copy_(Wh, non_blocking=True)
            Xd.copy_(Xh, non_blocking=True)
            st["uploaded"][k].record(up)
        comp.wait_event(st["uploaded"][k])
        if st["used"][k]:
            comp.wait_event(st["read"][k])
        enqueue_layer(awq, Wd, Xd, alphas, G, False, b)
        st["computed"][k].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(st["computed"][k])
            for hbuf, o in zip(outs[key][k], b.outputs()):
                hbuf.copy_(o, non_blocking=True)
            st["read"][k].record(down)
        st["used"][k] = True
        h2d += Wh.numel() * 2 + Xh.numel() * 2
        d2h += sum(o.numel() * o.element_size() for o in b.outputs())

    for _, W, _x in layers[:14]:                                   # warm-up
        one((W.shape[0], W.shape[1]))
    torch.cuda.synchronize()
    h2d = d2h = 0
    t0 = time.perf_counter()
    for _, W, _x in layers:
        one((W.shape[0], W.shape[1]))
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    awq.awq_stream_status()
    return {"value": round(len(layers) / dt, 1), "unit": "layers/s", "seconds_per_stack": round(dt, 4),
            "h2d_bytes_per_stack": h2d, "d2h_bytes_per_stack": d2h, "group_size": G,
            "pipelining": "two buffer sets per shape; H2D and D2H on their own streams overlap "
                          "compute; one pinned host W and X per shape"}


def stack_cpu_baseline(G=128, budget_s=4.0):
    """The oracle (statistic, search, pack) on a bounded row slice of one layer of each of the
    stack's three shapes (host draws, T = 2048), extrapolated linearly in rows and by the shape
    counts to the 224 linears."""
    wl = synth.WORKLOADS["llama7b-stack"]
    alphas = synth.alpha_grid(wl.n_alpha)
    counts = {}
    first = {}
    for li, spec in enumerate(wl.layers):
        key = (spec.n, spec.k)
        counts[key] = counts.get(key, 0) + 1
        first.setdefault(key, li)
    total = 0.0
    detail = {}
    sample = 0.0
    for key, li in first.items():
        layer = synth.make_layer("llama7b-stack", li)
        rows, m = choose_rows(layer, alphas, (), G, budget_s)
        sec, d = oracle_layer_seconds(layer, alphas, (), G, rows)
        total += sec * counts[key]
        sample += d["t_stats"] + d["t_rows"]
        detail[f"{key[0]}x{key[1]}"] = {"rows": rows, "seconds_per_layer": round(sec, 2),
                                        "layers": counts[key]}
    return {"value": round(len(wl.layers) / total, 5), "unit": "layers/s",
            "seconds_per_stack": round(total, 1), "cores": blas_threads(), "kind": "oracle",
            "cpu_model": cpu_model(), "per_shape": detail, "sample_seconds": round(sample, 1),
            "sample": "oracle (fp64 numpy) statistic, 20-alpha search and pack on a row slice of "
                      "the first layer of each shape of the stack (all T=2048 tokens), time "
                      "extrapolated linearly in rows and by the number of layers of each shape"}


def run_ours(args):
    import torch

    from post_weight_quantization_stats_b300 import awq

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    awq.lib()
    peaks = measured_peaks()
    wl, spec = layer_units(args.workload)
    layer = layer_for_rank(args.workload, rank)
    dev = torch.device("cuda", local_rank)
    step = LayerStep(awq, torch, layer, wl, dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)

    for _ in range(max(args.warmup, 0)):
        step.enqueue()
    awq.awq_stream_status()

    props = torch.cuda.get_device_properties(local_rank)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:" \
              f"{getattr(props, 'pci_device_id', 0):02X}.0"
    clocks = clock_sampler(bus)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    launches0 = awq.awq_launch_count()
    awq.awq_profile_begin()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record()
        step.enqueue()
        ev[i][1].record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    prof = awq.awq_profile_end()
    barrier(world)
    launches = awq.awq_launch_count() - launches0
    clk = clocks.stop()
    awq.awq_stream_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * args.steps / (total_ms / 1e3)

    alg = algorithmic(spec, step.G, len(step.alphas), step.gemm_m)
    kern = {}
    for name, (n, ms_tot) in prof.items():
        avg_us = ms_tot * 1e3 / n
        row = {"launches": n, "avg_us": round(avg_us, 3), "share": None}
        if name in alg and "bytes" in alg[name]:
            per = avg_us * alg[name].get("launches", 1)
            row["GB/s"] = round(alg[name]["bytes"] / (per * 1e-6) / 1e9, 1)
        if name in alg and "flops" in alg[name]:
            row["TFLOP/s"] = round(alg[name]["flops"] / (avg_us * 1e-6) / 1e12, 1)
        kern[name] = row
    tot_kernel_ms = sum(ms for _, ms in prof.values())
    for name, (n, ms_tot) in prof.items():
        kern[name]["share"] = round(ms_tot / tot_kernel_ms, 4) if tot_kernel_ms else None
    rooflines = kernel_rooflines(prof, alg, peaks, args.workload == WORKLOAD)
    dominant = max(rooflines, key=lambda name: prof[name][1]) if rooflines else None
    roofline = rooflines.pop(dominant) if dominant else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": args.workload, "N": step.N, "K": step.K, "T": step.T,
                   "group_size": step.G, "n_alpha": len(step.alphas),
                   "gemm_m": list(step.gemm_m), "l2": "flushed between steps (256 MB write)",
                   "parallelism": f"replicas x{world}: one independent layer per GPU"},
        "roofline": roofline,
        "roofline_other": rooflines,
        "gpu_launches": launches,
        "kernels": kern,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 4),
    }
    if rank == 0 and not args.no_hbm_sweep:
        # every workload's shapes at its own batch sizes: the benchmark layer (4096^2), the
        # Llama-7B MLP (4096 <-> 11008) and the Llama-70B MLP (8192 <-> 28672)
        m7 = sorted(set(step.gemm_m) | {1, 1024})
        m_mlp = list(synth.WORKLOADS["llama7b-mlp"].gemm_m)
        m70 = sorted(set(synth.WORKLOADS["llama70b-mlp"].gemm_m) | {2, 4, 16, 128})
        shapes = [(step.N, step.K), (11008, 4096), (4096, 11008), (28672, 8192), (8192, 28672)]
        line["w4a16"] = w4a16_sweep(awq, torch, shapes, [m7, m_mlp, m_mlp, m70, m70], step.G, peaks)
        dec = [r for r in line["w4a16"] if r["M"] == 1 and r["N"] == 28672]
        dec_down = [r for r in line["w4a16"] if r["M"] == 1 and r["N"] == 8192 and r["K"] == 28672]
        pre = [r for r in line["w4a16"] if r["M"] == 1024 and r["N"] == 28672]
        gemv_src = ("w4a16_gemv.cuh",)
        if dec:
            line["roofline_w4a16_decode"] = {
                "bound": "hbm", "kernel": dec[0]["kernel"], "shape": "M=1, 8192 -> 28672",
                "achieved": dec[0]["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec[0]["frac_hbm"],
                "traffic": profiled_traffic("w4a16_gemv_llama70b_up_m1.md", gemv_src)}
        if dec_down:
            line["roofline_w4a16_decode_down"] = {
                "bound": "hbm", "kernel": dec_down[0]["kernel"], "shape": "M=1, 28672 -> 8192",
                "achieved": dec_down[0]["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec_down[0]["frac_hbm"],
                "traffic": profiled_traffic("w4a16_gemv_llama70b_down_m1.md", gemv_src)}
        if pre:
            line["roofline_w4a16_gemm"] = {
                "bound": "tensor", "kernel": pre[0]["kernel"], "shape": "M=1024, 8192 -> 28672",
                "achieved": pre[0]["TFLOP/s"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": pre[0]["frac_tensor"], "traffic": None}
        sd = stack_decode(awq, torch, peaks, G=128, ms=tuple(range(1, 65)), reps=3)
        line["w4a16_stack_decode"] = dict(sd[0], timing="one CUDA graph of all linears, "
                                                        "weights streamed from HBM")
        line["w4a16_stack_decode_sweep"] = [{k: r[k] for k in ("M", "ms_per_token_step",
                                                                "tokens_per_s", "frac_hbm")}
                                            for r in sd]
        sdf = stack_decode(awq, torch, peaks, G=128, ms=(1, 2, 4, 8, 16, 64), reps=3,
                           fuse_shared_input=True)
        line["w4a16_stack_decode_fused"] = [
            {k: r[k] for k in ("M", "launches", "ms_per_token_step", "tokens_per_s", "frac_hbm")}
            for r in sdf]
        sd64 = stack_decode(awq, torch, peaks, G=64, ms=(1, 8, 64), reps=3)
        line["w4a16_stack_decode_g64"] = [{k: r[k] for k in ("M", "ms_per_token_step",
                                                              "tokens_per_s", "frac_hbm")}
                                          for r in sd64]
    if rank == 0 and args.workload == WORKLOAD:
        line["clip"] = clip_timing(awq, torch, step, synth.clip_ratios(10))
    if rank == 0 and not args.no_workloads:
        line["search_layers"] = search_workloads(awq, torch, peaks)
        stack, swl, slayers = stack_search(awq, torch, peaks)
        if not args.no_e2e:
            stack["e2e"] = stack_search_e2e(awq, torch, slayers, synth.alpha_grid(swl.n_alpha))
        del slayers
        torch.cuda.empty_cache()
        if world == 1 and not args.no_cpu_baseline:
            stack["cpu_baseline"] = stack_cpu_baseline()
        line["stack_search"] = stack
    if not args.no_e2e:
        line["e2e"] = e2e_run(awq, torch, step, layer, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(layer, step.alphas, step.gemm_m, step.G)
        line["cpu_baseline"].pop("seconds_per_layer", None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# kernel name -> (kernel description, bound, committed ncu summary or None, source files)
ROOFLINE_KERNELS = {
    "gram_search": ("search_kernel: one persistent cooperative launch, tcgen05 kind::f16 X^T X "
                    "triangle then D B^T over the triangle per alpha, next residual built in "
                    "extra warps", "tensor", "gram_search_llama7b_attn_4096.md",
                    ("gram_persistent.cuh", "gram_score.cuh", "quant.cuh")),
    "score_gram": ("tri_kernel<SCORE>: tcgen05 kind::f16 D B^T over the triangle, fp32 "
                   "accumulate, d . (D B^T) epilogue", "tensor", None,
                   ("gram_score.cuh", "quant.cuh")),
    "gram": ("tri_kernel<GRAM>: tcgen05 kind::f16 lower triangle of X^T X", "tensor", None,
             ("gram_score.cuh", "quant.cuh")),
    "score": ("score_kernel: tcgen05 kind::f16 X D^T, fp32 accumulate, sum of squares", "tensor",
              None, ("score_gemm.cuh",)),
    "residual": ("residual_kernel: W - Q(W diag s) diag(s)^-1 as fp16", "hbm", None,
                 ("quant.cuh",)),
}


def kernel_rooflines(prof, alg, peaks, bench_workload):
    """Roofline objects of the search kernels that ran: algorithmic work per launch over the
    launch's average event-timed duration, against the measured peak of its bound."""
    out = {}
    for name, (desc, bound, md, src) in ROOFLINE_KERNELS.items():
        n, ms_tot = prof.get(name, (0, 0.0))
        if not n:
            continue
        avg_s = ms_tot / 1e3 / n
        if bound == "tensor":
            work = alg[name]["flops"]
            achieved, peak, unit = work / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
            note = (f"{peaks['source']} dense bf16 burst (fp16 runs at the bf16 rate); "
                    f"sustained {peaks['bf16_tflops_sustained']}")
        else:
            work = alg[name]["bytes"]
            achieved, peak, unit = work / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
            note = f"{peaks['source']} HBM copy bandwidth"
        out[name] = {"bound": bound, "kernel": desc, "achieved": round(achieved, 1),
                     "peak": peak, "unit": unit, "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(md, src) if bench_workload else None,
                     "peak_note": note, "avg_us": round(avg_s * 1e6, 3),
                     ("flops_per_launch" if bound == "tensor" else "bytes_per_launch"): work}
    return out


def e2e_run(awq, torch, step, layer, args, world):
    """The same step through the public API from pinned host buffers, every step's H2D of W and
    X and D2H of every result inside the timed region. Two sets of device buffers alternate and
    the copies run on their own streams (one per direction), so the upload of step i+1 and the
    download of step i-1 overlap the computation of step i, as a layer-by-layer quantisation
    pipeline would run; each buffer set is reused only after its previous step's results have
    been read back."""
    W_h = torch.from_numpy(layer["W"]).pin_memory()
    X_h = torch.from_numpy(layer["X"]).pin_memory()
    wl, _ = layer_units(args.workload)
    bufs = [step, LayerStep(awq, torch, layer, wl, step.W.device)]
    hosts = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in b.outputs()] for b in bufs]
    h2d = W_h.numel() * 2 + X_h.numel() * 2
    d2h = sum(o.numel() * o.element_size() for o in step.outputs())
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded = [ev(), ev()]
    computed = [ev(), ev()]
    read_back = [ev(), ev()]
    used = [False, False]

    def one(i):
        k = i % 2
        b = bufs[k]
        with torch.cuda.stream(up):
            if used[k]:
                up.wait_event(computed[k])          # the step before last has read W and X
            b.W.copy_(W_h, non_blocking=True)
            b.X.copy_(X_h, non_blocking=True)
            uploaded[k].record(up)
        comp.wait_event(uploaded[k])
        if used[k]:
            comp.wait_event(read_back[k])           # its results have been read back
        b.enqueue()
        computed[k].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[k])
            for h, o in zip(hosts[k], b.outputs()):
                h.copy_(o, non_blocking=True)
            read_back[k].record(down)
        used[k] = True

    for i in range(max(2, args.warmup)):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, world)
    return {"value": world * args.steps / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "pipelining": "two buffer sets; H2D and D2H on their own streams overlap compute"}


def run_case(args):
    """One kernel family on a small case, for profiler captures (no timing, no JSON line)."""
    import torch

    from post_weight_quantization_stats_b300 import awq

    torch.cuda.set_device(0)
    awq.lib()
    if args.case == "search":
        wl, _ = layer_units(args.workload)
        step = LayerStep(awq, torch, synth.make_layer(args.workload, 0), wl, torch.device("cuda", 0))
        for _ in range(3):
            step.enqueue()
    elif args.case == "clip":
        wl, _ = layer_units(args.workload)
        step = LayerStep(awq, torch, synth.make_layer(args.workload, 0), wl, torch.device("cuda", 0))
        step.enqueue()
        clip_timing(awq, torch, step, synth.clip_ratios(10), reps=2)
    elif args.case.startswith("w4a16:"):
        N, K, M = (int(v) for v in args.case.split(":")[1:4])
        gen = torch.Generator(device="cuda").manual_seed(5)
        q = torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), dtype=torch.int32, device="cuda",
                          generator=gen)
        sc = (torch.rand((K // 128, N), device="cuda", generator=gen) * 0.01 + 1e-3).half()
        z = torch.randint(0, 16, (K // 128, N), dtype=torch.uint8, device="cuda", generator=gen)
        inv = torch.rand(K, device="cuda", generator=gen) + 0.5
        X = torch.randn((M, K), device="cuda", generator=gen).half()
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        for _ in range(4):
            awq.awq_w4a16_gemm(X, M, N, K, q, sc, z, inv, 128, False, Y)
    else:
        raise SystemExit(f"bench.py: unknown --case {args.case}")
    awq.awq_stream_status()
    print(f"case {args.case} ok")
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
