"""Host-side logic of bench.py on the CPU: clock parsing, algorithmic byte/flop counts, the
per-rank layer assignment and max-over-ranks timing under a 2-rank gloo group, and the
reference (oracle) arm end to end on the small workload."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_summarize_clocks():
    rows = [["0", "1965", "2032", "900.1", "0x0", "Not Active", "Not Active", "Not Active", "Active"],
            ["0", "1980", "2032", "950.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
            ["0", "N/A", "2032", "950.0", "0x0", "Not Active", "Active", "Not Active", "Not Active"]]
    c = bench.summarize_clocks(rows)
    assert c["sm_mhz"] == pytest.approx(1972.5) and c["sm_max_mhz"] == 2032
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"] and c["samples"] == 3


def test_algorithmic_counts():
    wl, spec = bench.layer_units("llama7b-attn-4096")
    a = bench.algorithmic(spec, 128, 20, wl.gemm_m)
    assert a["score"]["flops"] == 2 * 8192 * 4096 * 4096
    assert a["packed_bytes"] == 4096 * 4096 // 2 + 3 * 4096 * 32
    assert a["calib_stats"]["bytes"] == 2 * 8192 * 4096 + 4 * 4096
    assert a["gemv"][1]["bytes"] == a["packed_bytes"] + 2 * 4096 + 2 * 4096 + 4 * 4096


def test_layer_for_rank_is_independent_and_deterministic():
    a0 = bench.layer_for_rank("tiny-512", 0)
    a1 = bench.layer_for_rank("tiny-512", 1)
    b1 = bench.layer_for_rank("tiny-512", 1)
    assert a0["W"].shape == a1["W"].shape
    assert not np.array_equal(a0["W"], a1["W"])
    assert np.array_equal(a1["W"], b1["W"]) and np.array_equal(a1["X"], b1["X"])


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    m = bench.max_over_ranks(float(rank + 1) * 1.5, world)
    r, lr, w = bench.dist_env()
    out.put((rank, m, r, lr, w))
    dist.destroy_process_group()


def test_two_rank_timing_reduction_gloo():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.0, 3.0]                 # max over ranks
    assert [(r[2], r[3], r[4]) for r in res] == [(0, 0, 2), (1, 1, 2)]


def test_reference_arm_emits_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny-512", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, check=True, timeout=600, cwd=ROOT)
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_profiled_traffic_follows_every_kernel_source(tmp_path, monkeypatch):
    """The roofline's `traffic` comes from a committed ncu summary only while the digest of all
    the kernel's source files matches the one recorded with the counters: changing any of them
    (not just the first) voids it."""
    csrc = tmp_path / "post_weight_quantization_stats_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cuh").write_text("kernel a\n")
    (csrc / "b.cuh").write_text("helpers b\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.source_digest(("a.cuh", "b.cuh"))
    (tmp_path / "profiles" / "k.md").write_text(
        f"source_sha256_16: {sha}\n\n| traffic_bytes_per_launch | 12345 |\n")
    assert bench.profiled_traffic("k.md", ("a.cuh", "b.cuh")) == 12345
    (csrc / "b.cuh").write_text("helpers b, changed\n")
    assert bench.profiled_traffic("k.md", ("a.cuh", "b.cuh")) is None
    assert bench.profiled_traffic("k.md", ("a.cuh", "missing.cuh")) is None


def test_stack_shapes_fused_keeps_the_weights():
    """The fused decode step concatenates q/k/v and gate/up along N: 4 launches per block
    instead of 7, over exactly the same weight elements, with each fused matrix reading one
    input (the same K)."""
    plain = bench.stack_shapes()
    fused = bench.stack_shapes(fuse_shared_input=True)
    assert len(plain) == 224 and len(fused) == 128
    assert sum(n * k for n, k in plain) == sum(n * k for n, k in fused)
    for b in range(32):
        q, k, v, o, gate, up, down = plain[7 * b:7 * b + 7]
        qkv, o2, gate_up, down2 = fused[4 * b:4 * b + 4]
        assert qkv == (q[0] + k[0] + v[0], q[1]) and q[1] == k[1] == v[1]
        assert gate_up == (gate[0] + up[0], gate[1]) and gate[1] == up[1]
        assert o2 == o and down2 == down


def test_clip_ratio_grid_matches_the_oracle():
    """The benchmark's clipping grid is the oracle's (1, 0.95, ..., 0.55)."""
    from oracle import awq_ref as ref
    from post_weight_quantization_stats_b300 import synth
    assert np.array_equal(synth.clip_ratios(10), ref.clip_ratio_grid(10))
    assert synth.clip_ratios(10)[0] == 1.0 and np.all(np.diff(synth.clip_ratios(10)) < 0)
