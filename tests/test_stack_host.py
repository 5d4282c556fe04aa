"""Host side of the resumable layer-stack run (stack.py): interruption, restart, truncated
manifest lines, missing result files. A numpy quantiser stands in for the GPU one."""

import json
import os

import numpy as np
import pytest

from post_weight_quantization_stats_b300 import stack


def _layers(n):
    def mk(i):
        rng = np.random.Generator(np.random.PCG64(i))
        return lambda: (rng.standard_normal((4, 8)), rng.standard_normal((3, 8)))
    return [(i, f"l{i}", mk(i)) for i in range(n)]


class Counting:
    def __init__(self):
        self.calls = 0

    def __call__(self, W, X):
        self.calls += 1
        err = np.abs((X @ W.T)).sum(axis=0)
        return {"best": int(np.argmin(err)), "err": err, "W": W}


class Stop(Exception):
    pass


def _stop_after(k):
    def f(index):
        if index == k:
            raise Stop()
    return f


def _contents(d, recs):
    return {i: {k: v.tolist() for k, v in stack.load_layer(d, r).items()} for i, r in recs.items()}


def test_interrupt_and_resume_matches_a_clean_run(tmp_path):
    clean = str(tmp_path / "clean")
    want = stack.quantize_layers(_layers(5), clean, Counting())
    d = str(tmp_path / "run")
    with pytest.raises(Stop):
        stack.quantize_layers(_layers(5), d, Counting(), on_layer=_stop_after(2))
    assert sorted(stack.read_manifest(d)) == [0, 1, 2]
    q = Counting()
    got = stack.quantize_layers(_layers(5), d, q)
    assert q.calls == 2                      # only layers 3 and 4 ran again
    assert sorted(got) == list(range(5))
    assert _contents(d, got) == _contents(clean, want)
    with open(os.path.join(d, stack.MANIFEST)) as f:
        assert [json.loads(l)["index"] for l in f] == [0, 1, 2, 3, 4]


def test_truncated_line_and_missing_file_rerun(tmp_path):
    d = str(tmp_path / "run")
    stack.quantize_layers(_layers(4), d, Counting())
    path = os.path.join(d, stack.MANIFEST)
    lines = open(path).read().splitlines()
    # layer 2's line cut short by a crash; layer 3's result file lost
    with open(path, "w") as f:
        f.write("\n".join(lines[:2] + [lines[2][:17]] + lines[3:]) + "\n")
    os.remove(os.path.join(d, json.loads(lines[3])["file"]))
    assert sorted(stack.read_manifest(d)) == [0, 1]
    q = Counting()
    got = stack.quantize_layers(_layers(4), d, q)
    assert q.calls == 2 and sorted(got) == [0, 1, 2, 3]
