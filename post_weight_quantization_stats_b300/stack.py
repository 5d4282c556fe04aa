"""AWQ over a stack of linear layers, resumable after an interruption.

Every layer is independent given its calibration input ("AWQ Math", "Searching the scale": the
search is per layer and needs only that layer's input), so a long run (the 224 linears of a
7B-like stack) is a loop over layers whose results are written out one by one:

* each finished layer's results (alpha index, the alpha errors, s, the packed codes, fp16 steps
  and zero points) go to ``<out_dir>/<index>_<name>.npz``, written to a temporary name and
  renamed, so a file that exists is complete;
* then one JSON line ``{"index", "name", "file", "best", "err_best"}`` is appended to
  ``<out_dir>/manifest.jsonl`` and flushed to disk;
* a restart reads the manifest and skips every layer listed there whose file exists; a
  truncated last line (a crash while appending) is ignored and that layer runs again.

The default quantiser runs the library's statistic, search and pack on the GPU; any callable
with the same contract can stand in (the host-side tests use a numpy one).
"""

from __future__ import annotations

import json
import os

import numpy as np

MANIFEST = "manifest.jsonl"


def read_manifest(out_dir: str) -> dict:
    """{index: record} of the finished layers (complete lines whose file exists)."""
    path = os.path.join(out_dir, MANIFEST)
    done = {}
    if not os.path.exists(path):
        return done
    with open(path) as f:
        for line in f:
            try:
                rec = json.loads(line)
            except json.JSONDecodeError:
                continue                      # a line cut short by a crash
            if os.path.exists(os.path.join(out_dir, rec["file"])):
                done[int(rec["index"])] = rec
    return done


def gpu_quantizer(alphas, group_size=128, symmetric=False, bits=4):
    """Statistic, alpha search and pack of one layer through libawq (``bits``-wide codes);
    returns host arrays."""
    import torch

    from . import awq

    def run(W, X):
        m = awq.calib_stats(X)
        err, best, s, inv_s = awq.search_scale(W, X, alphas, group_size, symmetric, mean_abs=m,
                                               bits=bits)
        q, sc, z = awq.quantize_pack(W, s, group_size, symmetric, bits=bits)
        awq.awq_stream_status()
        torch.cuda.synchronize()
        return {"best": int(best.item()), "err": err.cpu().numpy(), "m": m.cpu().numpy(),
                "s": s.cpu().numpy(), "inv_s": inv_s.cpu().numpy(),
                "qweight": q.cpu().numpy().view(np.uint32), "scales": sc.cpu().numpy(),
                "zeros": z.cpu().numpy()}
    return run


def quantize_layers(layers, out_dir: str, quantizer, on_layer=None) -> dict:
    """Run ``quantizer(W, X)`` on every layer of ``layers`` (an iterable of
    ``(index, name, load)``, ``load()`` returning W and X) that the manifest in ``out_dir`` does
    not list yet, writing its results as described above. ``on_layer(index)`` is called after
    each layer is recorded. Returns the manifest records of all layers, finished before or now."""
    os.makedirs(out_dir, exist_ok=True)
    done = read_manifest(out_dir)
    path = os.path.join(out_dir, MANIFEST)
    for index, name, load in layers:
        if index in done:
            continue
        W, X = load()
        res = quantizer(W, X)
        fname = f"{index:04d}_{name}.npz"
        tmp = os.path.join(out_dir, fname + ".tmp.npz")
        np.savez(tmp, **res)
        os.replace(tmp, os.path.join(out_dir, fname))
        rec = {"index": int(index), "name": name, "file": fname, "best": int(res["best"]),
               "err_best": float(np.asarray(res["err"])[int(res["best"])])}
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
            f.flush()
            os.fsync(f.fileno())
        done[int(index)] = rec
        if on_layer is not None:
            on_layer(index)
    return done


def load_layer(out_dir: str, rec: dict) -> dict:
    """The arrays written for one manifest record."""
    with np.load(os.path.join(out_dir, rec["file"])) as z:
        return {k: z[k] for k in z.files}
