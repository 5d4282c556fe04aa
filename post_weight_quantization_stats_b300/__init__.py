"""AWQ per-linear-layer step and W4A16 matmul on B300 (sm_103a).

The compute lives in ``libawq.so`` (hand-written CUDA behind a C ABI, ``include/awq.h``);
:mod:`post_weight_quantization_stats_b300.awq` is the thin ctypes binding with the same call
names. Importing this package loads nothing; the binding loads the library on first use and
raises if it is missing.
"""

__all__ = ["awq", "synth"]
