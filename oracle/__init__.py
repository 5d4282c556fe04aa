"""CPU oracle for the AWQ per-linear-layer step: test infrastructure, not product code.

Only the test suite, the package entry point's smoke check and the benchmark's CPU-baseline leg
may import this package. The CUDA path never calls it and shares no code with it.
"""
