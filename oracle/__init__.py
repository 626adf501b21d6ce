"""Exact CPU reference (the oracle) for the order-invariant softmax reduction.

TEST INFRASTRUCTURE ONLY.  `oracle.exact` is the definition written out in exact rational
arithmetic (tiny shapes); `oracle.native` is an independent exact C implementation (whole
rows of the full-size workloads).  Only tests/, the smoke check and the benchmark's
CPU-baseline leg may import this package; the CUDA product path never does.
"""
