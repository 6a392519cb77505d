"""bit_weight_only_gb300 -- weight-only quantized decode GEMV for GB300 (sm_103a).

    y[M x N] = x[M x K] . dequant(W)^T,   M = 1..16

Packed low-bit weights (Q4_0, 4/8-bit scalar codebooks, PQ2_0 ternary,
AQLM 2x8) stream from HBM, are decoded in registers and accumulated in fp32
by hand-written CUDA kernels behind a small C ABI (``include/qgemv.h``).
``bit_weight_only_gb300.qgemv`` is the thin Python binding over that ABI; the
shared library is loaded on first use and a missing library is an error
(there is no CPU fallback).  ``bit_weight_only_gb300.inputs`` draws the
seeded synthetic workloads.
"""

__all__ = ["qgemv", "inputs"]
