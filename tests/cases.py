"""Canonical test inputs, drawn only from the seeded generators.

``make_case`` returns the canonical packed bytes, scales and codebooks of one
format as numpy arrays; both the CUDA path and the oracle are fed from them.
Q4_0 here uses random (valid) blocks; the end-to-end tests that start from
fp32 weights let each side run its own quantizer.
"""
from __future__ import annotations

import numpy as np

from bit_weight_only_gb300 import inputs

MIN_K = {"q4_0": 32, "cbk4": 2, "cbk8": 1, "pq2_0": 128, "aqlm_2x8": 8, "aqlm_1x16": 8, "cbk4_row": 2,
         "cbk8_row": 1}


def make_case(fmt: str, N: int, K: int, tag: str = "case", seed: int = 0):
    g = inputs.rng(f"{tag}/{fmt}/{N}x{K}", seed)
    if fmt == "q4_0":
        return inputs.q4_0_random_blocks(g, N, K), None, None
    if fmt in ("cbk4", "cbk8"):
        L = 16 if fmt == "cbk4" else 256
        cb = inputs.cbk_centroids(L)
        return inputs.cbk_packed(g, N, K, 4 if L == 16 else 8, inputs.cbk_cell_probs(cb)), None, cb
    if fmt == "pq2_0":
        return inputs.pq2_packed(g, N, K), None, None
    if fmt == "aqlm_2x8":
        return inputs.aqlm_inputs(g, N, K)
    if fmt == "aqlm_1x16":
        return inputs.aqlm_1x16_inputs(g, N, K)
    if fmt == "cbk8_row":  # codebooks fp32 [N, 256], one per output row
        cb = inputs.cbk_row_codebooks(g, N, L=256)
        return inputs.cbk_packed(g, N, K, 8, inputs.cbk_cell_probs(inputs.cbk_centroids(256))), None, cb
    if fmt == "cbk4_row":  # codebooks fp32 [N, 16], one per output row
        cb = inputs.cbk_row_codebooks(g, N)
        return inputs.cbk_packed(g, N, K, 4, inputs.cbk_cell_probs(inputs.cbk_centroids(16))), None, cb
    raise ValueError(fmt)


def make_x(M: int, K: int, tag: str = "x", seed: int = 0) -> np.ndarray:
    return inputs.x_fp16(inputs.rng(f"{tag}/{M}x{K}", seed), M, K)


def unpack_xq(xq, M: int, K: int):
    """(codes int8 [M, K] in input order, scales fp32 [M, K/128], code sums
    int32 [M, K/128]) of a prepared INT8 activation buffer (the layout
    include/qgemv.h gives for qgemv_prepare_x_int8)."""
    b = xq.cpu().numpy() if hasattr(xq, "cpu") else np.asarray(xq)
    G = K // 128
    codes = b[:M * K].view(np.int8).reshape(M, G, 128)
    e = np.arange(128)
    staged = 16 * (e >> 4) + 4 * (e & 3) + ((e >> 2) & 3)   # byte of input e within its group
    q = codes[:, :, staged].reshape(M, K)
    a = b[M * K:M * K + 4 * M * G].view(np.float32).reshape(M, G)
    s = b[M * K + 4 * M * G:M * K + 8 * M * G].view(np.int32).reshape(M, G)
    return q, a, s
