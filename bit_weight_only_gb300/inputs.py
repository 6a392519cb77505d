"""Seeded synthetic inputs for the quantized decode GEMV.

This module only draws random numbers with the distributions of the
workloads; it holds none of the method's arithmetic (no dequantization, no
quantizer, no dot products), so both the CUDA path and the CPU oracle may be
fed from it.  Host (numpy) generators serve tests of any size the host can
hold; the ``*_cuda`` variants draw the same distributions directly on a
device for the large benchmark stacks.

Distributions (per workload):
  x                    fp16 ~ N(0, 1), rounded to nearest even.
  Q4_0 weights         fp32 ~ N(0, 0.02), quantized afterwards by the caller.
  codebook (CBK4/8)    L fp16 centroids = N(0, sigma) mid-rank quantiles
                       sigma * Phi^-1((i + 1/2) / L), sorted; indices i.i.d.
                       with the Gaussian mass of each centroid's cell (cells
                       split at midpoints between neighbouring centroids).
  PQ2_0                2-bit fields i.i.d. with P(code 0, 1, 2, 3) =
                       (0.3, 0.4, 0.3, 0), i.e. ternary -1/0/+1 with
                       P(0) = 0.4; block scale fp16 |N(0, 0.02)|.
  AQLM 2x8             codes uniform uint8; two 256x8 codebooks fp16
                       ~ N(0, 0.01); per-row scale fp16 ~ U(0.5, 1.5).
Because every field inside a packed byte is drawn independently from the
same distribution, byte values are drawn from the product distribution of
their fields; the order of fields inside a byte does not change it.
"""
from __future__ import annotations

import zlib

import numpy as np
from scipy.special import ndtr, ndtri

PQ2_CODE_PROBS = (0.3, 0.4, 0.3, 0.0)


def rng(tag: str, seed: int = 0) -> np.random.Generator:
    """Independent PCG64 stream for one named tensor of one workload."""
    return np.random.Generator(
        np.random.PCG64(np.random.SeedSequence([seed, zlib.crc32(tag.encode())])))


def torch_seed(tag: str, seed: int = 0) -> int:
    """Seed for a torch.Generator drawing the tensor named ``tag``."""
    return (seed * 0x9E3779B1 + zlib.crc32(tag.encode())) & 0x7FFFFFFFFFFF


# ----------------------------------------------------------------- host ----

def x_fp16(g: np.random.Generator, M: int, K: int) -> np.ndarray:
    return g.standard_normal((M, K), dtype=np.float32).astype(np.float16)


def w_fp32(g: np.random.Generator, N: int, K: int, sigma: float = 0.02) -> np.ndarray:
    return (g.standard_normal((N, K), dtype=np.float32) * np.float32(sigma))


def q4_0_random_blocks(g: np.random.Generator, N: int, K: int,
                       sigma_d: float = 0.003) -> np.ndarray:
    """Canonical Q4_0 rows with uniformly random nibbles and a signed fp16
    scale ~ N(0, sigma_d): every byte pattern of a block is a valid block."""
    nb = K // 32
    blocks = np.empty((N, nb, 18), dtype=np.uint8)
    d = (g.standard_normal((N, nb), dtype=np.float32) * np.float32(sigma_d)).astype(np.float16)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = g.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    return blocks.reshape(N, nb * 18)


def cbk_centroids(L: int, sigma: float = 0.02) -> np.ndarray:
    """Sorted fp16 mid-rank quantiles of N(0, sigma); strictly increasing."""
    c = (sigma * ndtri((np.arange(L) + 0.5) / L)).astype(np.float16)
    if not np.all(np.diff(c.astype(np.float64)) > 0):
        raise ValueError("fp16 centroids are not strictly increasing")
    return c


def cbk_cell_probs(centroids: np.ndarray, sigma: float = 0.02) -> np.ndarray:
    """Gaussian mass of each centroid's cell (cells split at midpoints)."""
    c = np.asarray(centroids, dtype=np.float64)
    edges = np.concatenate(([-np.inf], (c[1:] + c[:-1]) / 2.0, [np.inf]))
    p = np.diff(ndtr(edges / sigma))
    return p / p.sum()


def byte_probs(field_probs, bits: int) -> np.ndarray:
    """Distribution of a byte whose 8/bits fields are i.i.d. ``field_probs``."""
    fp = np.asarray(field_probs, dtype=np.float64)
    per = 8 // bits
    vals = np.arange(256)
    p = np.ones(256)
    for i in range(per):
        p *= fp[(vals >> (bits * i)) & ((1 << bits) - 1)]
    return p / p.sum()


def draw_bytes(g: np.random.Generator, shape, probs) -> np.ndarray:
    cdf = np.cumsum(np.asarray(probs, dtype=np.float64))
    cdf[-1] = 1.0
    u = g.random(shape)
    return np.searchsorted(cdf, u, side="right").clip(0, 255).astype(np.uint8)


def cbk_packed(g: np.random.Generator, N: int, K: int, bits: int, probs) -> np.ndarray:
    """Index bytes of a CBK4 ([N, K/2]) or CBK8 ([N, K]) matrix."""
    if bits == 4:
        return draw_bytes(g, (N, K // 2), byte_probs(probs, 4))
    if bits == 8:
        return draw_bytes(g, (N, K), probs)
    raise ValueError("bits must be 4 or 8")


def cbk_row_codebooks(g: np.random.Generator, N: int, L: int = 16, sigma=(0.01, 0.03)) -> np.ndarray:
    """Per-output-row fp32 codebooks [N, L]: row n's L mid-rank quantiles of
    N(0, s_n), s_n drawn uniformly from `sigma`, plus a jitter of a tenth of
    the smallest gap (so rows differ beyond a scale); sorted ascending."""
    base = ndtri((np.arange(L) + 0.5) / L)
    s = g.uniform(sigma[0], sigma[1], size=(N, 1))
    gap = np.min(np.diff(base))
    jitter = g.uniform(-0.1, 0.1, size=(N, L)) * gap
    return np.sort((base[None, :] + jitter) * s, axis=1).astype(np.float32)


def pq2_packed(g: np.random.Generator, N: int, K: int, sigma: float = 0.02) -> np.ndarray:
    """Canonical PQ2_0 rows: N*K/128 blocks of {fp16 d, 32 code bytes}."""
    nb = K // 128
    blocks = np.empty((N, nb, 34), dtype=np.uint8)
    d = np.abs(g.standard_normal((N, nb), dtype=np.float32) * np.float32(sigma))
    blocks[:, :, 0:2] = d.astype(np.float16).view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = draw_bytes(g, (N, nb, 32), byte_probs(PQ2_CODE_PROBS, 2))
    return blocks.reshape(N, nb * 34)


def aqlm_inputs(g: np.random.Generator, N: int, K: int):
    """(codes u8 [N, K/8, 2], scales fp16 [N], codebooks fp16 [2, 256, 8])."""
    codes = g.integers(0, 256, size=(N, K // 8, 2), dtype=np.uint8)
    codebooks = (g.standard_normal((2, 256, 8), dtype=np.float32) * np.float32(0.01)
                 ).astype(np.float16)
    scales = g.uniform(0.5, 1.5, size=N).astype(np.float32).astype(np.float16)
    return codes, scales, codebooks


def aqlm_1x16_inputs(g: np.random.Generator, N: int, K: int, sigma: float = 0.014):
    """(codes u16 [N, K/8], scales fp16 [N], codebook fp16 [65536, 8]): codes
    uniform, entries N(0, sigma) (about the spread of a 2x8 sum of two
    N(0, 0.01) entries), scales U(0.5, 1.5)."""
    codes = g.integers(0, 65536, size=(N, K // 8), dtype=np.uint16)
    codebook = (g.standard_normal((65536, 8), dtype=np.float32) * np.float32(sigma)).astype(np.float16)
    scales = g.uniform(0.5, 1.5, size=N).astype(np.float32).astype(np.float16)
    return codes, scales, codebook


# --------------------------------------------------------------- device ----

def _torch():
    import torch
    return torch


def _gen(tag: str, seed: int, device):
    torch = _torch()
    gen = torch.Generator(device=device)
    gen.manual_seed(torch_seed(tag, seed))
    return gen


def x_fp16_cuda(tag: str, M: int, K: int, device="cuda", seed: int = 0):
    torch = _torch()
    return torch.randn((M, K), generator=_gen(tag, seed, device), device=device,
                       dtype=torch.float32).to(torch.float16)


def w_fp32_cuda(tag: str, N: int, K: int, sigma: float = 0.02, device="cuda",
                seed: int = 0):
    torch = _torch()
    return torch.randn((N, K), generator=_gen(tag, seed, device), device=device,
                       dtype=torch.float32) * sigma


def draw_bytes_cuda(tag: str, shape, probs, device="cuda", seed: int = 0,
                    chunk: int = 1 << 28):
    """Byte tensor of ``shape`` with i.i.d. bytes from ``probs`` (256 values)."""
    torch = _torch()
    cdf = torch.tensor(np.cumsum(np.asarray(probs, dtype=np.float64)),
                       dtype=torch.float64, device=device)
    cdf[-1] = 1.0
    gen = _gen(tag, seed, device)
    out = torch.empty(int(np.prod(shape)), dtype=torch.uint8, device=device)
    for s in range(0, out.numel(), chunk):
        e = min(out.numel(), s + chunk)
        u = torch.rand(e - s, generator=gen, device=device, dtype=torch.float64)
        out[s:e] = torch.searchsorted(cdf, u, right=True).clamp_(0, 255).to(torch.uint8)
    return out.view(*shape)


def cbk_packed_cuda(tag: str, N: int, K: int, bits: int, probs, device="cuda",
                    seed: int = 0):
    if bits == 4:
        return draw_bytes_cuda(tag, (N, K // 2), byte_probs(probs, 4), device, seed)
    return draw_bytes_cuda(tag, (N, K), probs, device, seed)


def pq2_packed_cuda(tag: str, N: int, K: int, sigma: float = 0.02, device="cuda",
                    seed: int = 0):
    torch = _torch()
    nb = K // 128
    blocks = torch.empty((N, nb, 34), dtype=torch.uint8, device=device)
    d = (torch.randn((N, nb), generator=_gen(tag + "/d", seed, device), device=device)
         * sigma).abs_().to(torch.float16)
    blocks[:, :, 0:2] = d.view(torch.uint8).view(N, nb, 2)
    blocks[:, :, 2:] = draw_bytes_cuda(tag + "/qs", (N, nb, 32),
                                       byte_probs(PQ2_CODE_PROBS, 2), device, seed)
    return blocks.view(N, nb * 34)


def aqlm_inputs_cuda(tag: str, N: int, K: int, device="cuda", seed: int = 0):
    torch = _torch()
    codes = torch.randint(0, 256, (N, K // 8, 2), generator=_gen(tag + "/codes", seed, device),
                          device=device, dtype=torch.int32).to(torch.uint8)
    codebooks = (torch.randn((2, 256, 8), generator=_gen(tag + "/cb", seed, device),
                             device=device) * 0.01).to(torch.float16)
    scales = (torch.rand(N, generator=_gen(tag + "/s", seed, device), device=device)
              + 0.5).to(torch.float16)
    return codes, scales, codebooks


def aqlm_1x16_inputs_cuda(tag: str, N: int, K: int, sigma: float = 0.014, device="cuda", seed: int = 0):
    torch = _torch()
    # uniform 16-bit patterns, held as int16 (torch has no uint16 arithmetic)
    codes = torch.randint(-32768, 32768, (N, K // 8), generator=_gen(tag + "/codes", seed, device),
                          device=device, dtype=torch.int32).to(torch.int16)
    codebook = (torch.randn((65536, 8), generator=_gen(tag + "/cb", seed, device),
                            device=device) * sigma).to(torch.float16)
    scales = (torch.rand(N, generator=_gen(tag + "/s", seed, device), device=device)
              + 0.5).to(torch.float16)
    return codes, scales, codebook
