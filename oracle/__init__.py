"""CPU oracle for the weight-only quantized decode GEMV (fp64, plain C).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``bit_weight_only_gb300``), and it never imports
it.  The arithmetic lives in ``oracle.c``; this module only marshals numpy
arrays into it.

What it computes:  y[m][n] = sum_k x[m][k] * w[n][k] with w the exact fp64
decode of the canonical packed bytes, plus the per-output bound
B[m][n] = sum_k |x[m][k] * w[n][k]| used by the GEMV tolerance
|y - y_ref| <= 1e-3 * B + 1e-6.  See ``oracle.c`` for the formats, the pages
they come from and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

Q4_0, CBK4, CBK8, PQ2_0, AQLM_2X8, CBK4_ROW, AQLM_1X16, CBK8_ROW = 1, 2, 3, 4, 5, 6, 7, 8
FORMATS = {"q4_0": Q4_0, "cbk4": CBK4, "cbk8": CBK8, "pq2_0": PQ2_0,
           "aqlm_2x8": AQLM_2X8, "cbk4_row": CBK4_ROW, "aqlm_1x16": AQLM_1X16, "cbk8_row": CBK8_ROW}

_lib = None


def _load():
    global _lib
    if _lib is None:
        # A test may point the loader at a deliberately broken build of the
        # same source (mutation checks of the pins); normally it is built here.
        path = os.environ.get("ORACLE_LIB_OVERRIDE") or _build.build()
        lib = ctypes.CDLL(path)
        i64, c_int, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        lib.oracle_float_to_half.restype = ctypes.c_uint16
        lib.oracle_packed_bytes.argtypes = [c_int, i64, i64]
        lib.oracle_packed_bytes.restype = i64
        lib.oracle_scales_count.argtypes = [c_int, i64, i64]
        lib.oracle_scales_count.restype = i64
        lib.oracle_codebook_count.argtypes = [c_int]
        lib.oracle_codebook_count.restype = i64
        lib.oracle_codebook_bytes.argtypes = [c_int, i64]
        lib.oracle_codebook_bytes.restype = i64
        lib.oracle_dequant_row.argtypes = [c_int, i64, i64, vp, vp, vp, i64, vp]
        lib.oracle_dequant_row.restype = c_int
        lib.oracle_dequant.argtypes = [c_int, i64, i64, vp, vp, vp, vp]
        lib.oracle_dequant.restype = c_int
        lib.oracle_gemv.argtypes = [c_int, i64, i64, vp, vp, vp, vp, i64, vp, i64,
                                    vp, vp, c_int]
        lib.oracle_gemv.restype = c_int
        lib.oracle_quantize_q4_0.argtypes = [vp, i64, i64, vp]
        lib.oracle_quantize_q4_0.restype = c_int
        lib.oracle_quantize_x_int8.argtypes = [vp, i64, i64, vp, vp]
        lib.oracle_quantize_x_int8.restype = c_int
        lib.oracle_gemv_pq2_int8.argtypes = [i64, i64, vp, vp, i64, vp, vp, c_int]
        lib.oracle_gemv_pq2_int8.restype = c_int
        lib.oracle_gemv_pq2_int8_q.argtypes = [i64, i64, vp, vp, vp, i64, vp, vp, c_int]
        lib.oracle_gemv_pq2_int8_q.restype = c_int
        lib.oracle_quantize_f32_int8.argtypes = [vp, i64, i64, vp, vp]
        lib.oracle_quantize_f32_int8.restype = c_int
        lib.oracle_hadamard.argtypes = [vp, i64, i64, c_int, vp, vp]
        lib.oracle_hadamard.restype = c_int
        lib.oracle_hadamard_f32.argtypes = [vp, i64, i64, c_int, vp, vp]
        lib.oracle_hadamard_f32.restype = c_int
        _lib = lib
    return _lib


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    return None if a is None else np.ascontiguousarray(a).view(np.uint8).reshape(-1)


def _u16(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return a.reshape(-1)


def packed_bytes(fmt, N: int, K: int) -> int:
    """Size in bytes of the canonical packed weights (0 if (N, K) is invalid)."""
    return int(_load().oracle_packed_bytes(_fmt(fmt), N, K))


def scales_count(fmt, N: int, K: int) -> int:
    return int(_load().oracle_scales_count(_fmt(fmt), N, K))


def codebook_count(fmt) -> int:
    return int(_load().oracle_codebook_count(_fmt(fmt)))


def codebook_bytes(fmt, N: int) -> int:
    """Bytes of the codebooks input of an N-row matrix (cbk4_row: fp32 [N][16])."""
    return int(_load().oracle_codebook_bytes(_fmt(fmt), N))


def half_to_double(bits: int) -> float:
    return float(_load().oracle_half_to_double(int(bits) & 0xFFFF))


def float_to_half(value: float) -> int:
    return int(_load().oracle_float_to_half(float(value)))


def _check(fmt, N, K, packed, scales, codebooks):
    f = _fmt(fmt)
    nbytes = packed_bytes(f, N, K)
    if nbytes == 0:
        raise ValueError(f"invalid (format, N, K) = ({fmt}, {N}, {K})")
    p = _u8(packed)
    if p.size != nbytes:
        raise ValueError(f"packed has {p.size} bytes, expected {nbytes}")
    s = _u16(scales)
    if scales_count(f, N, K) and (s is None or s.size != scales_count(f, N, K)):
        raise ValueError("scales missing or of the wrong size")
    if f in (CBK4_ROW, CBK8_ROW):  # fp32 [N][16] or [N][256], passed as bytes
        c = None if codebooks is None else np.ascontiguousarray(codebooks, dtype=np.float32).view(np.uint8).reshape(-1)
        if c is None or c.size != codebook_bytes(f, N):
            raise ValueError("codebooks missing or of the wrong size")
        return f, p, s, c
    c = _u16(codebooks)
    if codebook_count(f) and (c is None or c.size != codebook_count(f)):
        raise ValueError("codebooks missing or of the wrong size")
    return f, p, s, c


def dequant(fmt, N: int, K: int, packed, scales=None, codebooks=None) -> np.ndarray:
    """Exact fp64 decode of the whole matrix, shape [N, K]."""
    f, p, s, c = _check(fmt, N, K, packed, scales, codebooks)
    w = np.empty((N, K), dtype=np.float64)
    rc = _load().oracle_dequant(f, N, K, _ptr(p), _ptr(s), _ptr(c), _ptr(w))
    if rc:
        raise RuntimeError(f"oracle_dequant failed ({rc})")
    return w


def dequant_rows(fmt, N: int, K: int, packed, scales, codebooks, rows) -> np.ndarray:
    """Exact fp64 decode of the listed rows, shape [len(rows), K]."""
    f, p, s, c = _check(fmt, N, K, packed, scales, codebooks)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, K), dtype=np.float64)
    lib = _load()
    for i, n in enumerate(rows):
        rc = lib.oracle_dequant_row(f, N, K, _ptr(p), _ptr(s), _ptr(c), int(n),
                                    _ptr(out[i]))
        if rc:
            raise RuntimeError(f"oracle_dequant_row failed ({rc})")
    return out


def gemv(fmt, N: int, K: int, packed, scales, codebooks, x, rows=None,
         nthreads: int | None = None):
    """Reference GEMV.  x: fp16 [M, K].  Returns (y, bound), fp64 [M, len(rows)]
    (all N rows when ``rows`` is None)."""
    f, p, s, c = _check(fmt, N, K, packed, scales, codebooks)
    x = np.ascontiguousarray(x, dtype=np.float16)
    if x.ndim != 2 or x.shape[1] != K:
        raise ValueError("x must be fp16 [M, K]")
    M = x.shape[0]
    if rows is None:
        nrows, r = N, None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        if r.size and (r.min() < 0 or r.max() >= N):
            raise ValueError("row index out of range")
        nrows = r.size
    y = np.empty((M, nrows), dtype=np.float64)
    b = np.empty((M, nrows), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().oracle_gemv(f, N, K, _ptr(p), _ptr(s), _ptr(c), _ptr(_u16(x)), M,
                             _ptr(r), nrows, _ptr(y), _ptr(b), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_gemv failed ({rc})")
    return y, b


def quantize_q4_0(w, N: int, K: int) -> np.ndarray:
    """Q4_0 quantizer: fp32 [N, K] -> canonical blocks (uint8, N*K/32*18 bytes)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.shape != (N, K):
        raise ValueError("w must be fp32 [N, K]")
    out = np.empty(packed_bytes(Q4_0, N, K), dtype=np.uint8)
    rc = _load().oracle_quantize_q4_0(_ptr(w), N, K, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_quantize_q4_0 failed ({rc})")
    return out


def gemv_residual(fmt, N: int, K: int, packed, scales, codebooks, x, residual, rows=None,
                  nthreads: int | None = None):
    """Reference GEMV with the residual add of the fused attention-output and
    MLP-down projections ("Trapetum benchmarks", "Short-context decode, step
    by step"): y = residual + x . W^T, in fp64.  residual: [M, N].  Returns
    (y, bound), bound being the GEMV's sum of |x * w| (fp64, [M, len(rows)])."""
    y, b = gemv(fmt, N, K, packed, scales, codebooks, x, rows=rows, nthreads=nthreads)
    r = np.asarray(residual, dtype=np.float64)
    if r.shape != (y.shape[0], N):
        raise ValueError("residual must be [M, N]")
    if rows is not None:
        r = r[:, np.asarray(rows, dtype=np.int64)]
    return y + r, b


def within_tolerance_residual(y, y_ref, bound):
    """Acceptance with a residual: the GEMV's bound, plus one fp32 rounding of
    the sum (2^-24 of its magnitude; 2^-23 of the exact value covers both)."""
    y = np.asarray(y, dtype=np.float64)
    return np.abs(y - y_ref) <= 1e-3 * bound + 1e-6 + 2.0 ** -23 * np.abs(y_ref)


def within_tolerance(y, y_ref, bound, rel: float = 1e-3, abs_: float = 1e-6):
    """Elementwise GEMV acceptance: |y - y_ref| <= rel * bound + abs."""
    y = np.asarray(y, dtype=np.float64)
    return np.abs(y - y_ref) <= rel * bound + abs_


def quantize_x_int8(x):
    """The PQ2_0 integer path's activation quantizer (reading R11): fp16
    [M, K] (K % 128 == 0) -> (q int8 [M, K], a fp32 [M, K/128]) with
    x ~ a * q per group of 128."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.int8)
    a = np.empty((M, K // 128), dtype=np.float32)
    rc = _load().oracle_quantize_x_int8(_ptr(_u16(x)), M, K, _ptr(q), _ptr(a))
    if rc:
        raise ValueError(f"oracle_quantize_x_int8 failed ({rc})")
    return q, a


def gemv_pq2_int8(N: int, K: int, packed, x, nthreads: int | None = None):
    """PQ2_0 GEMV on the integer path: INT8 activations per group of 128,
    integer inner sums, d * a applied per block.  Returns (y, bound), fp64
    [M, N]; bound is the sum of |terms| of the same expansion."""
    p = _u8(packed)
    if p is None or p.size != packed_bytes("pq2_0", N, K):
        raise ValueError("packed missing or of the wrong size")
    x = np.ascontiguousarray(x, dtype=np.float16)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemv_pq2_int8(N, K, _ptr(p), _ptr(_u16(x)), M, _ptr(y), _ptr(b),
                                      int(nthreads or os.cpu_count() or 1))
    if rc:
        raise RuntimeError(f"oracle_gemv_pq2_int8 failed ({rc})")
    return y, b


def quantize_f32_int8(v):
    """The quantizer of ``quantize_x_int8`` on fp32 activations [M, K]."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    M, K = v.shape
    q = np.empty((M, K), dtype=np.int8)
    a = np.empty((M, K // 128), dtype=np.float32)
    rc = _load().oracle_quantize_f32_int8(_ptr(v), M, K, _ptr(q), _ptr(a))
    if rc:
        raise ValueError(f"oracle_quantize_f32_int8 failed ({rc})")
    return q, a


def gemv_pq2_int8_q(N: int, K: int, packed, q, a, nthreads: int | None = None):
    """PQ2_0 integer-path GEMV on given INT8 codes q [M, K] and group scales
    a [M, K/128].  Returns (y, bound), fp64 [M, N]."""
    p = _u8(packed)
    if p is None or p.size != packed_bytes("pq2_0", N, K):
        raise ValueError("packed missing or of the wrong size")
    q = np.ascontiguousarray(q, dtype=np.int8)
    a = np.ascontiguousarray(a, dtype=np.float32)
    M = q.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemv_pq2_int8_q(N, K, _ptr(p), _ptr(q), _ptr(a), M, _ptr(y), _ptr(b),
                                        int(nthreads or os.cpu_count() or 1))
    if rc:
        raise RuntimeError(f"oracle_gemv_pq2_int8_q failed ({rc})")
    return y, b


def _signs(signs, K):
    if signs is None:
        return None
    s = np.ascontiguousarray(signs, dtype=np.int8)
    if s.shape != (K,) or not np.all(np.abs(s) == 1):
        raise ValueError("signs must be +-1, one per input position")
    return s


def hadamard(x, B: int = 1024, signs=None):
    """Exact fp64 Hadamard mixing of each block of B inputs (reading R13):
    y = B^-1/2 H_B (s . x).  x: [M, K]; signs: +-1 [K] or None."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    M, K = x.shape
    s = _signs(signs, K)
    y = np.empty((M, K), dtype=np.float64)
    rc = _load().oracle_hadamard(_ptr(x), M, K, int(B), _ptr(s), _ptr(y))
    if rc:
        raise ValueError(f"oracle_hadamard failed ({rc})")
    return y


def hadamard_f32(x, B: int = 1024, signs=None):
    """The page's fp32 butterfly form of ``hadamard`` (the values the INT8
    codes of the fused prologue are decided on)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    s = _signs(signs, K)
    y = np.empty((M, K), dtype=np.float32)
    rc = _load().oracle_hadamard_f32(_ptr(x), M, K, int(B), _ptr(s), _ptr(y))
    if rc:
        raise ValueError(f"oracle_hadamard_f32 failed ({rc})")
    return y


def prepare_x_int8(x, B: int = 0, signs=None):
    """The activation prologue of the PQ2_0 integer path: with B > 0 the
    Hadamard mixing (fp32 butterfly) and then INT8 quantization of the fp32
    result; with B = 0 the INT8 quantization of x itself.  x fp16 [M, K].
    Returns (q, a)."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    if B == 0:
        return quantize_x_int8(x)
    return quantize_f32_int8(hadamard_f32(x.astype(np.float32), B, signs))


def silu(v):
    """SiLU (the gate activation of the pages' MLP), v / (1 + exp(-v)), fp64."""
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def gemv_glu(fmt, N: int, K: int, packed_gate, packed_up, x, nthreads: int | None = None,
             codebooks_gate=None, codebooks_up=None):
    """The fused gate/up projection of a decoder MLP: y = SiLU(x . G^T) * (x . U^T)
    for two matrices of the same format and shape [N, K] (no scales; each
    its own codebooks where the format has them).  Returns
    (y, g, u, bound_g, bound_u), fp64 [M, N]."""
    g, bg = gemv(fmt, N, K, packed_gate, None, codebooks_gate, x, nthreads=nthreads)
    u, bu = gemv(fmt, N, K, packed_up, None, codebooks_up, x, nthreads=nthreads)
    return silu(g) * u, g, u, bg, bu


def within_tolerance_glu(y, g, u, bound_g, bound_u):
    """Acceptance for SiLU(g) * u (reading R14): each GEMV output may be off by
    its own bound e = 1e-3 * B + 1e-6; SiLU's slope is below 1.1, so the
    product may be off by 1.1 e_g (|u| + e_u) + |SiLU(g)| e_u, plus a few fp32
    roundings of the result (expf, the division and the product)."""
    y = np.asarray(y, dtype=np.float64)
    eg = 1e-3 * np.asarray(bound_g) + 1e-6
    eu = 1e-3 * np.asarray(bound_u) + 1e-6
    sg = np.abs(silu(g))
    au = np.abs(u)
    lim = 1.1 * eg * (au + eu) + sg * eu + 2.0 ** -20 * (sg + 1.1 * eg) * (au + eu)
    return np.abs(y - silu(g) * u) <= lim
