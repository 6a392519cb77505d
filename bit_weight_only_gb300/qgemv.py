"""Thin ctypes binding of the C ABI in ``include/qgemv.h``.

The functions keep the C names and only marshal arguments (pointers and
sizes); every step of the computation runs in ``libqgemv.so``.  The library
is loaded on first use from ``bit_weight_only_gb300/_build``; if it is
missing, ``load()`` raises: there is no CPU fallback.

``QGemv`` wraps one handle for torch users: it takes canonical inputs as
torch tensors or numpy arrays (host or CUDA) and runs on CUDA tensors.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

Q4_0, CBK4, CBK8, PQ2_0, AQLM_2X8, AQLM_1X16, CBK4_ROW, CBK8_ROW = 1, 2, 3, 4, 5, 7, 8, 9
FORMATS = {"q4_0": Q4_0, "cbk4": CBK4, "cbk8": CBK8, "pq2_0": PQ2_0, "aqlm_2x8": AQLM_2X8,
           "aqlm_1x16": AQLM_1X16, "cbk4_row": CBK4_ROW, "cbk8_row": CBK8_ROW}
QGEMV_OK, QGEMV_ERR_ARG, QGEMV_ERR_ALIGN, QGEMV_ERR_CUDA, QGEMV_ERR_TIMEOUT, QGEMV_ERR_NOMEM = range(6)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libqgemv.so")

# Every exported symbol of include/qgemv.h with its ctypes signature.
_SIGNATURES = {
    "qgemv_packed_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qgemv_create": (ctypes.c_void_p, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_create_stacked": (ctypes.c_void_p, [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p]),
    "qgemv_run": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_run_residual": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_set_batch_invariant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "qgemv_set_x_int8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "qgemv_create_glu": (ctypes.c_void_p, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_xq_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int64]),
    "qgemv_prepare_x_int8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_run_xq": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_quantize_x_int8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_dequant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_quantize_q4_0": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_void_p]),
    "qgemv_status": (ctypes.c_int, [ctypes.c_void_p]),
    "qgemv_run_q4_0_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p]),
    "qgemv_stream_k_plan": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]),
    "qgemv_destroy": (None, [ctypes.c_void_p]),
    "qgemv_last_error": (ctypes.c_char_p, []),
    "qgemv_last_error_code": (ctypes.c_int, []),
}

_lib = None


class QgemvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qgemv error {code}: {msg}")
        self.code = code


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libqgemv.so (once) and declare the ABI's signatures."""
    global _lib
    if _lib is None:
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"libqgemv.so not built ({path}); run "
                              "`python -m bit_weight_only_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _check(rc: int):
    if rc != QGEMV_OK:
        raise QgemvError(rc, qgemv_last_error())
    return rc


def _stream_ptr(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


# --------------------------------------------------------- C-ABI mirrors ----

def qgemv_packed_bytes(fmt, N: int, K: int) -> int:
    return int(load().qgemv_packed_bytes(_fmt(fmt), N, K))


def qgemv_create(fmt, N: int, K: int, packed: int, scales: int | None,
                 codebooks: int | None) -> int:
    """Pointers are raw addresses (host or device).  Returns the handle."""
    h = load().qgemv_create(_fmt(fmt), N, K, packed, scales, codebooks)
    if not h:
        raise QgemvError(qgemv_last_error_code(), qgemv_last_error())
    return h


def qgemv_create_stacked(fmt, seg_rows, K: int, packed: int, scales: int | None,
                         codebooks: int | None) -> int:
    """Several projections sharing K, rows stacked; one codebook per segment."""
    rows = (ctypes.c_int64 * len(seg_rows))(*[int(r) for r in seg_rows])
    h = load().qgemv_create_stacked(_fmt(fmt), len(seg_rows), rows, K, packed, scales, codebooks)
    if not h:
        raise QgemvError(qgemv_last_error_code(), qgemv_last_error())
    return h


def qgemv_create_glu(fmt, N: int, K: int, packed_gate: int, packed_up: int,
                     codebooks_gate: int | None = None, codebooks_up: int | None = None) -> int:
    """Gate and up projections in one handle whose runs store SiLU(gate) * up."""
    h = load().qgemv_create_glu(_fmt(fmt), N, K, packed_gate, packed_up, codebooks_gate, codebooks_up)
    if not h:
        raise QgemvError(qgemv_last_error_code(), qgemv_last_error())
    return h


def qgemv_run(h: int, x: int, M: int, y: int, stream=None) -> int:
    return _check(load().qgemv_run(h, x, M, y, _stream_ptr(stream)))


def qgemv_run_residual(h: int, x: int, M: int, y: int, residual: int, stream=None) -> int:
    return _check(load().qgemv_run_residual(h, x, M, y, residual, _stream_ptr(stream)))


def qgemv_dequant(h: int, w_out: int, stream=None) -> int:
    return _check(load().qgemv_dequant(h, w_out, _stream_ptr(stream)))


def qgemv_quantize_q4_0(w: int, N: int, K: int, packed_out: int, stream=None) -> int:
    return _check(load().qgemv_quantize_q4_0(w, N, K, packed_out, _stream_ptr(stream)))


def qgemv_run_q4_0_noalloc(packed: int, N: int, K: int, x: int, M: int, y: int,
                           stream=None) -> int:
    """Allocation-free Q4_0 GEMV on canonical device blocks (no handle)."""
    return _check(load().qgemv_run_q4_0_noalloc(packed, N, K, x, M, y, _stream_ptr(stream)))


def qgemv_set_batch_invariant(h: int, on: bool) -> int:
    return _check(load().qgemv_set_batch_invariant(h, 1 if on else 0))


def qgemv_set_x_int8(h: int, on: bool) -> int:
    return _check(load().qgemv_set_x_int8(h, 1 if on else 0))


def qgemv_quantize_x_int8(x: int, M: int, K: int, q_out: int, a_out: int, stream=None) -> int:
    return _check(load().qgemv_quantize_x_int8(x, M, K, q_out, a_out, _stream_ptr(stream)))


def qgemv_xq_bytes(M: int, K: int) -> int:
    return int(load().qgemv_xq_bytes(M, K))


def qgemv_prepare_x_int8(x: int, M: int, K: int, signs: int | None, hadamard_block: int, xq: int,
                         stream=None) -> int:
    return _check(load().qgemv_prepare_x_int8(x, M, K, signs, hadamard_block, xq, _stream_ptr(stream)))


def qgemv_run_xq(h: int, xq: int, M: int, y: int, residual: int | None = None, stream=None) -> int:
    return _check(load().qgemv_run_xq(h, xq, M, y, residual, _stream_ptr(stream)))


def qgemv_status(h: int) -> int:
    return _check(load().qgemv_status(h))


def qgemv_stream_k_plan(units: int, grid: int, units_per_row_tile: int, rows: int, split_unit: int = 1) -> list:
    """The stream-K split the handles use (host only): per CTA a dict of its
    two shared-row-tile segments, each field a pair (first, last row tile);
    "side1" and "fin" are the two flag bits."""
    out = (ctypes.c_int64 * (12 * grid))()
    _check(load().qgemv_stream_k_plan(units, grid, units_per_row_tile, rows, split_unit, out))
    keys = ("rt", "cf", "S", "r0", "nr", "flags")
    plan = [{k: (out[12 * c + 2 * i], out[12 * c + 2 * i + 1]) for i, k in enumerate(keys)}
            for c in range(grid)]
    for d in plan:
        f = d.pop("flags")
        d["side1"] = (f[0] & 1, f[1] & 1)
        d["fin"] = ((f[0] >> 1) & 1, (f[1] >> 1) & 1)
    return plan


def qgemv_destroy(h: int) -> None:
    load().qgemv_destroy(h)


def qgemv_last_error() -> str:
    return (load().qgemv_last_error() or b"").decode()


def qgemv_last_error_code() -> int:
    return int(load().qgemv_last_error_code())


# ----------------------------------------------------------- torch helper --

def _addr(a):
    """(address, keepalive) of a torch tensor / numpy array / None."""
    if a is None:
        return None, None
    if isinstance(a, np.ndarray):
        a = np.ascontiguousarray(a)
        return a.ctypes.data, a
    a = a.contiguous()
    return a.data_ptr(), a


def _current(stream):
    """The stream a torch-level call runs on: the one given, else torch's
    current stream (the C calls themselves take NULL as the legacy default
    stream)."""
    if stream is not None:
        return stream
    import torch
    return torch.cuda.current_stream().cuda_stream


class QGemv:
    """One packed weight matrix on the GPU.

    ``QGemv(fmt, N, K, packed, scales=None, codebooks=None)`` copies the
    canonical inputs into the library; ``gemv(x)`` returns y = x . W^T as a
    new fp32 CUDA tensor, ``run(x, y)`` writes into ``y``.  Runs are ordered
    on ``stream`` when one is given, else on torch's current stream, like the
    torch operations around them."""

    def __init__(self, fmt, N: int, K: int, packed, scales=None, codebooks=None):
        self.fmt, self.N, self.K = _fmt(fmt), int(N), int(K)
        p, kp = _addr(packed)
        s, ks = _addr(scales)
        c, kc = _addr(codebooks)
        self.handle = qgemv_create(self.fmt, self.N, self.K, p, s, c)
        del kp, ks, kc

    @classmethod
    def stacked(cls, fmt, seg_rows, K: int, packed, scales=None, codebooks=None):
        """One handle over projections with the same K (rows stacked in
        order, codebook s for segment s; AQLM 2x8: a codebook pair per
        segment, the N row scales in order, segments on 2048-row blocks):
        one run computes them all."""
        self = cls.__new__(cls)
        self.fmt, self.N, self.K = _fmt(fmt), int(sum(seg_rows)), int(K)
        p, kp = _addr(packed)
        s, ks = _addr(scales)
        c, kc = _addr(codebooks)
        self.handle = qgemv_create_stacked(self.fmt, list(seg_rows), self.K, p, s, c)
        del kp, ks, kc
        return self

    @classmethod
    def glu(cls, fmt, N: int, K: int, packed_gate, packed_up, codebooks_gate=None, codebooks_up=None):
        """Fused MLP gate/up: ``gemv(x)`` returns SiLU(x . G^T) * (x . U^T),
        fp32 [M, N] (codebooks: each matrix's fp16 codebook for CBK4 / CBK8,
        CBK4_ROW's per-row fp32 [N, 16] arrays)."""
        self = cls.__new__(cls)
        self.fmt, self.N, self.K = _fmt(fmt), int(N), int(K)
        g, kg = _addr(packed_gate)
        u, ku = _addr(packed_up)
        cg, kcg = _addr(codebooks_gate)
        cu, kcu = _addr(codebooks_up)
        self.handle = qgemv_create_glu(self.fmt, self.N, self.K, g, u, cg, cu)
        del kg, ku, kcg, kcu
        return self

    def run(self, x, y, stream=None):
        M = x.shape[0]
        qgemv_run(self.handle, x.data_ptr(), M, y.data_ptr(), _current(stream))
        return y

    def run_residual(self, x, y, residual, stream=None):
        """y = residual + x . W^T (residual may be y itself)."""
        qgemv_run_residual(self.handle, x.data_ptr(), x.shape[0], y.data_ptr(), residual.data_ptr(),
                           _current(stream))
        return y

    def gemv(self, x, stream=None):
        import torch
        y = torch.empty((x.shape[0], self.N), dtype=torch.float32, device=x.device)
        return self.run(x.contiguous(), y, stream)

    def dequant(self, stream=None):
        import torch
        w = torch.empty((self.N, self.K), dtype=torch.float32, device="cuda")
        qgemv_dequant(self.handle, w.data_ptr(), _current(stream))
        return w

    def status(self):
        return qgemv_status(self.handle)

    def set_batch_invariant(self, on: bool = True):
        qgemv_set_batch_invariant(self.handle, on)

    def set_x_int8(self, on: bool = True):
        qgemv_set_x_int8(self.handle, on)

    def run_xq(self, xq, M: int, y, residual=None, stream=None):
        """y (+ residual) from prepared INT8 activations (``prepare_x_int8``)."""
        qgemv_run_xq(self.handle, xq.data_ptr(), M, y.data_ptr(),
                     None if residual is None else residual.data_ptr(), _current(stream))
        return y

    def close(self):
        if getattr(self, "handle", None):
            qgemv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def quantize_q4_0(w, stream=None):
    """Q4_0 quantizer on the GPU: fp32 CUDA tensor [N, K] -> uint8 CUDA tensor."""
    import torch
    N, K = w.shape
    out = torch.empty(qgemv_packed_bytes(Q4_0, N, K), dtype=torch.uint8, device=w.device)
    qgemv_quantize_q4_0(w.contiguous().data_ptr(), N, K, out.data_ptr(), _current(stream))
    return out


def quantize_x_int8(x, stream=None):
    """PQ2_0 INT8 activation quantizer on the GPU: fp16 CUDA tensor [M, K]
    -> (int8 [M, K], fp32 scales [M, K/128]) CUDA tensors."""
    import torch
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    a = torch.empty((M, K // 128), dtype=torch.float32, device=x.device)
    qgemv_quantize_x_int8(x.contiguous().data_ptr(), M, K, q.data_ptr(), a.data_ptr(), _current(stream))
    return q, a


def prepare_x_int8(x, hadamard_block: int = 0, signs=None, stream=None):
    """PQ2_0 activation prologue on the GPU: fp16 CUDA tensor [M, K] -> the
    prepared uint8 CUDA buffer of ``qgemv_xq_bytes(M, K)`` bytes (INT8 codes in
    staging order, group scales, group code sums), after the Hadamard mixing
    of blocks of 1024 when ``hadamard_block`` is 1024 (signs: int8 CUDA
    tensor [K] of +-1, or None)."""
    import torch
    M, K = x.shape
    xq = torch.empty(qgemv_xq_bytes(M, K), dtype=torch.uint8, device=x.device)
    qgemv_prepare_x_int8(x.contiguous().data_ptr(), M, K, None if signs is None else signs.data_ptr(),
                         hadamard_block, xq.data_ptr(), _current(stream))
    return xq

