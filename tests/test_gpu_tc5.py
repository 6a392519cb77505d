"""GPU parity of the tensor-memory GEMV kernel (tc5_kernel.cuh: weights
decoded into tensor memory, tcgen05.mma with fp32 accumulators) for Q4_0,
PQ2_0, CBK4 and CBK8, forced on at every M with the QGEMV_TC5 create-time
hook (by default it serves the larger M only).

Bars, as for the other kernels:
  * every output within |y - y_ref| <= 1e-3 * sum_k |x_k w_nk| + 1e-6 of the
    fp64 oracle, at M = 1..16, on shapes with several row and k tiles and
    ragged tails, with row tiles shared between CTAs and owned whole, and at
    full workload sizes on sampled rows;
  * one-hot activations return W's columns bit for bit (the kernel's own
    decode: codes, offsets and centroids exact in fp16, products exact, sums
    in fp32), at every code of the format;
  * run to run and eager vs CUDA graph bitwise; the residual form equals the
    plain run plus the residual; a stacked table handle switches codebooks
    between row tiles; the output guard bands stay untouched.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, qgemv
from cases import make_case, make_x
from test_gpu_onehot import (case_with_all_codes, check_columns, codes_of_columns, columns, run_onehot,
                             CODES)

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.late]

FORMATS = ["q4_0", "pq2_0", "cbk4", "cbk8"]
SMALL = {"q4_0": (300, 1120), "pq2_0": (300, 2176), "cbk4": (300, 1090), "cbk8": (300, 777)}
MULTI = {"q4_0": (2500, 8192), "pq2_0": (2500, 16384), "cbk4": (2500, 8192), "cbk8": (2500, 4096)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb, stacked_rows=None):
    monkeypatch.setenv("QGEMV_TC5", "1")
    if stacked_rows is not None:
        h = qgemv.QGemv.stacked(fmt, stacked_rows, K, packed, scales, cb)
    else:
        h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    monkeypatch.delenv("QGEMV_TC5")
    return h


def gemv_checked(h, x_np):
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    return y.cpu().numpy()


def assert_within(y, y_ref, bound, what):
    ok = oracle.within_tolerance(y, y_ref, bound)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} outputs out of tolerance, e.g. "
                             f"{[(tuple(i), float(y[tuple(i)]), float(y_ref[tuple(i)])) for i in idx]}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", list(range(1, 17)))
def test_tc5_small_all_m(fmt, M, monkeypatch):
    N, K = SMALL[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="tc5small")
    x = make_x(M, K, tag="tc5small")
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
    assert_within(gemv_checked(h, x), y_ref, bound, f"{fmt} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", [1, 5, 8, 9, 16])
def test_tc5_many_tiles_per_cta(fmt, M, monkeypatch):
    N, K = MULTI[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="tc5multi")
    x = make_x(M, K, tag="tc5multi")
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
    assert_within(gemv_checked(h, x), y_ref, bound, f"{fmt} {N}x{K} M={M}")


MIN_K = {"q4_0": 32, "pq2_0": 128, "cbk4": 2, "cbk8": 1}


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N, Kmul", [(1, 1), (1, 7), (127, 2), (128, 3), (129, 5), (4095, 4)])
def test_tc5_edge_shapes(fmt, N, Kmul, monkeypatch):
    K = MIN_K[fmt] * Kmul
    packed, scales, cb = make_case(fmt, N, K, tag="tc5edge")
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    for M in (1, 9, 16):
        x = make_x(M, K, tag="tc5edge")
        y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
        assert_within(gemv_checked(h, x), y_ref, bound, f"{fmt} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("shape", ["small", "multi"])
@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_tc5_one_hot_columns(fmt, shape, M, monkeypatch):
    N, K = SMALL[fmt] if shape == "small" else (1000, MULTI[fmt][1])
    packed, scales, cb = case_with_all_codes(fmt, N, K, tag=f"tc5onehot/{shape}")
    cols = columns(fmt, K)
    assert np.unique(codes_of_columns(fmt, N, K, packed, cols)).size == CODES[fmt]
    W = oracle.dequant(fmt, N, K, packed, scales, cb)
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    y, z = run_onehot(h, N, K, cols, M)
    check_columns(y, z, W, cols, f"tc5 {fmt} {N}x{K} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_tc5_run_to_run_graph_and_residual(fmt, monkeypatch):
    N, K = MULTI[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="tc5repro")
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    x = torch.from_numpy(make_x(12, K, tag="tc5repro")).cuda()
    y1 = h.gemv(x)
    y2 = h.gemv(x)
    s = torch.cuda.Stream()
    y3 = torch.empty_like(y1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        h.run(x, y3, stream=s)
    y3.zero_()
    g.replay()
    g.replay()
    r = torch.randn_like(y1)
    y4 = torch.empty_like(y1)
    h.run_residual(x, y4, r)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y1, y2)
    assert torch.equal(y1, y3)
    assert torch.equal(y4, y1 + r)


@pytest.mark.parametrize("fmt", ["cbk4", "cbk8"])
def test_tc5_stacked_codebooks(fmt, monkeypatch):
    K = 4096
    rows = [384, 256, 300]
    L = 16 if fmt == "cbk4" else 256
    parts = [make_case(fmt, r, K, tag=f"tc5stk{i}") for i, r in enumerate(rows)]
    cbs = [(parts[0][2].astype(np.float32) * s).astype(np.float16) for s in (1.0, -0.75, 1.25)]
    packed = np.concatenate([p[0] for p in parts])
    h = tc5_handle(monkeypatch, fmt, sum(rows), K, packed, None, np.concatenate(cbs), stacked_rows=rows)
    assert cbs[0].size == L
    for M in (3, 16):
        x = make_x(M, K, tag="tc5stk")
        y = gemv_checked(h, x)
        n0 = 0
        for r, p, cbk in zip(rows, parts, cbs):
            y_ref, bound = oracle.gemv(fmt, r, K, p[0], None, cbk, x)
            assert_within(y[:, n0:n0 + r], y_ref, bound, f"stacked {fmt} M={M}")
            n0 += r


@pytest.mark.parametrize("fmt", FORMATS)
def test_tc5_output_guard_bands_untouched(fmt, monkeypatch):
    N, K = SMALL[fmt]
    M = 11
    packed, scales, cb = make_case(fmt, N, K, tag="tc5guard")
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    x = torch.from_numpy(make_x(M, K, tag="tc5guard")).cuda()
    pad = 64
    buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[pad:pad + M * N]
    h.run(x, y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[-pad:] == 12345.0)
    assert not torch.any(y == 12345.0)


@pytest.mark.parametrize("fmt, N, K, Ms", [
    ("q4_0", 8192, 28672, (9, 16)),
    ("pq2_0", 8192, 28672, (1, 16)),
    ("cbk4", 8192, 28672, (16,)),
    ("cbk8", 32000, 4096, (16,)),
    ("pq2_0", 34816, 5120, (8,)),
])
def test_tc5_full_size_sampled_rows(fmt, N, K, Ms, monkeypatch):
    packed, scales, cb = make_case(fmt, N, K, tag="tc5full")
    h = tc5_handle(monkeypatch, fmt, N, K, packed, scales, cb)
    g = np.random.default_rng(0)
    rows = np.array(sorted(set([0, 1, 127, 128, N // 2, N - 129, N - 1] + g.integers(0, N, 40).tolist())))
    for M in Ms:
        x = make_x(M, K, tag="tc5full")
        y = gemv_checked(h, x)[:, rows]
        y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x, rows=rows)
        assert_within(y, y_ref, bound, f"{fmt} {N}x{K} M={M}")


def test_tc5_lost_cta_times_out_and_context_survives(monkeypatch):
    """QGEMV_FAULT_SKIP_CTA on the tensor-memory kernel: the CTAs sharing the
    skipped CTA's row tiles give up their bounded waits, the status reports
    the timeout, and a normal handle then computes correctly (made on the
    host; nothing traps or hangs)."""
    import time
    N, K = 128, 65536
    packed, scales, cb = make_case("q4_0", N, K, tag="tc5fault")
    x_np = make_x(16, K, tag="tc5fault")
    x = torch.from_numpy(x_np).cuda()
    monkeypatch.setenv("QGEMV_FAULT_SKIP_CTA", "0")
    bad = tc5_handle(monkeypatch, "q4_0", N, K, packed, scales, cb)
    monkeypatch.delenv("QGEMV_FAULT_SKIP_CTA")
    good = tc5_handle(monkeypatch, "q4_0", N, K, packed, scales, cb)
    t0 = time.time()
    bad.gemv(x)
    with pytest.raises(qgemv.QgemvError) as err:
        bad.status()
    assert err.value.code == qgemv.QGEMV_ERR_TIMEOUT
    assert time.time() - t0 < 60
    y = gemv_checked(good, x_np)
    y_ref, bound = oracle.gemv("q4_0", N, K, packed, scales, cb, x_np)
    assert_within(y, y_ref, bound, "after a timeout")
