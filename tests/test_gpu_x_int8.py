"""GPU parity of the PQ2_0 integer path (INT8 activations, qgemv_set_x_int8)
and of its activation quantizer (qgemv_quantize_x_int8), against the
oracle's ``quantize_x_int8`` / ``gemv_pq2_int8``.

Bars:
  * quantizer: codes and scales bit for bit the oracle's (both sides decide
    every code with the same IEEE fp32 divisions and ties-to-even rounding);
  * GEMV: |y - y_ref| <= 1e-3 * B + 1e-6 per output, y_ref the exact value of
    the integer path (fp64) and B its sum of |terms|;
  * activations on the INT8 grid: the integer path meets the same bound
    against the exact (non-quantized) PQ2_0 GEMV;
  * every row is computed alone, so a row's bits do not depend on M;
  * the residual form is fl32(plain + residual), bit for bit;
  * the mode is refused for other formats and switching it off restores the
    exact path bit for bit.
Prepared activations (qgemv_prepare_x_int8, with and without the fused
Hadamard mixing of blocks of 1024): codes, scales and code sums bit for bit
the oracle's ``prepare_x_int8``; qgemv_run_xq within the bound of the
oracle's integer GEMV on those codes, and without mixing bit for bit the
INT8-mode qgemv_run.
Shapes cover ragged row and k tails, split row tiles and the full-size
5120 / 17408 PQ2_0 projections (gate+up 34816 x 5120, down 5120 x 17408).
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv
from cases import make_case, make_x, unpack_xq

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.late]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def _special_x(M, K, tag):
    """Seeded activations with a zero group, a scale-1 group holding ties, and
    a group of tiny values (fp16 subnormals among them)."""
    x = make_x(M, K, tag=tag)
    x[0, 128:256] = 0
    if K >= 384:
        x[M - 1, 256:384] = 0
        x[M - 1, 256:264] = [127.0, 2.5, 3.5, -2.5, -0.5, 1.5, -126.5, 0.25]
    if K >= 512:
        x[0, 384:512] = (x[0, 384:512].astype(np.float32) * np.float32(1e-5)).astype(np.float16)
    return x


@pytest.mark.parametrize("M,K", [(1, 128), (3, 2304), (2, 5120), (4, 17408)])
def test_quantizer_matches_oracle_bit_for_bit(M, K):
    x_np = _special_x(M, K, tag="i8q")
    q, a = qgemv.quantize_x_int8(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    qo, ao = oracle.quantize_x_int8(x_np)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ao.view(np.uint32))


@pytest.mark.parametrize("N,K", [(300, 1280), (700, 2304), (5120, 17408), (34816, 5120)])
def test_int8_gemv_matches_oracle(N, K):
    if N * K > (1 << 24):  # full sizes: drawn on the device, the same bytes fed to both sides
        packed_dev = inputs.pq2_packed_cuda(f"i8/{N}x{K}", N, K)
        packed = packed_dev.cpu().numpy()
        h = qgemv.QGemv("pq2_0", N, K, packed_dev)
        del packed_dev
    else:
        packed, _, _ = make_case("pq2_0", N, K, tag="i8")
        h = qgemv.QGemv("pq2_0", N, K, packed)
    x_np = _special_x(1, K, tag="i8")
    h.set_x_int8(True)
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y_ref, bound = oracle.gemv_pq2_int8(N, K, packed, x_np)
    ok = oracle.within_tolerance(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{N}x{K}: {np.count_nonzero(~ok)} outputs out of tolerance"


def test_int8_on_grid_activations_reach_the_exact_gemv():
    N, K = 700, 2304
    packed, _, _ = make_case("pq2_0", N, K, tag="i8grid")
    g = np.random.default_rng(11)
    q = g.integers(-127, 128, size=(2, K))
    q[:, ::128] = 127
    x_np = (q * 2.0 ** -7).astype(np.float16)
    h = qgemv.QGemv("pq2_0", N, K, packed)
    h.set_x_int8(True)
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    y_ref, bound = oracle.gemv("pq2_0", N, K, packed, None, None, x_np)
    assert oracle.within_tolerance(y.cpu().numpy(), y_ref, bound).all()


@pytest.mark.parametrize("M", [2, 3, 5, 16])
@pytest.mark.parametrize("inv", [False, True])
def test_int8_rows_do_not_depend_on_M(M, inv):
    """Up to three rows run the CUDA-core kernel (every row alone, the same
    instructions in every instantiation); four or more the tensor-core
    kernel, which computes every row as its own MMA column in one order.  So
    a row's bits are the same in every call on the same kernel; across the
    two they may differ within the bound, unless batch-invariant mode puts
    every M on the tensor-core kernel."""
    N, K = 700, 2304
    packed, _, _ = make_case("pq2_0", N, K, tag="i8m")
    x_np = make_x(M, K, tag="i8m")
    h = qgemv.QGemv("pq2_0", N, K, packed)
    h.set_x_int8(True)
    if inv:
        h.set_batch_invariant(True)
    x = torch.from_numpy(x_np).cuda()
    y = h.gemv(x)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y_ref, bound = oracle.gemv_pq2_int8(N, K, packed, x_np)
    assert oracle.within_tolerance(y.cpu().numpy(), y_ref, bound).all()
    for m in sorted({0, M // 2, M - 1}):
        y4 = h.gemv(x[[m, m, m, m]])  # the tensor-core kernel
        y1 = h.gemv(x[m:m + 1])       # the CUDA-core kernel (tensor-core in batch-invariant mode)
        torch.cuda.synchronize()
        y1_ref, b1 = oracle.gemv_pq2_int8(N, K, packed, x_np[m:m + 1])
        assert oracle.within_tolerance(y1.cpu().numpy(), y1_ref, b1).all()
        assert oracle.within_tolerance(y4.cpu().numpy(), np.repeat(y1_ref, 4, axis=0), np.repeat(b1, 4, axis=0)).all()
        same = y4 if (M >= 4 or inv) else y1
        assert torch.equal(same[0], y[m]), f"row {m} of M={M} differs from the same kernel's other call"
        if inv:
            assert torch.equal(y1[0], y[m]) and torch.equal(y4[0], y[m])


@pytest.mark.parametrize("N,K", [(300, 1280), (5120, 17408), (34816, 5120)])
@pytest.mark.parametrize("M", [3, 8, 9, 16])
def test_int8_tensor_core_rows_match_oracle(N, K, M):
    """Several activation rows: the prologue and the INT8 tensor-core kernel,
    at ragged and full sizes, against the exact integer-path value."""
    if N * K > (1 << 24):
        packed_dev = inputs.pq2_packed_cuda(f"i8tc/{N}x{K}", N, K)
        packed = packed_dev.cpu().numpy()
        h = qgemv.QGemv("pq2_0", N, K, packed_dev)
        del packed_dev
        rows = np.unique(np.concatenate([[0, 1, 127, 128, N // 2, N - 1],
                                         np.random.default_rng(3).integers(0, N, 40)]))
    else:
        packed, _, _ = make_case("pq2_0", N, K, tag="i8tc")
        h = qgemv.QGemv("pq2_0", N, K, packed)
        rows = None
    x_np = _special_x(M, K, tag="i8tc")
    h.set_x_int8(True)
    y = h.gemv(torch.from_numpy(x_np).cuda()).cpu().numpy()
    assert h.status() == qgemv.QGEMV_OK
    if rows is not None:
        y = y[:, rows]
        y_ref, bound = oracle.gemv_pq2_int8(rows.size, K, packed.reshape(N, -1)[rows], x_np)
    else:
        y_ref, bound = oracle.gemv_pq2_int8(N, K, packed, x_np)
    ok = oracle.within_tolerance(y, y_ref, bound)
    assert ok.all(), f"{N}x{K} M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"


def test_int8_residual_is_plain_plus_residual():
    N, K, M = 700, 2304, 3
    packed, _, _ = make_case("pq2_0", N, K, tag="i8r")
    x = torch.from_numpy(make_x(M, K, tag="i8r")).cuda()
    r = torch.from_numpy(np.random.default_rng(5).standard_normal((M, N)).astype(np.float32)).cuda()
    h = qgemv.QGemv("pq2_0", N, K, packed)
    h.set_x_int8(True)
    y_plain = h.gemv(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run_residual(x, y, r)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y, y_plain + r)


def test_int8_stacked_handle():
    K = 1280
    seg = [256, 130]
    N = sum(seg)
    packed, _, _ = make_case("pq2_0", N, K, tag="i8s")
    x_np = make_x(1, K, tag="i8s")
    h = qgemv.QGemv.stacked("pq2_0", seg, K, packed)
    h.set_x_int8(True)
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    y_ref, bound = oracle.gemv_pq2_int8(N, K, packed, x_np)
    assert oracle.within_tolerance(y.cpu().numpy(), y_ref, bound).all()


def test_int8_mode_switch_and_refusal():
    N, K = 300, 1280
    packed, _, cb = make_case("cbk4", N, K, tag="i8refuse")
    hc = qgemv.QGemv("cbk4", N, K, packed, None, cb)
    with pytest.raises(qgemv.QgemvError) as e:
        hc.set_x_int8(True)
    assert e.value.code == qgemv.QGEMV_ERR_ARG

    packed, _, _ = make_case("pq2_0", N, K, tag="i8switch")
    x_np = make_x(1, K, tag="i8switch")
    x = torch.from_numpy(x_np).cuda()
    h = qgemv.QGemv("pq2_0", N, K, packed)
    y_exact = h.gemv(x)
    h.set_x_int8(True)
    y_i8 = h.gemv(x)
    h.set_x_int8(False)
    y_back = h.gemv(x)
    torch.cuda.synchronize()
    assert torch.equal(y_back, y_exact)
    assert not torch.equal(y_i8, y_exact)  # quantized activations: a different (lossy) value
    y_ref, bound = oracle.gemv("pq2_0", N, K, packed, None, None, x_np)
    assert oracle.within_tolerance(y_exact.cpu().numpy(), y_ref, bound).all()


def test_quantizer_argument_errors():
    lib = qgemv.load()
    x = torch.zeros((1, 256), dtype=torch.float16, device="cuda")
    q = torch.zeros((1, 256), dtype=torch.int8, device="cuda")
    a = torch.zeros((1, 2), dtype=torch.float32, device="cuda")
    assert lib.qgemv_quantize_x_int8(x.data_ptr(), 1, 200, q.data_ptr(), a.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_quantize_x_int8(x.data_ptr(), 0, 256, q.data_ptr(), a.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_quantize_x_int8(None, 1, 256, q.data_ptr(), a.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    torch.cuda.synchronize()


def _signs(K, B):
    return np.random.default_rng(K).choice([-1, 1], size=K).astype(np.int8) if B else None


def _pq2_handle(N, K, tag):
    if N * K > (1 << 24):
        packed_dev = inputs.pq2_packed_cuda(f"{tag}/{N}x{K}", N, K)
        packed = packed_dev.cpu().numpy()
        return qgemv.QGemv("pq2_0", N, K, packed_dev), packed
    packed, _, _ = make_case("pq2_0", N, K, tag=tag)
    return qgemv.QGemv("pq2_0", N, K, packed), packed


@pytest.mark.parametrize("B", [0, 1024])
@pytest.mark.parametrize("M,K", [(1, 1024), (3, 5120), (2, 17408)])
def test_prepared_activations_match_oracle(B, M, K):
    x_np = _special_x(M, K, tag="i8p")
    signs = _signs(K, B)
    xq = qgemv.prepare_x_int8(torch.from_numpy(x_np).cuda(), B,
                              None if signs is None else torch.from_numpy(signs).cuda())
    torch.cuda.synchronize()
    q, a, qs = unpack_xq(xq, M, K)
    qo, ao = oracle.prepare_x_int8(x_np, B, signs)
    assert np.array_equal(q, qo)
    assert np.array_equal(a.view(np.uint32), ao.view(np.uint32))
    assert np.array_equal(qs, qo.reshape(M, K // 128, 128).sum(axis=2, dtype=np.int64))


@pytest.mark.parametrize("B", [0, 1024])
@pytest.mark.parametrize("N,K,M", [(700, 2048, 1), (5120, 17408, 1), (34816, 5120, 2), (700, 3072, 5),
                                   (700, 3072, 16)])
def test_run_xq_matches_oracle(B, N, K, M):
    h, packed = _pq2_handle(N, K, "i8xq")
    x_np = make_x(M, K, tag="i8xq")
    signs = _signs(K, B)
    x = torch.from_numpy(x_np).cuda()
    xq = qgemv.prepare_x_int8(x, B, None if signs is None else torch.from_numpy(signs).cuda())
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run_xq(xq, M, y)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    q, a = oracle.prepare_x_int8(x_np, B, signs)
    y_ref, bound = oracle.gemv_pq2_int8_q(N, K, packed, q, a)
    ok = oracle.within_tolerance(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{N}x{K} M={M} B={B}: {np.count_nonzero(~ok)} outputs out of tolerance"
    if B == 0:  # the same codes and arithmetic as the INT8 mode of qgemv_run
        h.set_x_int8(True)
        y2 = h.gemv(x)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)


def test_run_xq_residual_and_refusals():
    N, K, M = 700, 2048, 3
    h, _ = _pq2_handle(N, K, "i8xqr")
    x = torch.from_numpy(make_x(M, K, tag="i8xqr")).cuda()
    xq = qgemv.prepare_x_int8(x, 1024, None)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run_xq(xq, M, y)
    r = torch.from_numpy(np.random.default_rng(6).standard_normal((M, N)).astype(np.float32)).cuda()
    yr = torch.empty_like(y)
    h.run_xq(xq, M, yr, residual=r)
    torch.cuda.synchronize()
    assert torch.equal(yr, y + r)

    lib = qgemv.load()
    packed, _, cb = make_case("cbk4", N, K, tag="i8xqrefuse")
    hc = qgemv.QGemv("cbk4", N, K, packed, None, cb)
    assert lib.qgemv_run_xq(hc.handle, xq.data_ptr(), M, y.data_ptr(), None, None) == qgemv.QGEMV_ERR_ARG
    s = torch.ones(K, dtype=torch.int8, device="cuda")
    assert lib.qgemv_prepare_x_int8(x.data_ptr(), M, K, None, 512, xq.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_prepare_x_int8(x.data_ptr(), M, K, s.data_ptr(), 0, xq.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_prepare_x_int8(x.data_ptr(), M, 1280, None, 1024, xq.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert qgemv.qgemv_xq_bytes(M, K) == M * K + 8 * M * (K // 128)
    assert qgemv.qgemv_xq_bytes(M, 100) == 0
    torch.cuda.synchronize()
