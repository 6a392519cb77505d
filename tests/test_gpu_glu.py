"""GPU parity of the fused MLP gate/up projection (qgemv_create_glu):
y = SiLU(x . G^T) * (x . U^T) -- Q4_0, PQ2_0, CBK4 and CBK8 in one launch
for every M (the tensor-core kernel from M = 2; CBK4/CBK8 with the gate and
up tables in one table region), CBK4_ROW once per activation row --
against the oracle's ``gemv_glu`` with the bound of ``within_tolerance_glu`` (each GEMV
sum within its own 1e-3 * sum |x w| + 1e-6, propagated through SiLU and the
product, plus a few fp32 roundings).

Covered: Q4_0, PQ2_0, CBK4 and CBK8 (each matrix its own codebook, the up
one different from the gate one) and CBK4_ROW (per-row codebooks
interleaved with their rows); shapes whose row tiles are split between CTAs
(the pair finisher) and owned whole (the epilogue); the 7B MLP's gate/up
11008 x 4096 and the 5120/17408 model's 17408 x 5120 at full size on
sampled outputs; M = 1, 3, 9 and 16 (both activation blocks of the
tensor-core kernel); the dequant of the interleaved rows (two codebooks for
CBK4); and the refusals (AQLM, N not a multiple of 64, residual, INT8 mode).
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.late]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def _pair(fmt, N, K, tag):
    if fmt == "q4_0":
        g = inputs.rng(f"{tag}/gate")
        u = inputs.rng(f"{tag}/up")
        return (oracle.quantize_q4_0(inputs.w_fp32(g, N, K), N, K),
                oracle.quantize_q4_0(inputs.w_fp32(u, N, K), N, K))
    return (make_case(fmt, N, K, tag=f"{tag}/gate")[0], make_case(fmt, N, K, tag=f"{tag}/up")[0])


def _codebooks(fmt, N, K, tag):
    if fmt in ("cbk4", "cbk8"):  # one codebook per matrix, the up one different from the gate one
        cg = make_case(fmt, N, K, tag=f"{tag}/gate")[2]
        return cg, (cg.astype(np.float32) * np.float32(-0.75)).astype(np.float16)
    if fmt != "cbk4_row":
        return None, None
    return make_case(fmt, N, K, tag=f"{tag}/gate")[2], make_case(fmt, N, K, tag=f"{tag}/up")[2]


@pytest.mark.parametrize("fmt", ["q4_0", "pq2_0", "cbk4", "cbk8", "cbk4_row"])
@pytest.mark.parametrize("N,K", [(192, 1024), (704, 2048), (4096, 4096)])
@pytest.mark.parametrize("M", [1, 3, 9, 16])
def test_glu_matches_oracle(fmt, N, K, M):
    tag = f"glu/{fmt}/{N}x{K}"
    pg, pu = _pair(fmt, N, K, tag)
    cg, cu = _codebooks(fmt, N, K, tag)
    h = qgemv.QGemv.glu(fmt, N, K, pg, pu, cg, cu)
    x_np = make_x(M, K, tag="glu")
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert y.shape == (M, N)
    y_ref, g, u, bg, bu = oracle.gemv_glu(fmt, N, K, pg, pu, x_np, codebooks_gate=cg, codebooks_up=cu)
    ok = oracle.within_tolerance_glu(y.cpu().numpy(), g, u, bg, bu)
    assert ok.all(), f"{fmt} {N}x{K} M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"


@pytest.mark.parametrize("fmt,N,K,M", [("q4_0", 11008, 4096, 1), ("pq2_0", 17408, 5120, 1),
                                       ("cbk4", 11008, 4096, 1), ("cbk4", 11008, 4096, 8)])
def test_glu_full_size_sampled(fmt, N, K, M):
    pg, pu = _pair(fmt, N, K, f"glufull/{fmt}")
    cg, cu = _codebooks(fmt, N, K, f"glufull/{fmt}")
    h = qgemv.QGemv.glu(fmt, N, K, pg, pu, cg, cu)
    x_np = make_x(M, K, tag="glufull")
    y = h.gemv(torch.from_numpy(x_np).cuda()).cpu().numpy()
    assert h.status() == qgemv.QGEMV_OK
    rows = np.unique(np.concatenate([[0, 63, 64, 127, N // 2, N - 65, N - 1],
                                     np.random.default_rng(1).integers(0, N, 48)]))
    g, bg = oracle.gemv(fmt, N, K, pg, None, cg, x_np, rows=rows)
    u, bu = oracle.gemv(fmt, N, K, pu, None, cu, x_np, rows=rows)
    ok = oracle.within_tolerance_glu(y[:, rows], g, u, bg, bu)
    assert ok.all(), f"{fmt} {N}x{K}: {np.count_nonzero(~ok)} sampled outputs out of tolerance"


@pytest.mark.parametrize("fmt", ["pq2_0", "cbk4", "cbk8"])
def test_glu_dequant_is_the_interleaved_rows(fmt):
    N, K = 192, 1024
    pg, pu = _pair(fmt, N, K, "gludq")
    cg, cu = _codebooks(fmt, N, K, "gludq")
    h = qgemv.QGemv.glu(fmt, N, K, pg, pu, cg, cu)
    # the handle's N is the output width; its decoded matrix has 2N rows
    w = torch.empty((2 * N, K), dtype=torch.float32, device="cuda")
    qgemv.qgemv_dequant(h.handle, w.data_ptr())
    torch.cuda.synchronize()
    G = oracle.dequant(fmt, N, K, pg, None, cg)
    U = oracle.dequant(fmt, N, K, pu, None, cu)
    inter = np.concatenate([blk for b in range(N // 64) for blk in (G[64 * b:64 * b + 64], U[64 * b:64 * b + 64])])
    assert np.array_equal(w.cpu().numpy().astype(np.float64), inter)


def test_glu_refusals():
    lib = qgemv.load()
    N, K = 192, 1024
    pg, pu = _pair("pq2_0", N, K, "glurefuse")
    packed, _, cb = make_case("cbk4", N, K, tag="glurefuse")
    with pytest.raises(qgemv.QgemvError):  # a codebook format without its codebooks
        qgemv.QGemv.glu("cbk4", N, K, packed, packed)
    ap, asc, acb = make_case("aqlm_2x8", N, K, tag="glurefuse")
    with pytest.raises(qgemv.QgemvError):  # no GLU form
        qgemv.QGemv.glu("aqlm_2x8", N, K, ap, ap)
    with pytest.raises(qgemv.QgemvError):
        qgemv.QGemv.glu("pq2_0", 100, K, pg[:100 * (K // 128) * 34], pu[:100 * (K // 128) * 34])
    h = qgemv.QGemv.glu("pq2_0", N, K, pg, pu)
    x = torch.from_numpy(make_x(1, K, tag="glurefuse")).cuda()
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    r = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    assert lib.qgemv_run_residual(h.handle, x.data_ptr(), 1, y.data_ptr(), r.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_set_x_int8(h.handle, 1) == qgemv.QGEMV_ERR_ARG
    torch.cuda.synchronize()


def test_glu_lost_cta_times_out_and_context_survives(monkeypatch):
    """QGEMV_FAULT_SKIP_CTA: one 128-row tile (64 gate/up pairs) split over
    every CTA, CTA 0 a no-op: the pair finisher's bounded waits give up, the
    status reports the timeout, and a normal GLU handle then computes
    correctly (the failure is made on the host; nothing traps or hangs)."""
    import time
    N, K = 64, 32768
    pg, pu = _pair("pq2_0", N, K, "glufault")
    x_np = make_x(1, K, tag="glufault")
    x = torch.from_numpy(x_np).cuda()
    monkeypatch.setenv("QGEMV_FAULT_SKIP_CTA", "0")
    bad = qgemv.QGemv.glu("pq2_0", N, K, pg, pu)
    monkeypatch.delenv("QGEMV_FAULT_SKIP_CTA")
    good = qgemv.QGemv.glu("pq2_0", N, K, pg, pu)
    t0 = time.time()
    bad.gemv(x)
    with pytest.raises(qgemv.QgemvError) as err:
        bad.status()
    assert err.value.code == qgemv.QGEMV_ERR_TIMEOUT
    assert time.time() - t0 < 60
    y = good.gemv(x)
    torch.cuda.synchronize()
    assert good.status() == qgemv.QGEMV_OK
    y_ref, g, u, bg, bu = oracle.gemv_glu("pq2_0", N, K, pg, pu, x_np)
    assert oracle.within_tolerance_glu(y.cpu().numpy(), g, u, bg, bu).all()
