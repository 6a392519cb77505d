"""GPU parity of CBK4 with per-output-row fp32 codebooks (the pages' own
4-bit file layout) against the oracle's ``cbk4_row`` format.

Bars:
  * dequant: bit for bit the oracle's value (each weight is an fp32
    centroid);
  * GEMV: |y - y_ref| <= 1e-3 * sum |x w| + 1e-6 per output;
  * a row's bits do not depend on M;
  * the residual form is fl32(plain + residual), bit for bit;
  * stacking is refused.
Shapes: ragged rows and k (N = 300, K = 2050), the smallest K, several row
tiles per CTA run (every row tile rebuilds the shared table), and the 7B
gate (11008 x 4096) and down (4096 x 11008) projections at full size on
sampled rows.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.late]

FMT = "cbk4_row"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def _gemv(h, x_np):
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K", [(300, 2050), (129, 2), (700, 4096)])
def test_dequant_bit_exact(N, K):
    packed, _, cb = make_case(FMT, N, K, tag="c4rdq")
    h = qgemv.QGemv(FMT, N, K, packed, None, cb)
    w = h.dequant()
    torch.cuda.synchronize()
    w_ref = oracle.dequant(FMT, N, K, packed, None, cb)
    assert np.array_equal(w.cpu().numpy().astype(np.float64), w_ref)


@pytest.mark.parametrize("N,K", [(300, 2050), (129, 2), (700, 4096), (1000, 1024)])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 11, 16])
def test_gemv_matches_oracle(N, K, M):
    packed, _, cb = make_case(FMT, N, K, tag="c4r")
    h = qgemv.QGemv(FMT, N, K, packed, None, cb)
    x_np = make_x(M, K, tag="c4r")
    y = _gemv(h, x_np)
    y_ref, bound = oracle.gemv(FMT, N, K, packed, None, cb, x_np)
    ok = oracle.within_tolerance(y, y_ref, bound)
    assert ok.all(), f"{N}x{K} M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"


def _sample_rows(N, n=48, seed=0):
    g = np.random.default_rng(seed)
    rows = set([0, 1, 127, 128, N // 2, N - 129, N - 2, N - 1])
    rows.update(g.integers(0, N, size=n).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


@pytest.mark.parametrize("N,K", [(11008, 4096), (4096, 11008)])
def test_full_size_sampled_rows(N, K):
    packed, _, cb = make_case(FMT, N, K, tag="c4rfull")
    h = qgemv.QGemv(FMT, N, K, packed, None, cb)
    rows = _sample_rows(N)
    for M in (1, 8):
        x_np = make_x(M, K, tag="c4rfull")
        y = _gemv(h, x_np)[:, rows]
        y_ref, bound = oracle.gemv(FMT, N, K, packed, None, cb, x_np, rows=rows)
        ok = oracle.within_tolerance(y, y_ref, bound)
        assert ok.all(), f"{N}x{K} M={M}: {np.count_nonzero(~ok)} sampled outputs out of tolerance"


@pytest.mark.parametrize("inv", [True, False])
def test_rows_do_not_depend_on_M(inv):
    """Batch-invariant mode: a row's bits never depend on M.  Otherwise calls
    of eight or more rows run the eight-row launches (another slice order):
    their rows agree among themselves, and with fewer-row calls within the
    bound."""
    N, K = 700, 4096
    packed, _, cb = make_case(FMT, N, K, tag="c4rinv")
    h = qgemv.QGemv(FMT, N, K, packed, None, cb)
    x_np = make_x(16, K, tag="c4rinv")
    x = torch.from_numpy(x_np).cuda()
    if not inv:
        y16 = h.gemv(x)
        y8 = h.gemv(x[8:])
        y3 = h.gemv(x[:3])
        torch.cuda.synchronize()
        assert torch.equal(y8, y16[8:])
        y_ref, bound = oracle.gemv(FMT, N, K, packed, None, cb, x_np)
        assert oracle.within_tolerance(y16.cpu().numpy(), y_ref, bound).all()
        assert oracle.within_tolerance(y3.cpu().numpy(), y_ref[:3], bound[:3]).all()
        return
    h.set_batch_invariant(True)
    y16 = h.gemv(x)
    for M in (1, 2, 3, 5):
        yM = h.gemv(x[:M])
        torch.cuda.synchronize()
        assert torch.equal(yM, y16[:M]), f"M={M} rows differ from the M=16 call"
    y1 = h.gemv(x[11:12])
    torch.cuda.synchronize()
    assert torch.equal(y1[0], y16[11])


def test_residual_is_plain_plus_residual():
    N, K, M = 700, 4096, 3
    packed, _, cb = make_case(FMT, N, K, tag="c4rr")
    h = qgemv.QGemv(FMT, N, K, packed, None, cb)
    x = torch.from_numpy(make_x(M, K, tag="c4rr")).cuda()
    r = torch.from_numpy(np.random.default_rng(3).standard_normal((M, N)).astype(np.float32)).cuda()
    y_plain = h.gemv(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run_residual(x, y, r)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y, y_plain + r)


def test_stacking_is_refused():
    N, K = 256, 64
    packed, _, cb = make_case(FMT, N, K, tag="c4rstack")
    with pytest.raises(qgemv.QgemvError) as e:
        qgemv.QGemv.stacked(FMT, [128, 128], K, packed, None, cb)
    assert e.value.code == qgemv.QGEMV_ERR_ARG
