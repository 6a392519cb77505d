"""GPU parity of AQLM 1x16 (one 65,536 x 8 fp16 codebook gathered from L2,
16-bit codes, fp32 products) against the oracle.

Bars:
  * dequant: bit for bit the oracle's value (s * C[code][j] is exact in fp32);
  * GEMV: |y - y_ref| <= 1e-3 * sum |x w| + 1e-6 per output;
  * a row's bits do not depend on M (one launch reads each code and entry
    once for all rows, and each row's arithmetic is the same for every M);
  * the residual form is fl32(plain + residual), bit for bit;
  * stacking is refused.
Shapes: ragged code vectors (K/8 not a multiple of 8), a single group, x
only 4-byte aligned, more rows than one pass of the grid, and the 70B layer
at full size (gate/up 28672 x 8192, down 8192 x 28672, q/o
8192 x 8192) on sampled rows, at M = 1 and the verify batch M = 16.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.late]

FMT = "aqlm_1x16"


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


@pytest.mark.parametrize("N,K", [(300, 1032), (129, 8), (700, 2056)])
def test_dequant_bit_exact(N, K):
    codes, scales, cb = make_case(FMT, N, K, tag="a16dq")
    h = qgemv.QGemv(FMT, N, K, codes, scales, cb)
    w = h.dequant()
    torch.cuda.synchronize()
    w_ref = oracle.dequant(FMT, N, K, codes, scales, cb)
    assert np.array_equal(w.cpu().numpy().astype(np.float64), w_ref)


@pytest.mark.parametrize("N,K", [(300, 1032), (129, 8), (700, 2056)])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 16])
def test_gemv_matches_oracle(N, K, M):
    codes, scales, cb = make_case(FMT, N, K, tag="a16")
    h = qgemv.QGemv(FMT, N, K, codes, scales, cb)
    x_np = make_x(M, K, tag="a16")
    y = _gemv(h, x_np)
    y_ref, bound = oracle.gemv(FMT, N, K, codes, scales, cb, x_np)
    ok = oracle.within_tolerance(y, y_ref, bound)
    assert ok.all(), f"{N}x{K} M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"


@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_x_only_4_byte_aligned(M):
    """x 4 bytes past a 16-byte boundary (the API's minimum): the activation
    loads (M = 1) and the shared-memory copies (M > 1) take 4-byte pieces."""
    N, K = 300, 2056
    codes, scales, cb = make_case(FMT, N, K, tag="a16al")
    x_np = make_x(M, K, tag="a16al")
    buf = torch.zeros(M * K + 8, dtype=torch.float16, device="cuda")
    x = buf[2:2 + M * K].view(M, K)
    assert x.data_ptr() % 16 == 4
    x.copy_(torch.from_numpy(x_np).cuda())
    h = qgemv.QGemv(FMT, N, K, codes, scales, cb)
    y = h.gemv(x)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y_ref, bound = oracle.gemv(FMT, N, K, codes, scales, cb, x_np)
    ok = oracle.within_tolerance(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"


@pytest.mark.parametrize("M", [1, 3, 8])
def test_rows_beyond_one_pass_of_the_grid(M):
    """More rows than one pass of the largest grid (65,535 CTAs of eight
    warps): CTAs take a second row each, and with M > 1 they copy the next
    rows' first activations while finishing the current ones."""
    N, K = 65535 * 8 + 301, 2064
    codes, scales, cb = make_case(FMT, N, K, tag="a16pass")
    h = qgemv.QGemv(FMT, N, K, codes, scales, cb)
    x_np = make_x(M, K, tag="a16pass")
    y = _gemv(h, x_np)
    rows = np.array(sorted(set([0, 7, 65535 * 8 - 1, 65535 * 8, 65535 * 8 + 7, N - 1] +
                               np.random.default_rng(3).integers(0, N, size=64).tolist())), dtype=np.int64)
    y_ref, bound = oracle.gemv(FMT, N, K, codes, scales, cb, x_np, rows=rows)
    ok = oracle.within_tolerance(y[:, rows], y_ref, bound)
    assert ok.all(), f"M={M}: {np.count_nonzero(~ok)} sampled outputs out of tolerance"


def _sample_rows(N, n=48, seed=0):
    g = np.random.default_rng(seed)
    rows = set([0, 1, 7, 8, N // 2, N - 9, N - 2, N - 1])
    rows.update(g.integers(0, N, size=n).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


@pytest.mark.parametrize("N,K", [(28672, 8192), (8192, 28672), (8192, 8192)])
def test_full_size_sampled_rows(N, K):
    codes_d, scales_d, cb_d = inputs.aqlm_1x16_inputs_cuda(f"a16full/{N}x{K}", N, K)
    h = qgemv.QGemv(FMT, N, K, codes_d, scales_d, cb_d)
    codes = codes_d.cpu().numpy().view(np.uint16)
    scales = scales_d.cpu().numpy()
    cb = cb_d.cpu().numpy()
    del codes_d
    rows = _sample_rows(N)
    for M in (1, 16):
        x_np = make_x(M, K, tag="a16full")
        y = _gemv(h, x_np)[:, rows]
        y_ref, bound = oracle.gemv(FMT, N, K, codes, scales, cb, x_np, rows=rows)
        ok = oracle.within_tolerance(y, y_ref, bound)
        assert ok.all(), f"{N}x{K} M={M}: {np.count_nonzero(~ok)} sampled outputs out of tolerance"


def test_rows_do_not_depend_on_M():
    N, K = 700, 2056
    codes, scales, cb = make_case(FMT, N, K, tag="a16inv")
    h = qgemv.QGemv(FMT, N, K, codes, scales, cb)
    x = torch.from_numpy(make_x(16, K, tag="a16inv")).cuda()
    y16 = h.gemv(x)
    for M in (1, 2, 3, 5, 9):
        yM = h.gemv(x[:M])
        torch.cuda.synchronize()
        assert torch.equal(yM, y16[:M]), f"M={M} rows differ from the M=16 call"
    y1 = h.gemv(x[7:8])
    torch.cuda.synchronize()
    assert torch.equal(y1[0], y16[7])


def test_residual_is_plain_plus_residual():
    N, K, M = 700, 2056, 3
    codes, scales, cb = make_case(FMT, N, K, tag="a16r")
    h = qgemv.QGemv(FMT, N, K, codes, scales, cb)
    x = torch.from_numpy(make_x(M, K, tag="a16r")).cuda()
    r = torch.from_numpy(np.random.default_rng(9).standard_normal((M, N)).astype(np.float32)).cuda()
    y_plain = h.gemv(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run_residual(x, y, r)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y, y_plain + r)


def test_stacking_is_refused():
    N, K = 256, 64
    codes, scales, cb = make_case(FMT, N, K, tag="a16stack")
    with pytest.raises(qgemv.QgemvError) as e:
        qgemv.QGemv.stacked(FMT, [128, 128], K, codes, scales, cb)
    assert e.value.code == qgemv.QGEMV_ERR_ARG
