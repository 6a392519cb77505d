"""GPU parity of qgemv_run_residual (y = residual + x . W^T, the residual add
of the attention-output and MLP-down projections done in the GEMV's store).

Bars:
  * against the fp64 oracle: |y - y_ref| <= 1e-3 * sum |x w| + 1e-6 plus one
    fp32 rounding of the sum;
  * against qgemv_run on the same handle: bit for bit fl32(y_plain + r);
  * in place (residual is y): identical to the separate-buffer call;
  * argument errors: NULL or misaligned residual.
Every kernel family is covered: M = 1 (CUDA-core kernel, AQLM table pass),
M = 3 and 8 (tensor-core kernel, AQLM tensor-core layout), M = 16 (two
activation blocks), on shapes with split row tiles and ragged tails.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FORMATS = ["q4_0", "pq2_0", "cbk4", "cbk8", "aqlm_2x8"]
SHAPES = {"q4_0": (700, 2048), "pq2_0": (700, 2304), "cbk4": (700, 2050), "cbk8": (700, 1025),
          "aqlm_2x8": (2100, 2056)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def _residual(M, N, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((M, N)) * 4.0).astype(np.float32)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_residual_matches_oracle_and_plain_run(fmt, M):
    N, K = SHAPES[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="residual")
    x_np = make_x(M, K, tag="residual")
    r_np = _residual(M, N, seed=100 + M)
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    x = torch.from_numpy(x_np).cuda()
    r = torch.from_numpy(r_np).cuda()
    y_plain = h.gemv(x)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    h.run_residual(x, y, r)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    # bit for bit: the plain result plus the residual in one fp32 add
    assert torch.equal(y, y_plain + r), f"{fmt} M={M}: not fl32(qgemv_run + residual)"
    y_ref, bound = oracle.gemv_residual(fmt, N, K, packed, scales, cb, x_np, r_np)
    ok = oracle.within_tolerance_residual(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{fmt} M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"
    # in place: residual is y itself
    y_in = r.clone()
    h.run_residual(x, y_in, y_in)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y_in, y), f"{fmt} M={M}: in-place result differs"


def test_residual_argument_errors():
    N, K = 256, 256
    packed, scales, cb = make_case("cbk4", N, K, tag="residual_args")
    h = qgemv.QGemv("cbk4", N, K, packed, scales, cb)
    x = torch.zeros((1, K), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    lib = qgemv.load()
    assert lib.qgemv_run_residual(h.handle, x.data_ptr(), 1, y.data_ptr(), None, None) == qgemv.QGEMV_ERR_ARG
    buf = torch.zeros(N + 1, dtype=torch.float32, device="cuda")
    bad = buf.data_ptr() + 2  # 2-byte offset: not 4-byte aligned
    assert lib.qgemv_run_residual(h.handle, x.data_ptr(), 1, y.data_ptr(), bad, None) == qgemv.QGEMV_ERR_ALIGN
    torch.cuda.synchronize()


def test_residual_in_stacked_handle():
    """A stacked handle (q|k|v-style) with a residual over its whole output."""
    K = 1024
    seg = [256, 128, 77]
    N = sum(seg)
    packed, _, cb = make_case("cbk4", N, K, tag="residual_stacked")
    codebooks = np.concatenate([cb] * len(seg))
    h = qgemv.QGemv.stacked("cbk4", seg, K, packed, None, codebooks)
    M = 2
    x_np = make_x(M, K, tag="residual_stacked")
    r_np = _residual(M, N, seed=7)
    x = torch.from_numpy(x_np).cuda()
    r = torch.from_numpy(r_np).cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    h.run_residual(x, y, r)
    y_plain = h.gemv(x)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y, y_plain + r)
