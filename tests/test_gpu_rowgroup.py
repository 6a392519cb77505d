"""GPU parity of the M = 1 row-group kernel of the table formats (whole
32-row groups per CTA, no split-K finish), forced on and off with the
QGEMV_ROWGROUP create-time hook so that both M = 1 kernels run on the same
shapes: against the fp64 oracle (|y - y_ref| <= 1e-3 * sum |x w| + 1e-6),
run to run bitwise, with a residual, and on a stacked handle whose row
tiles change codebook.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = {
    "cbk4": [(4096, 4096), (700, 2050), (129, 8192), (1, 512), (300, 1024)],
    "cbk8": [(4096, 4096), (700, 1025), (129, 4096), (1, 256), (300, 1024)],
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def _handle(monkeypatch, force, *args, stacked=False):
    monkeypatch.setenv("QGEMV_ROWGROUP", str(force))
    h = qgemv.QGemv.stacked(*args) if stacked else qgemv.QGemv(*args)
    monkeypatch.delenv("QGEMV_ROWGROUP")
    return h


@pytest.mark.parametrize("fmt", sorted(SHAPES))
@pytest.mark.parametrize("shape", range(5))
@pytest.mark.parametrize("force", [1, 0])
def test_rowgroup_matches_oracle(fmt, shape, force, monkeypatch):
    N, K = SHAPES[fmt][shape]
    packed, scales, cb = make_case(fmt, N, K, tag="rowgroup")
    x_np = make_x(1, K, tag="rowgroup")
    h = _handle(monkeypatch, force, fmt, N, K, packed, scales, cb)
    x = torch.from_numpy(x_np).cuda()
    y = h.gemv(x)
    y2 = h.gemv(x)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y, y2), "run to run"
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x_np)
    ok = oracle.within_tolerance(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{fmt} {N}x{K} force={force}: {np.count_nonzero(~ok)} outputs out of tolerance"
    r = torch.from_numpy(np.linspace(-3, 3, N, dtype=np.float32)[None, :]).cuda()
    yr = torch.empty_like(y)
    h.run_residual(x, yr, r)
    torch.cuda.synchronize()
    assert torch.equal(yr, y + r), "residual"


@pytest.mark.parametrize("fmt", sorted(SHAPES))
def test_rowgroup_stacked_codebooks(fmt, monkeypatch):
    K = 2048 if fmt == "cbk4" else 1024
    seg = [256, 128, 384, 77]
    N = sum(seg)
    packed, _, cb = make_case(fmt, N, K, tag="rowgroup_stacked")
    # a different codebook per segment: the centroids negated, scaled and shifted by segment
    cbs = [(cb.astype(np.float32) * (1.0 + 0.5 * s) * (-1.0) ** s).astype(np.float16) for s in range(len(seg))]
    codebooks = np.concatenate(cbs)
    x_np = make_x(1, K, tag="rowgroup_stacked")
    h = _handle(monkeypatch, 1, fmt, seg, K, packed, None, codebooks, stacked=True)
    y = h.gemv(torch.from_numpy(x_np).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y = y.cpu().numpy()
    row = 0
    for s, n in enumerate(seg):
        pk = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8).reshape(N, -1)[row:row + n])
        y_ref, bound = oracle.gemv(fmt, n, K, pk, None, cbs[s], x_np)
        ok = oracle.within_tolerance(y[:, row:row + n], y_ref, bound)
        assert ok.all(), f"segment {s}: {np.count_nonzero(~ok)} outputs out of tolerance"
        row += n
