"""Batch-invariant mode (qgemv_set_batch_invariant): a row's output bits do
not depend on how many rows share the call, nor on the row's position in
the batch.  Checked on shapes with several tiles per CTA and row tiles split
between CTAs, so the split-K fix-up is part of what must not change."""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = {"q4_0": (2500, 8192), "pq2_0": (2500, 16384), "cbk4": (2500, 8192), "cbk8": (2500, 4096),
          "aqlm_2x8": (4500, 16384)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


@pytest.mark.parametrize("fmt", sorted(SHAPES))
def test_row_bits_do_not_depend_on_m_or_position(fmt):
    N, K = SHAPES[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="invariant")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    h.set_batch_invariant(True)
    x_np = make_x(16, K, tag="invariant")
    x = torch.from_numpy(x_np).cuda()
    y16 = h.gemv(x)
    for M in range(1, 16):
        yM = h.gemv(x[:M].contiguous())
        assert torch.equal(yM, y16[:M]), f"{fmt}: rows of an M={M} call differ from the M=16 call"
    # the same rows in reverse order: each row's bits follow it
    y_rev = h.gemv(x.flip(0).contiguous())
    assert torch.equal(y_rev.flip(0), y16), f"{fmt}: a row's bits depend on its position"
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    # and the invariant results are still within the accuracy bound
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x_np[:2])
    assert oracle.within_tolerance(y16[:2].cpu().numpy(), y_ref, bound).all()


@pytest.mark.parametrize("fmt", ["q4_0", "cbk4"])
def test_mode_switch_applies_to_later_runs(fmt):
    N, K = SHAPES[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="invariant")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    x = torch.from_numpy(make_x(4, K, tag="invariant")).cuda()
    y1_fast = h.gemv(x[:1].contiguous())
    h.set_batch_invariant(True)
    y1_inv = h.gemv(x[:1].contiguous())
    y4 = h.gemv(x)
    assert torch.equal(y1_inv, y4[:1])
    h.set_batch_invariant(False)
    assert torch.equal(h.gemv(x[:1].contiguous()), y1_fast)   # each mode is reproducible
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
