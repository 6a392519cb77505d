"""Failure detection without a GPU fault.

Both failures are made on the host side through test hooks that the library
reads when a handle is created:
  * QGEMV_FAULT_ALLOC=n fails the n-th device allocation of the create call
    as if the device were out of memory: the call must report
    QGEMV_ERR_NOMEM and release what it had allocated.
  * QGEMV_FAULT_SKIP_CTA=c launches CTA c as a no-op, so the CTAs sharing a
    row tile with it never receive its partial sums.  Their fix-up waits are
    bounded (about 2 s): they give up, set the error word and return, and
    qgemv_status reports QGEMV_ERR_TIMEOUT.  Nothing traps or hangs, and the
    context stays usable: a normal handle computes correctly afterwards.
"""
import time

import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, qgemv
from cases import make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# One row tile split over every CTA: a lost CTA leaves all the others waiting.
SPLIT = {"q4_0": (100, 16384), "pq2_0": (100, 32768), "cbk4": (100, 16384), "cbk8": (100, 8192),
         "aqlm_2x8": (100, 16384)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


@pytest.mark.parametrize("fmt", sorted(SPLIT))
@pytest.mark.parametrize("M", [1, 4])
def test_lost_partial_times_out_and_the_context_stays_usable(fmt, M, monkeypatch):
    N, K = SPLIT[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="fault")
    x_np = make_x(M, K, tag="fault")
    x = torch.from_numpy(x_np).cuda()
    monkeypatch.setenv("QGEMV_ROWGROUP", "0")  # the split-K kernels, whose fix-up waits for the lost CTA
    monkeypatch.setenv("QGEMV_FAULT_SKIP_CTA", "0")
    bad = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    monkeypatch.delenv("QGEMV_FAULT_SKIP_CTA")
    good = qgemv.QGemv(fmt, N, K, packed, scales, cb)

    t0 = time.time()
    bad.gemv(x)
    with pytest.raises(qgemv.QgemvError) as err:
        bad.status()
    assert err.value.code == qgemv.QGEMV_ERR_TIMEOUT
    assert time.time() - t0 < 60
    assert bad.status() == qgemv.QGEMV_OK  # reading the status cleared the word

    y = good.gemv(x)
    torch.cuda.synchronize()
    assert good.status() == qgemv.QGEMV_OK
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x_np)
    assert oracle.within_tolerance(y.cpu().numpy(), y_ref, bound).all()


# CBK4 from host arrays: 7 device allocations (packed and codebook copies,
# tiles, codebook table, partial slots, plans, error word).
@pytest.mark.parametrize("n", range(1, 9))
def test_failed_allocation_is_reported_and_released(n, monkeypatch):
    N, K = 300, 1024
    packed, scales, cb = make_case("cbk4", N, K, tag="alloc")
    monkeypatch.setenv("QGEMV_FAULT_ALLOC", str(n))
    if n <= 7:
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(10):
            with pytest.raises(qgemv.QgemvError) as err:
                qgemv.QGemv("cbk4", N, K, packed, scales, cb)
            assert err.value.code == qgemv.QGEMV_ERR_NOMEM
            assert "out of device memory" in str(err.value)
        free1 = torch.cuda.mem_get_info()[0]
        assert free0 - free1 < 16 << 20, "failed creates leaked device memory"
    else:
        h = qgemv.QGemv("cbk4", N, K, packed, scales, cb)   # only 7 allocations: nothing fails
        x_np = make_x(1, K, tag="alloc")
        y = h.gemv(torch.from_numpy(x_np).cuda())
        torch.cuda.synchronize()
        y_ref, bound = oracle.gemv("cbk4", N, K, packed, scales, cb, x_np)
        assert oracle.within_tolerance(y.cpu().numpy(), y_ref, bound).all()
