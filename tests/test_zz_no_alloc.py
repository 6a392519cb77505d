"""The allocation-free Q4_0 entry point (qgemv_run_q4_0_noalloc).

It serves callers that cannot allocate device memory at the point where
they need the product: it takes the canonical blocks, x and y from the
caller and keeps its split-K scratch in a fixed static device array.  These
tests call it through the C ABI on two calls in a row and check every output
against the fp64 oracle (|y - y_ref| <= 1e-3 * sum_k |x w| + 1e-6) and
against the regular entry point (a handle made with qgemv_create), within
the same bound.  The shapes cover one K chunk, several whole chunks and a
short last chunk (K not a multiple of the 2048-input chunk: a zero-padded
activation tail and a short partial), at M = 1 to 16.  This file is
collected after every other test, so that a run stopping at the first
failure has already run them.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


@pytest.mark.parametrize("N, K, M", [(300, 800, 1),      # one K chunk: no scratch partials
                                     (2500, 8192, 4),    # four whole chunks
                                     (8192, 4096, 16),   # two chunks, widest M
                                     (4096, 11008, 8),   # six chunks, the last 768 inputs (7B down)
                                     (100, 2080, 3)])    # two chunks, the last 32 inputs
def test_noalloc_matches_oracle_and_regular_entry_point_on_two_calls(N, K, M):
    packed = inputs.q4_0_random_blocks(inputs.rng(f"noalloc/{N}x{K}"), N, K)
    x_np = inputs.x_fp16(inputs.rng(f"noalloc/x/{M}x{K}"), M, K)
    x = torch.from_numpy(x_np).cuda()
    h = qgemv.QGemv("q4_0", N, K, packed)
    y_regular = h.gemv(x)
    packed_dev = torch.from_numpy(packed).cuda()
    y_ref, bound = oracle.gemv("q4_0", N, K, packed, None, None, x_np)
    outs = []
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = qgemv.load().qgemv_run_q4_0_noalloc(packed_dev.data_ptr(), N, K, x.data_ptr(), M,
                                                 y.data_ptr(), None)
        assert rc == qgemv.QGEMV_OK, qgemv.qgemv_last_error()
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy())
    regular = y_regular.cpu().numpy()
    for y in outs:
        ok = oracle.within_tolerance(y, y_ref, bound)
        assert ok.all(), f"{np.count_nonzero(~ok)} outputs out of tolerance against the oracle"
        assert np.all(np.abs(y.astype(np.float64) - regular) <= 1e-3 * bound + 1e-6)
    assert np.array_equal(outs[0], outs[1])


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = qgemv.load()
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 16 chunks x 16 rows of x x 65536 outputs x 4 bytes = 64 MiB > 8 MiB
    rc = lib.qgemv_run_q4_0_noalloc(dummy.data_ptr(), 65536, 32768, dummy.data_ptr(), 16,
                                    dummy.data_ptr(), None)
    assert rc == qgemv.QGEMV_ERR_ARG
    assert "static scratch holds" in qgemv.qgemv_last_error()
