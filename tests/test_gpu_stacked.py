"""GPU parity of stacked handles (several projections sharing K in one
handle, one codebook per segment) against the oracle run per segment."""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv
from cases import make_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def segment_case(fmt, seg_rows, K, tag):
    """Per segment: canonical packed bytes and (CBK) its own codebook."""
    packs, cbs = [], []
    for s, rows in enumerate(seg_rows):
        g = inputs.rng(f"{tag}/{fmt}/{s}/{rows}x{K}")
        if fmt in ("cbk4", "cbk8"):
            L = 16 if fmt == "cbk4" else 256
            base = inputs.cbk_centroids(L)
            # a different (still fp16-exact, increasing) codebook per segment
            cb = (base.astype(np.float32) * np.float32(1.0 + 0.25 * s)).astype(np.float16)
            packs.append(inputs.cbk_packed(g, rows, K, 4 if L == 16 else 8, inputs.cbk_cell_probs(base)))
            cbs.append(cb)
        elif fmt == "q4_0":
            packs.append(inputs.q4_0_random_blocks(g, rows, K))
        else:
            packs.append(inputs.pq2_packed(g, rows, K))
    return packs, cbs


def oracle_stacked(fmt, seg_rows, K, packs, cbs, x):
    ys, bs = [], []
    for s, rows in enumerate(seg_rows):
        y, b = oracle.gemv(fmt, rows, K, packs[s], None, cbs[s] if cbs else None, x)
        ys.append(y)
        bs.append(b)
    return np.concatenate(ys, axis=1), np.concatenate(bs, axis=1)


def make_handle(fmt, seg_rows, K, packs, cbs):
    packed = np.concatenate(packs, axis=0)
    cb = np.concatenate(cbs) if cbs else None
    return qgemv.QGemv.stacked(fmt, seg_rows, K, packed, None, cb)


CASES = [
    ("cbk4", [256, 384, 300], 1024),      # ragged last segment
    ("cbk4", [128] * 20 + [77], 8192),     # CTA runs cross many segment boundaries
    ("cbk8", [512, 256], 777),
    ("cbk8", [128, 128, 128, 5], 4096),
    ("q4_0", [384, 200], 2048),            # plain concatenation formats
    ("pq2_0", [256, 129], 2048),
]


@pytest.mark.parametrize("fmt, seg_rows, K", CASES)
@pytest.mark.parametrize("M", [1, 3, 16])
def test_stacked_gemv_matches_oracle_per_segment(fmt, seg_rows, K, M):
    packs, cbs = segment_case(fmt, seg_rows, K, "stk")
    h = make_handle(fmt, seg_rows, K, packs, cbs)
    x = make_x(M, K, tag="stk")
    y = h.gemv(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y_ref, bound = oracle_stacked(fmt, seg_rows, K, packs, cbs, x)
    ok = oracle.within_tolerance(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"{np.count_nonzero(~ok)} outputs out of tolerance"


@pytest.mark.parametrize("fmt, seg_rows, K", CASES[:4])
def test_stacked_dequant_bit_exact(fmt, seg_rows, K):
    packs, cbs = segment_case(fmt, seg_rows, K, "stkdq")
    h = make_handle(fmt, seg_rows, K, packs, cbs)
    w = h.dequant().cpu().numpy()
    ref = np.concatenate([oracle.dequant(fmt, r, K, packs[s], None, cbs[s])
                          for s, r in enumerate(seg_rows)], axis=0)
    assert np.array_equal(w, ref.astype(np.float32))


def test_stacked_one_hot_columns_bit_exact():
    seg_rows, K = [128, 256, 100], 640
    packs, cbs = segment_case("cbk4", seg_rows, K, "stkoh")
    h = make_handle("cbk4", seg_rows, K, packs, cbs)
    cols = [0, 1, 63, 64, 511, 512, 639]
    x = np.zeros((len(cols), K), dtype=np.float16)
    for i, k in enumerate(cols):
        x[i, k] = 1.0
    y = h.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    W = np.concatenate([oracle.dequant("cbk4", r, K, packs[s], None, cbs[s])
                        for s, r in enumerate(seg_rows)], axis=0)
    for i, k in enumerate(cols):
        assert np.array_equal(y[i], W[:, k].astype(np.float32)), f"column {k}"


def test_stacked_rejects_bad_segments():
    K = 256
    g = inputs.rng("stkbad")
    packed = inputs.cbk_packed(g, 300, K, 4, inputs.cbk_cell_probs(inputs.cbk_centroids(16)))
    cb = np.concatenate([inputs.cbk_centroids(16)] * 2)
    with pytest.raises(qgemv.QgemvError, match="multiple of 128"):
        qgemv.QGemv.stacked("cbk4", [100, 200], K, packed, None, cb)
