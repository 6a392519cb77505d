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


# ------------------------------------------------------------- AQLM 2x8 --
# Segments start on the table kernel's 2048-row blocks; each has its own
# codebook pair and its rows their own scales.

def aqlm_segment_case(seg_rows, K, tag):
    codes, scales, cbs = [], [], []
    for s, rows in enumerate(seg_rows):
        c, sc, cb = inputs.aqlm_inputs(inputs.rng(f"{tag}/aqlm/{s}/{rows}x{K}"), rows, K)
        codes.append(c)
        scales.append(sc)
        cbs.append(cb)
    return codes, scales, cbs


def aqlm_handle(seg_rows, K, codes, scales, cbs):
    return qgemv.QGemv.stacked("aqlm_2x8", seg_rows, K, np.concatenate(codes), np.concatenate(scales),
                               np.concatenate(cbs))


def aqlm_oracle(seg_rows, K, codes, scales, cbs, x):
    ys, bs = [], []
    for s, rows in enumerate(seg_rows):
        y, b = oracle.gemv("aqlm_2x8", rows, K, codes[s], scales[s], cbs[s], x)
        ys.append(y)
        bs.append(b)
    return np.concatenate(ys, axis=1), np.concatenate(bs, axis=1)


def aqlm_dequant_ref(seg_rows, K, codes, scales, cbs):
    return np.concatenate([oracle.dequant("aqlm_2x8", r, K, codes[s], scales[s], cbs[s])
                           for s, r in enumerate(seg_rows)], axis=0)


AQLM_CASES = [
    ([2048, 2048, 700], 1032),       # ragged last segment and last chunk
    ([2048] * 5 + [300], 4096),      # CTA runs cross row blocks of different segments
    ([4096, 2048], 256),             # a segment of two row blocks
]


@pytest.mark.parametrize("seg_rows, K", AQLM_CASES)
@pytest.mark.parametrize("M", [1, 2, 3, 5])
def test_stacked_aqlm_matches_oracle_per_segment(seg_rows, K, M):
    codes, scales, cbs = aqlm_segment_case(seg_rows, K, "stka")
    h = aqlm_handle(seg_rows, K, codes, scales, cbs)
    x = make_x(M, K, tag="stka")
    y = h.gemv(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y_ref, bound = aqlm_oracle(seg_rows, K, codes, scales, cbs, x)
    ok = oracle.within_tolerance(y.cpu().numpy(), y_ref, bound)
    assert ok.all(), f"M={M}: {np.count_nonzero(~ok)} outputs out of tolerance"


@pytest.mark.parametrize("seg_rows, K", AQLM_CASES)
def test_stacked_aqlm_dequant_bit_exact(seg_rows, K):
    codes, scales, cbs = aqlm_segment_case(seg_rows, K, "stkadq")
    h = aqlm_handle(seg_rows, K, codes, scales, cbs)
    w = h.dequant().cpu().numpy()
    ref = aqlm_dequant_ref(seg_rows, K, codes, scales, cbs)
    assert np.array_equal(w, ref.astype(np.float32))  # the exact value rounded once


@pytest.mark.parametrize("per_call", [1, 7])
def test_stacked_aqlm_one_hot_columns_bit_exact(per_call):
    """x = e_k returns column k of the stacked matrix, rounded once to fp32,
    from one-row calls and from calls of several rows (passes of two)."""
    seg_rows, K = [2048, 2048, 513], 1032
    codes, scales, cbs = aqlm_segment_case(seg_rows, K, "stkaoh")
    h = aqlm_handle(seg_rows, K, codes, scales, cbs)
    W = aqlm_dequant_ref(seg_rows, K, codes, scales, cbs)
    cols = [0, 7, 8, 127, 128, 1023, 1024, 1031]
    for i0 in range(0, len(cols), per_call):
        chunk = cols[i0:i0 + per_call]
        x = np.zeros((len(chunk), K), dtype=np.float16)
        for i, k in enumerate(chunk):
            x[i, k] = 1.0
        y = h.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        for i, k in enumerate(chunk):
            assert np.array_equal(y[i], W[:, k].astype(np.float32)), f"column {k}"


def test_stacked_aqlm_batch_invariant_rows():
    seg_rows, K = [2048, 1000], 1032
    codes, scales, cbs = aqlm_segment_case(seg_rows, K, "stkainv")
    h = aqlm_handle(seg_rows, K, codes, scales, cbs)
    h.set_batch_invariant(True)
    x = torch.from_numpy(make_x(9, K, tag="stkainv")).cuda()
    y9 = h.gemv(x)
    for M in (1, 2, 3):
        yM = h.gemv(x[:M])
        torch.cuda.synchronize()
        assert torch.equal(yM, y9[:M]), f"M={M} rows differ from the M=9 call"
    y_ref, bound = aqlm_oracle(seg_rows, K, codes, scales, cbs, x.cpu().numpy())
    assert oracle.within_tolerance(y9.cpu().numpy(), y_ref, bound).all()


def test_stacked_aqlm_rejects_unaligned_segments():
    seg_rows, K = [1024, 1024], 256
    codes, scales, cbs = aqlm_segment_case(seg_rows, K, "stkabad")
    with pytest.raises(qgemv.QgemvError, match="multiple of 2048"):
        aqlm_handle(seg_rows, K, codes, scales, cbs)
