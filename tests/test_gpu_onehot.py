"""One-hot activations read single columns of W out of every GEMV kernel the
dispatcher can pick at M = 1 and M = 2 (and the M = 3..8 tensor-core
geometries), bit for bit.

With x = e_k every output is one weight times one: y[n] = w[n][k], the exact
decoded value (rounded once to fp32 for AQLM 2x8, whose s * (c0 + c1) can
need 36 bits).  So these calls pin each kernel's *own* decode -- the
subnormal-field trick and block-sum offsets of the CUDA-core Q4_0 / PQ2_0
kernel, the lane-replicated tables of CBK4 / CBK8, the row-group kernel, the
AQLM table and tensor-core paths, the per-row codebook kernels, AQLM 1x16,
the INT8 path and the fused SiLU(gate) * up epilogue -- and not only the
separate decoder behind qgemv_dequant.  A wrong centroid, nibble order or
sign in a rarely hit code changes a whole column, however small it is
against the GEMV tolerance.

Columns sit at block, slice, tile and ragged-tail boundaries; the checks
assert that the chosen columns' weights use every code of the format (all
16 Q4_0 nibbles and CBK4 indices, all 4 PQ2_0 codes including +2, all 256
CBK8 indices and AQLM codes).  Rows of a call beyond the one-hots are zero
activations and must give exactly zero.  Shapes span several row and k
tiles with ragged tails, with row tiles shared between CTAs (stream-K) and
owned whole.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv
from cases import make_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KT = {"q4_0": 512, "pq2_0": 1024, "cbk4": 512, "cbk8": 256, "aqlm_2x8": 128, "cbk4_row": 512,
      "cbk8_row": 256, "aqlm_1x16": 128}
# (N, K): three row tiles with a ragged tail and k tiles with a ragged tail;
# then a shape with more tiles than fit one per CTA on some grids
SHAPES = {
    "q4_0": [(300, 1120), (1000, 8192)],
    "pq2_0": [(300, 2176), (1000, 16384)],
    "cbk4": [(300, 1090), (1000, 8192)],
    "cbk8": [(300, 777), (1000, 4096)],
    "aqlm_2x8": [(300, 808), (2500, 4096)],
    "cbk4_row": [(300, 1090), (1000, 8192)],
    "cbk8_row": [(300, 777), (1000, 4096)],
    "aqlm_1x16": [(300, 808), (1000, 4096)],
}
CODES = {"q4_0": 16, "pq2_0": 4, "cbk4": 16, "cbk8": 256, "aqlm_2x8": 256}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def columns(fmt, K, seed=0):
    """Boundary columns of blocks (8 / 32 / 128), slices, tiles and the tail,
    plus a few seeded ones."""
    kt = KT[fmt]
    base = [0, 1, 2, 3, 4, 7, 8, 15, 16, 17, 31, 32, 33, 63, 64, 95, 127, 128, 129, 255, 256,
            kt - 1, kt, kt + 1, 2 * kt - 1, 2 * kt, K // 2, K // 2 + 5, K - 33, K - 32, K - 9, K - 8,
            K - 2, K - 1]
    g = np.random.default_rng(seed)
    base += g.integers(0, K, size=12).tolist()
    return sorted({c for c in base if 0 <= c < K})


def case_with_all_codes(fmt, N, K, tag):
    """Canonical inputs; for PQ2_0 a tenth of the code bytes are redrawn
    uniformly so that code 3 (+2 d), which the workload never draws, occurs."""
    packed, scales, cb = make_case(fmt, N, K, tag=tag)
    if fmt == "pq2_0":
        packed = packed.copy()
        blk = packed.reshape(N, K // 128, 34)
        g = inputs.rng(f"{tag}/pq2_code3")
        sel = g.random((N, K // 128, 32)) < 0.1
        qs = blk[:, :, 2:]
        qs[sel] = g.integers(0, 256, size=int(sel.sum()), dtype=np.uint8)
        packed = blk.reshape(N, -1)
    return packed, scales, cb


def codes_of_columns(fmt, N, K, packed, cols):
    """The code of every weight in the chosen columns (test-side unpacking of
    the canonical bytes, only to check that every code is exercised)."""
    cols = np.asarray(cols)
    if fmt == "q4_0":
        b = packed.reshape(N, K // 32, 18)[:, cols // 32, 2:]
        i = cols % 32
        byte = b[:, np.arange(len(cols)), i % 16]
        return np.where(i < 16, byte & 15, byte >> 4)
    if fmt == "pq2_0":
        b = packed.reshape(N, K // 128, 34)[:, cols // 128, 2:]
        e = cols % 128
        byte = b[:, np.arange(len(cols)), e >> 2]
        return (byte >> (2 * (e & 3))) & 3
    if fmt == "cbk4":
        byte = packed.reshape(N, K // 2)[:, cols // 2]
        return np.where(cols % 2 == 0, byte & 15, byte >> 4)
    if fmt == "cbk8":
        return packed.reshape(N, K)[:, cols]
    if fmt == "aqlm_2x8":
        return packed.reshape(N, K // 8, 2)[:, cols // 8, :]
    raise ValueError(fmt)


def run_onehot(h, N, K, cols, M, value=1.0, x_int8_prepared=False):
    """y rows for x = value * e_k, k over cols, M one-hots per call (the last
    call padded with zero rows).  Returns (y [len(cols), N], zero-row
    outputs)."""
    out, zeros = [], []
    for c0 in range(0, len(cols), M):
        chunk = cols[c0:c0 + M]
        x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
        for i, k in enumerate(chunk):
            x[i, k] = value
        if x_int8_prepared:
            xq = qgemv.prepare_x_int8(x)
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            h.run_xq(xq, M, y)
        else:
            y = h.gemv(x)
        torch.cuda.synchronize()
        assert h.status() == qgemv.QGEMV_OK
        y = y.cpu().numpy()
        out.append(y[:len(chunk)])
        zeros.append(y[len(chunk):])
    return np.concatenate(out), np.concatenate(zeros)


def check_columns(y, zero_rows, W, cols, what, scale=1.0):
    for i, k in enumerate(cols):
        want = (scale * W[:, k]).astype(np.float32)
        if not np.array_equal(y[i], want):
            bad = np.flatnonzero(y[i] != want)[:4]
            raise AssertionError(f"{what}: column {k} differs at rows {bad.tolist()}: "
                                 f"{y[i][bad].tolist()} vs {want[bad].tolist()}")
    assert np.all(zero_rows == 0.0), f"{what}: zero activations gave nonzero outputs"


# The five headline formats: (label, M, create-time env, batch invariant).
# m1: the M = 1 CUDA-core kernel (AQLM: its table kernel, one row per pass);
# m1_rowgroup: the row-group kernel of the table formats; m2: the M = 2
# kernels (tensor-core NB = 1 with the tile-parity geometry of the table
# formats; AQLM: the two-row table pass); m5: the tensor-core NB = 1 kernels
# at M = 3..8 (AQLM: its tensor-core layout); m1_inv: batch-invariant mode,
# the tensor-core kernel's default geometry at M = 1.
CONFIGS = [("m1", 1, "0", False), ("m1_rowgroup", 1, "1", False), ("m2", 2, "0", False),
           ("m5", 5, "0", False), ("m1_inv", 1, "0", True)]


@pytest.mark.parametrize("fmt", ["q4_0", "pq2_0", "cbk4", "cbk8", "aqlm_2x8"])
@pytest.mark.parametrize("shape", [0, 1])
@pytest.mark.parametrize("label, M, rowgroup, inv", CONFIGS)
def test_one_hot_columns_every_kernel(fmt, shape, label, M, rowgroup, inv, monkeypatch):
    if label == "m1_rowgroup" and fmt not in ("cbk4", "cbk8"):
        pytest.skip("the row-group kernel serves the table formats")
    N, K = SHAPES[fmt][shape]
    packed, scales, cb = case_with_all_codes(fmt, N, K, tag=f"onehot{shape}")
    cols = columns(fmt, K)
    used = np.unique(codes_of_columns(fmt, N, K, packed, cols))
    assert used.size == CODES[fmt], f"the chosen columns use {used.size} of {CODES[fmt]} codes"
    W = oracle.dequant(fmt, N, K, packed, scales, cb)
    monkeypatch.setenv("QGEMV_ROWGROUP", rowgroup)
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    monkeypatch.delenv("QGEMV_ROWGROUP")
    if inv:
        h.set_batch_invariant(True)
    y, z = run_onehot(h, N, K, cols, M)
    check_columns(y, z, W, cols, f"{fmt} {N}x{K} {label}")


@pytest.mark.parametrize("fmt", ["cbk4_row", "cbk8_row", "aqlm_1x16"])
@pytest.mark.parametrize("shape", [0, 1])
@pytest.mark.parametrize("M", [1, 2, 3])
def test_one_hot_columns_next_formats(fmt, shape, M):
    N, K = SHAPES[fmt][shape]
    packed, scales, cb = make_case(fmt, N, K, tag=f"onehot{shape}")
    cols = columns(fmt, K)
    W = oracle.dequant(fmt, N, K, packed, scales, cb)
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    y, z = run_onehot(h, N, K, cols, M)
    check_columns(y, z, W, cols, f"{fmt} {N}x{K} M={M}")


@pytest.mark.parametrize("shape", [0, 1])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("prepared", [False, True])
def test_one_hot_columns_pq2_int8(shape, M, prepared):
    """INT8 activations on the grid: x = 127 e_k makes the group scale
    exactly 1 and the code 127, so y = 127 * w[:, k] exactly (127 (c - 1) d
    has at most 19 significant bits)."""
    N, K = SHAPES["pq2_0"][shape]
    packed, _, _ = case_with_all_codes("pq2_0", N, K, tag=f"onehot{shape}")
    cols = columns("pq2_0", K)
    W = oracle.dequant("pq2_0", N, K, packed)
    h = qgemv.QGemv("pq2_0", N, K, packed)
    h.set_x_int8(True)
    y, z = run_onehot(h, N, K, cols, M, value=127.0, x_int8_prepared=prepared)
    check_columns(y, z, W, cols, f"pq2_0 int8 {N}x{K} M={M}", scale=127.0)


def test_one_hot_columns_stacked_m1(monkeypatch):
    """A stacked CBK4 handle (two codebooks, the table rebuilt where a CTA's
    run crosses into the second projection) through the M = 1 kernel."""
    K = 1090
    rows = [256, 300]
    parts = [make_case("cbk4", r, K, tag=f"onehot/stk{i}") for i, r in enumerate(rows)]
    # the second projection decodes with another codebook (the first one's times 1.5, in fp16)
    cbs = [parts[0][2], (parts[0][2].astype(np.float32) * 1.5).astype(np.float16)]
    packed = np.concatenate([p[0] for p in parts])
    W = np.concatenate([oracle.dequant("cbk4", r, K, p[0], None, c) for r, p, c in zip(rows, parts, cbs)])
    cols = columns("cbk4", K)
    monkeypatch.setenv("QGEMV_ROWGROUP", "0")
    h = qgemv.QGemv.stacked("cbk4", rows, K, packed, None, np.concatenate(cbs))
    monkeypatch.delenv("QGEMV_ROWGROUP")
    y, z = run_onehot(h, sum(rows), K, cols, 1)
    check_columns(y, z, W, cols, "stacked cbk4 M=1")


@pytest.mark.parametrize("fmt", ["q4_0", "pq2_0", "cbk4", "cbk8", "cbk4_row"])
@pytest.mark.parametrize("M", [1, 2])
def test_one_hot_glu_pairs(fmt, M):
    """The fused SiLU(gate) * up handle: with x = e_k its two sums are the
    exact weights g = G[:, k], u = U[:, k], so each output is SiLU(g) * u in
    fp32.  Its decode is the plain CUDA-core kernel's (checked bit for bit
    above); here the check is the pairing of gate and up rows and the
    epilogue, against SiLU(g) * u in fp64 within a few fp32 roundings (the
    device's expf may differ from a correctly rounded one in the last place)."""
    N, K = 704, 2048
    tag = f"onehot/glu/{fmt}"
    pg, _, cg = make_case(fmt, N, K, tag=f"{tag}/gate")  # codebooks: CBK4, CBK8, CBK4_ROW, else None
    pu, _, cu = make_case(fmt, N, K, tag=f"{tag}/up")
    if fmt in ("cbk4", "cbk8"):  # one codebook per matrix: make the up one differ from the gate one
        cu = (cg.astype(np.float32) * np.float32(-0.75)).astype(np.float16)
    G = oracle.dequant(fmt, N, K, pg, None, cg)
    U = oracle.dequant(fmt, N, K, pu, None, cu)
    h = qgemv.QGemv.glu(fmt, N, K, pg, pu, cg, cu)
    cols = columns(fmt, K)
    y, z = run_onehot(h, N, K, cols, M)
    for i, k in enumerate(cols):
        g, u = G[:, k], U[:, k]
        want = oracle.silu(g) * u
        err = np.abs(y[i].astype(np.float64) - want)
        assert np.all(err <= 8 * 2.0 ** -24 * np.abs(want) + 1e-38), f"{fmt} GLU column {k}"
    assert np.all(z == 0.0)
