"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars:
  * decoded weights (qgemv_dequant): bit-exact against the oracle's exact
    values rounded once to fp32 (a no-op except for AQLM, whose scaled sums
    are not all representable);
  * GEMV: |y - y_ref| <= 1e-3 * sum_k |x_k w_nk| + 1e-6 for every output;
  * one-hot x: the matching column of W, bit-exact;
  * run to run and eager vs CUDA graph: bitwise identical;
  * the Q4_0 quantizer: byte-identical to the oracle's quantizer.
Sizes span several row and k tiles with ragged tails; the full workload
sizes are checked on sampled rows.
"""
import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import build, inputs, qgemv
from cases import MIN_K, make_case, make_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FORMATS = ["q4_0", "pq2_0", "cbk4", "cbk8", "aqlm_2x8"]
SMALL = {"q4_0": (300, 800), "pq2_0": (300, 1152), "cbk4": (300, 802), "cbk8": (300, 777),
         "aqlm_2x8": (300, 808)}
# AQLM row blocks are 2048 rows x 128 inputs: 3 x 128 units keep several per CTA.
MULTI = {"q4_0": (2500, 8192), "pq2_0": (2500, 16384), "cbk4": (2500, 8192), "cbk8": (2500, 4096),
         "aqlm_2x8": (4500, 16384)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    qgemv.load()


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_gemv(h: qgemv.QGemv, x_np: np.ndarray) -> np.ndarray:
    x = cuda(x_np)
    y = h.gemv(x)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    return y.cpu().numpy()


def assert_within(y, y_ref, bound, what=""):
    ok = oracle.within_tolerance(y, y_ref, bound)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        details = [(tuple(i), float(y[tuple(i)]), float(y_ref[tuple(i)]), float(bound[tuple(i)]))
                   for i in idx]
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} outputs out of tolerance, e.g. {details}")


# ------------------------------------------------------------ decode ----

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("shape", ["small", "tiny", "edge"])
def test_dequant_bit_exact(fmt, shape):
    N, K = {"small": SMALL[fmt], "tiny": (1, MIN_K[fmt]),
            "edge": (129, MIN_K[fmt] * 9)}[shape]
    packed, scales, cb = make_case(fmt, N, K, tag="dq")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    w = h.dequant().cpu().numpy()
    ref = oracle.dequant(fmt, N, K, packed, scales, cb)
    if fmt != "aqlm_2x8":
        # one scale times a small integer or a centroid: exact in fp32
        assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
    # AQLM's s * (c0 + c1) needs up to 36 significant bits: the decoded fp32
    # weight is the exact value rounded once, to nearest even
    assert np.array_equal(w, ref.astype(np.float32))


# -------------------------------------------------------------- GEMV ----

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", list(range(1, 17)))
def test_gemv_small_all_m(fmt, M):
    N, K = SMALL[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="small")
    x = make_x(M, K, tag="small")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    y = gpu_gemv(h, x)
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
    assert_within(y, y_ref, bound, f"{fmt} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_gemv_many_tiles_per_cta(fmt, M):
    """More tiles than CTAs: CTAs own whole row tiles and share others."""
    N, K = MULTI[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="multi")
    x = make_x(M, K, tag="multi")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    y = gpu_gemv(h, x)
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
    assert_within(y, y_ref, bound, f"{fmt} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("shape", ["multi", "stack_qkv"])
def test_split_runs_match_oracle(fmt, shape, monkeypatch):
    """Each format's stream-K split (spread for Q4_0 and AQLM 2x8, front-loaded
    for the others) on the M = 1 CUDA-core kernel, the M = 2 and the
    two-block tensor-core kernels: the plan made on the host and the runs the
    kernels take agree, and every output is within the bound.  stack_qkv: a
    7B q|k|v-sized shape whose tile count is not a multiple of the grid."""
    N, K = MULTI[fmt] if shape == "multi" else (12288 if fmt != "aqlm_2x8" else 10240, 4096)
    packed, scales, cb = make_case(fmt, N, K, tag=f"split/{shape}")
    monkeypatch.setenv("QGEMV_ROWGROUP", "0")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    monkeypatch.delenv("QGEMV_ROWGROUP")
    for M in (1, 2, 11):
        x = make_x(M, K, tag="split")
        y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
        assert_within(gpu_gemv(h, x), y_ref, bound, f"{fmt} {N}x{K} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N, Kmul", [(1, 1), (1, 7), (127, 2), (128, 3), (129, 5), (4095, 4)])
def test_gemv_edge_shapes(fmt, N, Kmul):
    K = MIN_K[fmt] * Kmul
    packed, scales, cb = make_case(fmt, N, K, tag="edge")
    for M in (1, 16):
        x = make_x(M, K, tag="edge")
        h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
        y = gpu_gemv(h, x)
        y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x)
        assert_within(y, y_ref, bound, f"{fmt} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", [1, 2, 7, 16])
def test_gemv_x_only_4_byte_aligned(fmt, M):
    """x starting 4 bytes past a 16-byte boundary (the API's minimum): the
    activation loads must not assume 16-byte alignment."""
    N, K = 300, 1024
    packed, scales, cb = make_case(fmt, N, K, tag="xalign")
    x_np = make_x(M, K, tag="xalign")
    buf = torch.zeros(M * K + 8, dtype=torch.float16, device="cuda")
    x = buf[2:2 + M * K].view(M, K)
    assert x.data_ptr() % 16 == 4
    x.copy_(cuda(x_np))
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    y = h.gemv(x)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x_np)
    assert_within(y.cpu().numpy(), y_ref, bound, f"{fmt} M={M} x offset 4 B")


@pytest.mark.parametrize("fmt", FORMATS)
def test_one_hot_rows_extract_columns_bit_exact(fmt):
    N, K = SMALL[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="onehot")
    W = oracle.dequant(fmt, N, K, packed, scales, cb)
    cols = [0, 1, 31, 32, 63, 64, 127, 255, 256, 511, 512, K // 2 + 3, K - 33, K - 2, K - 1, 5]
    x = np.zeros((16, K), dtype=np.float16)
    for i, k in enumerate(cols):
        x[i, k] = 1.0
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    y = gpu_gemv(h, x)
    # column k of W, rounded once to fp32 (exact except for AQLM, where
    # c0 + c1 is exact in fp32 and the one product by s_n rounds)
    for i, k in enumerate(cols):
        assert np.array_equal(y[i], W[:, k].astype(np.float32)), f"column {k}"


@pytest.mark.parametrize("fmt", FORMATS)
def test_run_to_run_and_graph_bitwise(fmt):
    N, K = MULTI[fmt]
    packed, scales, cb = make_case(fmt, N, K, tag="repro")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    x = cuda(make_x(4, K, tag="repro"))
    y1 = h.gemv(x)
    y2 = h.gemv(x)
    s = torch.cuda.Stream()
    y3 = torch.empty_like(y1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        h.run(x, y3, stream=s)
    y3.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert torch.equal(y1, y2)
    assert torch.equal(y1, y3)


@pytest.mark.parametrize("fmt", FORMATS)
def test_output_guard_bands_untouched(fmt):
    N, K = SMALL[fmt]
    M = 5
    packed, scales, cb = make_case(fmt, N, K, tag="guard")
    h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
    x = cuda(make_x(M, K, tag="guard"))
    pad = 64
    buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[pad:pad + M * N]
    h.run(x, y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[-pad:] == 12345.0)
    assert not torch.any(y == 12345.0)


def test_run_argument_errors():
    N, K = SMALL["q4_0"]
    packed, scales, cb = make_case("q4_0", N, K)
    h = qgemv.QGemv("q4_0", N, K, packed, scales, cb)
    x = torch.zeros((16, K), dtype=torch.float16, device="cuda")
    y = torch.zeros((17 * N + 1,), dtype=torch.float32, device="cuda")
    lib = qgemv.load()
    assert lib.qgemv_run(h.handle, x.data_ptr(), 0, y.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_run(h.handle, x.data_ptr(), 17, y.data_ptr(), None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_run(h.handle, x.data_ptr(), 1, y.data_ptr() + 2, None) == qgemv.QGEMV_ERR_ALIGN
    assert lib.qgemv_run(h.handle, None, 1, y.data_ptr(), None) == qgemv.QGEMV_ERR_ARG


def test_create_accepts_device_pointers():
    N, K = SMALL["pq2_0"]
    packed, _, _ = make_case("pq2_0", N, K, tag="devptr")
    h_host = qgemv.QGemv("pq2_0", N, K, packed)
    h_dev = qgemv.QGemv("pq2_0", N, K, cuda(packed))
    assert torch.equal(h_host.dequant(), h_dev.dequant())


# --------------------------------------------------------- quantizer ----

def test_q4_0_quantizer_matches_oracle_bytes():
    g = inputs.rng("quant")
    N, K = 257, 1024
    w = inputs.w_fp32(g, N, K)
    w[0, :32] = 0.0                            # all-zero block
    w[1, :32] = 0.25; w[1, 5] = -0.25          # tie on |w|: first wins
    w[2, 0:32] = np.linspace(-1, 1, 32)        # clamp at +8 -> 15
    w[3, 40] = 1e-30                           # tiny values
    w[4, 64:96] = 1e-6 * np.arange(32)         # subnormal fp16 scale
    ref = oracle.quantize_q4_0(w, N, K)
    got = qgemv.quantize_q4_0(cuda(w)).cpu().numpy()
    assert np.array_equal(got, ref)


def test_q4_0_end_to_end_from_fp32_weights():
    """Workload 'Q4_0 4096x4096, M=1': each side quantizes W itself."""
    N = K = 4096
    w = inputs.w_fp32(inputs.rng("C1/w"), N, K)
    x = inputs.x_fp16(inputs.rng("C1/x"), 1, K)
    packed_gpu = qgemv.quantize_q4_0(cuda(w))
    h = qgemv.QGemv("q4_0", N, K, packed_gpu)
    y = gpu_gemv(h, x)
    packed_ref = oracle.quantize_q4_0(w, N, K)
    y_ref, bound = oracle.gemv("q4_0", N, K, packed_ref, None, None, x)
    assert_within(y, y_ref, bound, "C1")


# ---------------------------------------------- full sizes, sampled ----

def sample_rows(N, n=48, seed=0):
    g = np.random.default_rng(seed)
    rows = set([0, 1, 127, 128, N // 2, N - 129, N - 2, N - 1])
    rows.update(g.integers(0, N, size=n).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


@pytest.mark.parametrize("fmt, N, K, Ms", [
    ("q4_0", 8192, 28672, (1, 16)),      # down projection, batch sweep shape
    ("pq2_0", 8192, 28672, (1, 16)),
    ("cbk4", 8192, 28672, (1, 16)),
    ("cbk4", 11008, 4096, (1,)),         # 7B gate / up
    ("cbk4", 4096, 11008, (1,)),         # 7B down
    ("cbk8", 32000, 4096, (1, 4)),       # 7B LM head
    ("pq2_0", 34816, 5120, (1, 8)),      # fused gate+up, hidden 5120
    ("pq2_0", 5120, 17408, (1, 8)),      # down, MLP 17408
    ("aqlm_2x8", 28672, 8192, (1, 2)),   # 70B gate / up
    ("aqlm_2x8", 8192, 28672, (1, 3)),   # 70B down
    ("aqlm_2x8", 8192, 8192, (1, 16)),   # 70B q / o
])
def test_full_size_sampled_rows(fmt, N, K, Ms):
    if fmt == "q4_0":
        w = inputs.w_fp32(inputs.rng(f"full/{fmt}/{N}x{K}"), N, K)
        packed_gpu = qgemv.quantize_q4_0(cuda(w))
        h = qgemv.QGemv(fmt, N, K, packed_gpu)
        rows = sample_rows(N)
        packed_rows = oracle.quantize_q4_0(w[rows], rows.size, K)   # quantization is row-local
        del w, packed_gpu
        for M in Ms:
            x = make_x(M, K, tag="full")
            y = gpu_gemv(h, x)[:, rows]
            y_ref, bound = oracle.gemv(fmt, rows.size, K, packed_rows, None, None, x)
            assert_within(y, y_ref, bound, f"{fmt} {N}x{K} M={M}")
    else:
        packed, scales, cb = make_case(fmt, N, K, tag="full")
        h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
        rows = sample_rows(N)
        for M in Ms:
            x = make_x(M, K, tag="full")
            y = gpu_gemv(h, x)[:, rows]
            y_ref, bound = oracle.gemv(fmt, N, K, packed, scales, cb, x, rows=rows)
            assert_within(y, y_ref, bound, f"{fmt} {N}x{K} M={M}")


def test_torch_side_stream_orders_with_torch_work():
    """QGemv calls without an explicit stream run on torch's current stream:
    on a side stream, the activations written there just before and the
    output read there just after are ordered with the GEMV, and the result
    equals the default-stream run bit for bit."""
    N, K = MULTI["cbk4"]
    packed, scales, cb = make_case("cbk4", N, K, tag="sidestream")
    h = qgemv.QGemv("cbk4", N, K, packed, scales, cb)
    x_np = make_x(3, K, tag="sidestream")
    y_default = gpu_gemv(h, x_np)
    s = torch.cuda.Stream()
    src = cuda(x_np)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        x = torch.empty_like(src)
        torch.cuda._sleep(1_000_000)  # keep the side stream busy so that an unordered run would race
        x.copy_(src)
        y = h.gemv(x)
        y_host = y.to("cpu", non_blocking=False)
    torch.cuda.synchronize()
    assert h.status() == qgemv.QGEMV_OK
    assert np.array_equal(y_host.numpy(), y_default)
