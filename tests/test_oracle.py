"""Pins for the CPU oracle: values and identities fixed by the pages and by
mathematics, never by the oracle itself or by the CUDA path.

Each test names what it pins.  A plausible mistake in the oracle (a dropped
term, a wrong sign, a swapped nibble, a transposed operand) fails at least
one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_weight_only_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------- fp16 ----

def test_half_to_double_matches_ieee_library_for_all_bit_patterns():
    """Pin: every binary16 pattern decodes to numpy's IEEE value."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.all(both_nan | (got == r))
    for b in (0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x7C00, 0xFC00):
        assert oracle.half_to_double(b) == float(np.array([b], np.uint16).view(np.float16)[0])


def test_float_to_half_rounds_like_ieee_library():
    """Pin: fp32 -> fp16 is round-to-nearest-even, as numpy's cast."""
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(4000).astype(np.float32) * np.float32(0.02),
        g.standard_normal(2000).astype(np.float32) * np.float32(3e4),
        (g.random(2000) * 1e-4).astype(np.float32),        # subnormal range
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9,
                  2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 1 + 2.0 ** -11,
                  1 + 3 * 2.0 ** -11, np.inf, -np.inf], dtype=np.float32),
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------- byte budget --

def test_byte_budget_matches_pages(golden_dir):
    """Pin: bytes per block / per matrix as the pages print them."""
    gb = json.load(open(os.path.join(golden_dir, "byte_budget.json")))
    q = gb["q4_0"]
    assert oracle.packed_bytes("q4_0", 1, q["weights_per_block"]) == q["bytes_per_block"]
    assert 8 * q["bytes_per_block"] / q["weights_per_block"] == q["bits_per_weight"]
    p = gb["pq2_0"]
    assert oracle.packed_bytes("pq2_0", 1, p["weights_per_block"]) == p["bytes_per_block"]
    assert 8 * p["bytes_per_block"] / p["weights_per_block"] == p["bits_per_weight"]
    # PQ2 matrix is uint8 (N, K/128 * 34)
    assert oracle.packed_bytes("pq2_0", 5120, 17408) == 5120 * (17408 // 128) * 34
    a = gb["aqlm_2x8"]
    codes = oracle.packed_bytes("aqlm_2x8", a["N"], a["K"])
    assert round(codes / 1e6, 1) == a["codes_mb"]
    assert round(a["N"] * a["K"] * 2 / 1e6, 1) == a["fp16_mb"]
    assert codes * 8 / (a["N"] * a["K"]) == 2.0        # 2 bits per weight
    assert oracle.codebook_count("aqlm_2x8") == 2 * 256 * 8
    assert oracle.scales_count("aqlm_2x8", 7, 64) == 7
    # invalid shapes are rejected
    assert oracle.packed_bytes("q4_0", 4, 48) == 0
    assert oracle.packed_bytes("pq2_0", 4, 64) == 0
    assert oracle.packed_bytes("aqlm_2x8", 4, 12) == 0
    assert oracle.packed_bytes("cbk4", 4, 3) == 0


def test_cbk_byte_accounting_reconstructs_7b_file_sizes(golden_dir):
    """Derived pin (reading): 4-bit indices cost N*K/2 bytes, 8-bit N*K.

    Rebuilding the printed 7B file sizes from the Llama-2-7B shapes with
    per-output-row fp32 centroids, an fp16 embedding and fp32 norms lands
    a few hundred bytes (a container header) under each printed size."""
    gb = json.load(open(os.path.join(golden_dir, "byte_budget.json")))["cbk4_7b_files"]
    shapes = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
    idx = 32 * sum(oracle.packed_bytes("cbk4", n, k) for n, k in shapes)
    rows = 32 * sum(n for n, _ in shapes)
    assert idx == 3_238_002_688 and rows == 1_359_872
    emb = 32000 * 4096 * 2
    norms = 65 * 4096 * 4
    legacy = (idx + rows * 16 * 4 + emb + oracle.packed_bytes("cbk4", 32000, 4096)
              + 32000 * 16 * 4 + norms)
    # the per-row-codebook format's own accounting (indices + fp32 codebooks)
    # gives the same projections-plus-head bytes
    per_row = 32 * sum(oracle.packed_bytes("cbk4_row", n, k) + oracle.codebook_bytes("cbk4_row", n)
                       for n, k in shapes)
    per_row += oracle.packed_bytes("cbk4_row", 32000, 4096) + oracle.codebook_bytes("cbk4_row", 32000)
    assert 0 < gb["legacy_file_bytes"] - (per_row + emb + norms) < 1024
    new = (idx + rows * 16 * 4 + emb + oracle.packed_bytes("cbk8", 32000, 4096)
           + 32000 * 256 * 4 + norms)
    head8 = oracle.packed_bytes("cbk8_row", 32000, 4096) + oracle.codebook_bytes("cbk8_row", 32000)
    assert head8 == oracle.packed_bytes("cbk8", 32000, 4096) + 32000 * 256 * 4
    assert 0 < gb["legacy_file_bytes"] - legacy < 1024
    assert 0 < gb["new_file_bytes"] - new < 1024
    # the 8-bit head's extra bytes explain the two files' difference to 8 bytes
    assert abs((gb["new_file_bytes"] - gb["legacy_file_bytes"]) - (new - legacy)) <= 8


# ----------------------------------------------------------------- PQ2 ---

def _pq2_block(d: float, qs: bytes) -> np.ndarray:
    blk = np.zeros(34, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:] = np.frombuffer(qs, dtype=np.uint8)
    return blk


def test_pq2_worked_example(golden_dir):
    """Pin: the page's worked example, byte 0x64 with scale 0.5."""
    ex = json.load(open(os.path.join(golden_dir, "pq2_worked_example.json")))
    qs = bytes([ex["byte"]]) + bytes([0x55] * 31)       # 0x55: four code-1 fields = 0
    w = oracle.dequant("pq2_0", 1, 128, _pq2_block(ex["block_scale"], qs))
    assert list(w[0, :4]) == ex["values"]
    assert np.all(w[0, 4:] == 0.0)


def test_pq2_all_codes_brute_force(golden_dir):
    """Pin: each of the four codes, at each of the four field positions."""
    ex = json.load(open(os.path.join(golden_dir, "pq2_worked_example.json")))
    value = {int(k): v for k, v in ex["code_values"].items()}
    d = 0.25
    for pos in range(4):
        for code in range(4):
            byte = (0x55 & ~(3 << (2 * pos))) | (code << (2 * pos))
            qs = bytes([0x55] * 7 + [byte] + [0x55] * 24)
            w = oracle.dequant("pq2_0", 1, 128, _pq2_block(d, qs))[0]
            nz = np.nonzero(w)[0]
            if value[code] == 0:
                assert nz.size == 0
            else:
                assert list(nz) == [7 * 4 + pos]
                assert w[7 * 4 + pos] == value[code] * d


def test_pq2_second_block_and_row_use_their_own_scale():
    """Pin: block b of row n sits at byte (n*K/128 + b)*34 with its own d."""
    blocks = [_pq2_block(s, bytes([0xAA] * 32)) for s in (1.0, 2.0, 4.0, 8.0)]  # all +1
    packed = np.concatenate(blocks)
    w = oracle.dequant("pq2_0", 2, 256, packed)
    assert np.all(w[0, :128] == 1.0) and np.all(w[0, 128:] == 2.0)
    assert np.all(w[1, :128] == 4.0) and np.all(w[1, 128:] == 8.0)


# ------------------------------------------------------------ AQLM 1x16 ---

def test_aqlm_1x16_byte_budget(golden_dir):
    """Pin: 16-bit codes per 8 weights are still 2 bits per weight, and the
    codebook of 65,536 entries of 8 fp16 values is the page's 1 MiB."""
    gb = json.load(open(os.path.join(golden_dir, "aqlm_1x16.json")))
    N, K = 4096, 4096
    assert oracle.packed_bytes("aqlm_1x16", N, K) * 8 == N * K * gb["bits_per_weight"]
    assert oracle.packed_bytes("aqlm_1x16", N, K) == N * (K // gb["group"]) * gb["code_bits"] // 8
    assert oracle.codebook_count("aqlm_1x16") == gb["codebook_entries"] * gb["entry_values"]
    assert oracle.codebook_count("aqlm_1x16") * 2 == gb["codebook_bytes"]
    assert oracle.scales_count("aqlm_1x16", N, K) == N
    assert oracle.packed_bytes("aqlm_1x16", 4, 12) == 0


def test_aqlm_1x16_is_2x8_with_the_sum_codebook():
    """Pin (reduction): a 1x16 codebook whose entry a + 256 b is C0[a] + C1[b]
    decodes the 2x8 code bytes (a, b) to the 2x8 weights, exactly (the sums
    are exact in fp16: multiples of 2^-8 below 1/2)."""
    g = np.random.default_rng(21)
    N, K = 37, 256
    C = (g.integers(-64, 65, size=(2, 256, 8)) * 2.0 ** -8).astype(np.float16)
    C16 = (C[0][None, :, :].astype(np.float64) + C[1][:, None, :].astype(np.float64)).reshape(65536, 8)
    assert np.array_equal(C16.astype(np.float16).astype(np.float64), C16)   # exact in fp16
    C16 = C16.astype(np.float16)   # entry b * 256 + a
    codes = g.integers(0, 256, size=(N, K // 8, 2), dtype=np.uint8)
    scales = g.uniform(0.5, 1.5, size=N).astype(np.float16)
    w2 = oracle.dequant("aqlm_2x8", N, K, codes, scales, C)
    w16 = oracle.dequant("aqlm_1x16", N, K, codes, scales, C16)
    assert np.array_equal(w2, w16)
    x = inputs.x_fp16(inputs.rng("1x16/x"), 3, K)
    y2, b2 = oracle.gemv("aqlm_2x8", N, K, codes, scales, C, x)
    y16, b16 = oracle.gemv("aqlm_1x16", N, K, codes, scales, C16, x)
    assert np.array_equal(y2, y16) and np.array_equal(b2, b16)


def test_aqlm_1x16_single_entry_closed_form():
    """Pin: one group coded 0xBEEF (bytes EF BE) reads entry 48879 times the
    row scale; every other group reads the zero entry 0."""
    N, K = 3, 64
    cb = np.zeros((65536, 8), dtype=np.float16)
    cb[0xBEEF] = np.arange(1, 9) * 0.125
    cb[0xEFBE] = -1.0   # the byte-swapped index must not be read
    codes = np.zeros((N, K // 8), dtype=np.uint16)
    codes[1, 5] = 0xBEEF
    scales = np.array([1.0, 2.0, 4.0], dtype=np.float16)
    w = oracle.dequant("aqlm_1x16", N, K, codes, scales, cb)
    expect = np.zeros((N, K))
    expect[1, 40:48] = 2.0 * np.arange(1, 9) * 0.125
    assert np.array_equal(w, expect)


# ------------------------------------------------- PQ2 integer path ---

def test_int8_quantizer_scale_range_and_ties(golden_dir):
    """Pin: the group scale maps the group's largest |x| to +-q_max; ties
    round to even; a zero group has scale 0 and codes 0."""
    gi = json.load(open(os.path.join(golden_dir, "pq2_int8.json")))
    G, QM = gi["group"], gi["q_max"]
    x = np.zeros((2, 3 * G), dtype=np.float16)
    # group 0: amax = 127 makes the scale exactly 1, so x / a is x itself
    x[0, :8] = [127.0, 2.5, 3.5, -2.5, -0.5, 1.5, -126.5, 0.25]
    # group 1: random; group 2: all zero; row 1: negative extreme
    x[0, G:2 * G] = inputs.x_fp16(inputs.rng("int8/x"), 1, G)[0]
    x[1, :G] = -np.abs(inputs.x_fp16(inputs.rng("int8/x2"), 1, G)[0])
    q, a = oracle.quantize_x_int8(x)
    assert q.dtype == np.int8 and q.shape == x.shape and a.shape == (2, 3)
    assert a[0, 0] == 1.0
    assert list(q[0, :8]) == [127, 2, 4, -2, 0, 2, -126, 0]
    assert np.all(q[0, 8:G] == 0)
    assert a[0, 2] == 0.0 and np.all(q[0, 2 * G:] == 0)
    assert a[1, 1] == 0.0 and a[1, 2] == 0.0 and np.all(q[1, G:] == 0)
    for m, g in ((0, 1), (1, 0)):
        xg = x[m, g * G:(g + 1) * G].astype(np.float64)
        qg = q[m, g * G:(g + 1) * G].astype(np.int64)
        amax = np.abs(xg).max()
        assert abs(a[m, g] * QM - amax) <= amax * 2.0 ** -23
        assert np.abs(qg).max() == QM and np.all(np.abs(qg) <= QM)
        assert qg[np.argmax(np.abs(xg))] == np.sign(xg[np.argmax(np.abs(xg))]) * QM
        # each code is a nearest integer of x / a (up to one fp32 rounding)
        assert np.all(np.abs(xg / float(a[m, g]) - qg) <= 0.5 + QM * 2.0 ** -23)


def _on_grid_x(seed: str, M: int, K: int, zero_groups=()):
    """x_i = q_i * 2^-7 with integer |q_i| <= 127 and one +-127 per group:
    the int8 scale is then 2^-7 exactly and quantisation is lossless."""
    g = inputs.rng(seed)
    q = g.integers(-127, 128, size=(M, K))
    q[:, ::128] = np.where(g.random((M, K // 128)) < 0.5, -127, 127)
    for m, grp in zero_groups:
        q[m, grp * 128:(grp + 1) * 128] = 0
    return (q * 2.0 ** -7).astype(np.float16)


def test_pq2_int8_is_exact_for_activations_on_the_int8_grid():
    """Pin: when every activation is a_g * q_i exactly, the integer path
    reproduces the exact PQ2_0 GEMV (all sums are exact in fp64)."""
    N, K, M = 37, 1024, 3
    packed = inputs.pq2_packed(inputs.rng("int8/w"), N, K)
    x = _on_grid_x("int8/grid", M, K, zero_groups=[(1, 2), (2, 7)])
    q, a = oracle.quantize_x_int8(x)
    assert a[0, 0] == 2.0 ** -7 and a[1, 2] == 0.0
    assert np.array_equal(q.astype(np.float64) * np.repeat(a, 128, axis=1), x.astype(np.float64))
    y, b = oracle.gemv_pq2_int8(N, K, packed, x)
    ye, be = oracle.gemv("pq2_0", N, K, packed, None, None, x)
    assert np.array_equal(y, ye) and np.array_equal(b, be)


def test_pq2_int8_page_maximum_inner_sum(golden_dir):
    """Pin: all-(+1) codes against a group at the positive maximum give the
    page's largest inner sum; all-(-1) codes against the negative maximum
    give the same; the result is d * a * sum."""
    gi = json.load(open(os.path.join(golden_dir, "pq2_int8.json")))
    G = gi["group"]
    for code_byte, xv in ((0xAA, 1.0), (0x00, -1.0)):
        packed = np.concatenate([_pq2_block(0.5, bytes([code_byte] * 32)),
                                 _pq2_block(2.0, bytes([0x55] * 32))])
        x = np.full((1, 2 * G), xv, dtype=np.float16)
        y, b = oracle.gemv_pq2_int8(1, 2 * G, packed, x)
        a = float(np.float32(1.0) / np.float32(gi["q_max"]))
        assert y[0, 0] == 0.5 * a * gi["max_inner_sum"] and b[0, 0] == y[0, 0]
        assert gi["max_inner_sum"] == G * gi["q_max"]


def test_pq2_int8_error_within_quantisation_bound():
    """Pin: against the exact GEMV, the integer path errs by at most half a
    step of each group's scale per nonzero weight (plus one fp32 rounding of
    x / a), and it does err on general activations."""
    N, K, M = 64, 2048, 4
    packed = inputs.pq2_packed(inputs.rng("int8/w2"), N, K)
    x = inputs.x_fp16(inputs.rng("int8/x3"), M, K)
    y, b = oracle.gemv_pq2_int8(N, K, packed, x)
    ye, _ = oracle.gemv("pq2_0", N, K, packed, None, None, x)
    _, a = oracle.quantize_x_int8(x)
    W = np.abs(oracle.dequant("pq2_0", N, K, packed))
    step = np.repeat(a.astype(np.float64), 128, axis=1)          # [M, K]
    lim = (step * (0.5 + 127 * 2.0 ** -23)) @ W.T
    assert np.all(np.abs(y - ye) <= lim * (1 + 1e-12))
    assert np.count_nonzero(y != ye) > y.size // 2
    assert np.all(b >= np.abs(y))


# ------------------------------------------------------ Hadamard mixing ---

def test_hadamard_is_the_library_sylvester_matrix():
    """Pin (library routine): per block, y = B^-1/2 H (s . x) with scipy's
    Sylvester Hadamard matrix, for several B; blocks are independent."""
    sl = pytest.importorskip("scipy.linalg")
    g = np.random.default_rng(31)
    for B in (1, 2, 8, 64, 1024):
        K = 2 * B
        x = g.standard_normal((3, K))
        s = g.choice([-1, 1], size=K).astype(np.int8)
        y = oracle.hadamard(x, B, s)
        H = sl.hadamard(B) / np.sqrt(B)
        for b in range(2):
            blk = slice(b * B, (b + 1) * B)
            ref = (x[:, blk] * s[blk]) @ H.T
            assert np.allclose(y[:, blk], ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


def test_hadamard_closed_forms_and_involution():
    """Pin: e_0 spreads to B^-1/2 everywhere, a constant block concentrates
    in element 0, the normalised transform is its own inverse and keeps the
    norm, and signs act as a sign flip of the inputs."""
    B = 1024
    e0 = np.zeros((1, B))
    e0[0, 0] = 1.0
    assert np.array_equal(oracle.hadamard(e0, B), np.full((1, B), 1.0 / 32))
    ones = oracle.hadamard(np.ones((1, B)), B)
    assert ones[0, 0] == 32.0 and np.all(ones[0, 1:] == 0.0)
    g = np.random.default_rng(8)
    x = g.standard_normal((2, 2 * B))
    y = oracle.hadamard(x, B)
    assert np.allclose(oracle.hadamard(y, B), x, rtol=0, atol=1e-12)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    s = g.choice([-1, 1], size=2 * B).astype(np.int8)
    assert np.array_equal(oracle.hadamard(x, B, s), oracle.hadamard(x * s, B))


def test_hadamard_f32_butterfly_matches_the_definition():
    """Pin: on small integers every butterfly is exact in fp32, so the page's
    fp32 form equals the exact transform bit for bit (a wrong sign, pairing
    or skipped stage fails); on general inputs it is within log2(B) fp32
    roundings of it."""
    g = np.random.default_rng(5)
    B = 1024
    x = g.integers(-8, 9, size=(2, 3 * B)).astype(np.float32)
    s = g.choice([-1, 1], size=3 * B).astype(np.int8)
    yf = oracle.hadamard_f32(x, B, s).astype(np.float64)
    assert np.array_equal(yf, oracle.hadamard(x.astype(np.float64), B, s))
    xr = inputs.x_fp16(inputs.rng("had/x"), 2, 3 * B).astype(np.float32)
    yf = oracle.hadamard_f32(xr, B, s).astype(np.float64)
    ye = oracle.hadamard(xr.astype(np.float64), B, s)
    lim = 11 * 2.0 ** -24 * np.repeat(np.abs(xr).reshape(2, 3, B).sum(axis=2), B, axis=1) / 32
    assert np.all(np.abs(yf - ye) <= lim)
    assert np.count_nonzero(yf != ye) > 0


def test_prepared_activations_and_codes_gemv():
    """Pin: the fp32 quantizer agrees with the fp16 one on fp16 values; the
    prologue without mixing is the plain quantizer, with mixing it quantizes
    the fp32 transform; the GEMV on given codes reproduces the fp16-input
    integer GEMV."""
    K, N = 2048, 33
    x = inputs.x_fp16(inputs.rng("prep/x"), 3, K)
    q16, a16 = oracle.quantize_x_int8(x)
    q32, a32 = oracle.quantize_f32_int8(x.astype(np.float32))
    assert np.array_equal(q16, q32) and np.array_equal(a16, a32)
    q0, a0 = oracle.prepare_x_int8(x, 0)
    assert np.array_equal(q0, q16) and np.array_equal(a0, a16)
    s = np.random.default_rng(2).choice([-1, 1], size=K).astype(np.int8)
    qh, ah = oracle.prepare_x_int8(x, 1024, s)
    qr, ar = oracle.quantize_f32_int8(oracle.hadamard_f32(x.astype(np.float32), 1024, s))
    assert np.array_equal(qh, qr) and np.array_equal(ah, ar)
    packed = inputs.pq2_packed(inputs.rng("prep/w"), N, K)
    y1, b1 = oracle.gemv_pq2_int8_q(N, K, packed, q16, a16)
    y2, b2 = oracle.gemv_pq2_int8(N, K, packed, x)
    assert np.array_equal(y1, y2) and np.array_equal(b1, b2)


# --------------------------------------------------- SiLU(gate) * up ---

def test_silu_is_x_times_the_library_logistic():
    """Pin (library routine and closed forms): SiLU(v) = v * expit(v); SiLU(0)
    = 0; it tends to v for large v and to 0 for very negative v."""
    sp = pytest.importorskip("scipy.special")
    v = np.linspace(-30, 30, 1201)
    assert np.allclose(oracle.silu(v), v * sp.expit(v), rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12 and abs(oracle.silu(-40.0)) < 1e-15


def test_gemv_glu_one_hot_closed_form():
    """Pin: a one-hot x picks column k of both matrices, so the fused output
    is SiLU(G[:, k]) * U[:, k]."""
    N, K = 40, 256
    pg = inputs.pq2_packed(inputs.rng("glu/g"), N, K)
    pu = inputs.pq2_packed(inputs.rng("glu/u"), N, K)
    G = oracle.dequant("pq2_0", N, K, pg)
    U = oracle.dequant("pq2_0", N, K, pu)
    x = np.zeros((2, K), dtype=np.float16)
    x[0, 3] = 1.0
    x[1, 200] = 1.0
    y, g, u, _, _ = oracle.gemv_glu("pq2_0", N, K, pg, pu, x)
    assert np.array_equal(g[0], G[:, 3]) and np.array_equal(u[1], U[:, 200])
    v = G[:, 3]
    assert np.allclose(y[0], v / (1 + np.exp(-v)) * U[:, 3], rtol=1e-15, atol=0)


def test_glu_tolerance_rule():
    g = np.array([1.0, -2.0]); u = np.array([3.0, 0.5])
    bg = np.array([10.0, 10.0]); bu = np.array([1.0, 1.0])
    y_ref = oracle.silu(g) * u
    assert oracle.within_tolerance_glu(y_ref + 1e-3 * 10 * 3 * 1.05, g, u, bg, bu)[0]
    assert not oracle.within_tolerance_glu(y_ref + 0.1, g, u, bg, bu).any()


# ---------------------------------------------------------------- Q4_0 ---

def test_q4_0_roundtrip_is_exact_for_representable_blocks():
    """Pin (invariant): quantize(dequant-able weights) reproduces them.

    Weights (q - 8) * d with one element at q = 0 make d = signed-max/-8
    exact, so the quantizer must return those q and the decode those w."""
    g = np.random.default_rng(7)
    N, K = 6, 128
    q = g.integers(0, 16, size=(N, K))
    q[:, ::32] = 0                                   # the -8*d element of each block
    d = (2.0 ** g.integers(-9, -3, size=(N, K // 32))).astype(np.float32)
    d[::2] *= -1                                     # both signs of d
    w = ((q - 8) * np.repeat(d, 32, axis=1)).astype(np.float32)
    packed = oracle.quantize_q4_0(w, N, K)
    assert np.array_equal(oracle.dequant("q4_0", N, K, packed), w.astype(np.float64))


def test_q4_0_quantization_error_and_extreme_element():
    """Pin (closed form): |w - w_hat| <= |d|/2 (+ fp16 rounding of d) where
    w/d <= 7.5; weights past +7.5*d clamp to q = 15 and decode to 7*fp16(d);
    the largest-magnitude weight decodes to -8*fp16(d), keeping its sign."""
    g = np.random.default_rng(3)
    N, K = 16, 256
    w = inputs.w_fp32(g, N, K)
    w[0, 40] = 0.5      # block 1's largest magnitude (first of a tie)
    w[0, 45] = -0.5     # its negation: w/d = +8 clamps to q = 15
    packed = oracle.quantize_q4_0(w, N, K)
    wh = oracle.dequant("q4_0", N, K, packed).reshape(N, K // 32, 32)
    blocks = w.reshape(N, K // 32, 32)
    amax_idx = np.argmax(np.abs(blocks), axis=2)
    amax = np.take_along_axis(blocks, amax_idx[..., None], axis=2)[..., 0]
    d32 = (amax / np.float32(-8.0)).astype(np.float32)
    d16 = d32.astype(np.float16).astype(np.float64)
    ratio = blocks.astype(np.float64) / d32[..., None].astype(np.float64)
    clamped = ratio > 7.5
    assert clamped[0, 1, 45 - 32] and clamped.sum() > 1
    err = np.abs(wh - blocks.astype(np.float64))
    lim = np.abs(d32)[..., None] * (0.5 + 8 * 2.0 ** -11) + 1e-12
    assert np.all(err[~clamped] <= np.broadcast_to(lim, err.shape)[~clamped])
    assert np.array_equal(wh[clamped], np.broadcast_to(7 * d16[..., None], wh.shape)[clamped])
    got_max = np.take_along_axis(wh, amax_idx[..., None], axis=2)[..., 0]
    assert np.array_equal(got_max, -8.0 * d16)
    assert np.all(np.sign(got_max) == np.sign(amax))
    assert wh[0, 1, 40 - 32] == 0.5 and wh[0, 1, 45 - 32] == 7 * float(np.float16(0.5 / -8.0))


def test_q4_0_block_layout_positions():
    """Pin: each of the 32 positions of a block decodes from its own field,
    the scale is read from the block's first two bytes, and block b of row n
    sits at byte (n*K/32 + b)*18 (checked through the quantizer)."""
    N, K = 2, 64
    for pos in range(32):
        w = np.zeros((N, K), dtype=np.float32)
        w[1, 32 + pos] = -1.0                         # d = 1/8 for that block only
        packed = oracle.quantize_q4_0(w, N, K)
        blk = packed[(1 * 2 + 1) * 18:(1 * 2 + 2) * 18]
        assert blk[0:2].view(np.float16)[0] == np.float16(0.125)
        wh = oracle.dequant("q4_0", N, K, packed)
        expect = np.zeros((N, K))
        expect[1, 32 + pos] = -1.0
        assert np.array_equal(wh, expect)


def test_q4_0_all_zero_block_decodes_to_zero():
    packed = oracle.quantize_q4_0(np.zeros((1, 32), np.float32), 1, 32)
    assert np.all(packed[2:] == 0x88)
    assert np.all(oracle.dequant("q4_0", 1, 32, packed) == 0.0)


# ------------------------------------------------------------ codebooks --

def test_cbk4_identity_codebook_returns_indices():
    """Pin: w = c[idx]; with c[i] = i the decode is the index stream, low
    nibble first (reading), and every one of the 16 indices is reachable."""
    cb = np.arange(16, dtype=np.float16)
    row = np.array([(i & 15) | (((i + 5) & 15) << 4) for i in range(16)], dtype=np.uint8)
    w = oracle.dequant("cbk4", 1, 32, row, codebooks=cb)[0]
    assert list(w[0::2]) == [i & 15 for i in range(16)]
    assert list(w[1::2]) == [(i + 5) & 15 for i in range(16)]


def test_cbk4_value_multiset_is_codebook_of_nibbles():
    """Pin (order-free invariant): the decoded values of each row are the
    codebook entries of that row's nibbles, whatever their order."""
    g = np.random.default_rng(11)
    cb = inputs.cbk_centroids(16)
    packed = g.integers(0, 256, size=(5, 40), dtype=np.uint8)
    w = oracle.dequant("cbk4", 5, 80, packed, codebooks=cb)
    for n in range(5):
        nib = np.concatenate([packed[n] & 15, packed[n] >> 4])
        assert sorted(w[n]) == sorted(cb[nib].astype(np.float64))


def test_cbk4_row_with_one_shared_codebook_is_cbk4():
    """Pin (reduction to a pinned format): when every row's fp32 codebook is
    the same fp16-representable codebook, the per-row format decodes exactly
    like CBK4 with that codebook."""
    N, K = 9, 64
    g = inputs.rng("pin/cbk4_row/shared")
    packed = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    c16 = inputs.cbk_centroids(16)
    rows = np.tile(c16.astype(np.float32), (N, 1))
    assert np.array_equal(oracle.dequant("cbk4_row", N, K, packed, None, rows),
                          oracle.dequant("cbk4", N, K, packed, None, c16))


def test_cbk4_row_uses_each_rows_own_codebook():
    """Pin (closed form, brute force): row n's codebook c_n[i] = 1000 n + i
    (exact in fp32) decodes every nibble i of row n to 1000 n + i, for all 16
    values, low nibble first; changing one row's codebook changes only that
    row."""
    N, K = 4, 32
    packed = np.zeros((N, K // 2), dtype=np.uint8)
    for n in range(N):
        for j in range(K // 2):
            packed[n, j] = (j % 16) | (((j + n + 5) % 16) << 4)
    cb = (1000.0 * np.arange(N)[:, None] + np.arange(16)[None, :]).astype(np.float32)
    W = oracle.dequant("cbk4_row", N, K, packed, None, cb)
    for n in range(N):
        for j in range(K // 2):
            assert W[n, 2 * j] == 1000 * n + j % 16
            assert W[n, 2 * j + 1] == 1000 * n + (j + n + 5) % 16
    cb2 = cb.copy()
    cb2[2] = -cb2[2]
    W2 = oracle.dequant("cbk4_row", N, K, packed, None, cb2)
    assert np.array_equal(W2[[0, 1, 3]], W[[0, 1, 3]]) and np.array_equal(W2[2], -W[2])


def test_cbk8_row_with_one_shared_codebook_is_cbk8():
    """Pin (reduction): every row carrying the same fp16-representable
    256-entry codebook decodes as CBK8 with that codebook."""
    N, K = 9, 300
    g = inputs.rng("pin/cbk8_row/shared")
    cb = inputs.cbk_centroids(256)
    packed = g.integers(0, 256, size=(N, K), dtype=np.uint8)
    rows = np.tile(cb.astype(np.float32), (N, 1))
    assert np.array_equal(oracle.dequant("cbk8_row", N, K, packed, None, rows),
                          oracle.dequant("cbk8", N, K, packed, None, cb))


def test_cbk8_row_uses_each_rows_own_codebook():
    """Pin (closed form): with row n's centroid i = 1000 n + i every index of
    every row decodes to exactly that value."""
    N, K = 5, 256
    cb = (1000.0 * np.arange(N)[:, None] + np.arange(256)[None, :]).astype(np.float32)
    packed = np.tile(np.arange(256, dtype=np.uint8)[::-1], (N, 1))
    W = oracle.dequant("cbk8_row", N, K, packed, None, cb)
    assert np.array_equal(W, cb[:, ::-1].astype(np.float64))


def test_cbk8_all_256_indices():
    cb = (np.arange(256) / 256.0).astype(np.float16)
    row = np.arange(256, dtype=np.uint8)[::-1].copy()
    w = oracle.dequant("cbk8", 1, 256, row, codebooks=cb)[0]
    assert np.array_equal(w, np.arange(256)[::-1] / 256.0)


# ---------------------------------------------------------------- AQLM ---

def test_aqlm_single_codebook_reduction_and_linearity():
    """Pin: with C1 = 0 the decode is s * C0[code0] (a plain lookup); with
    C0 = 0 it is s * C1[code1]; the full decode is their sum (no dropped
    term); the per-row scale multiplies the summed vector."""
    g = np.random.default_rng(5)
    N, K = 3, 32
    codes, scales, cb = inputs.aqlm_inputs(g, N, K)
    scales = np.array([1.0, 2.0, 0.5], dtype=np.float16)
    only0 = cb.copy(); only0[1] = 0
    only1 = cb.copy(); only1[0] = 0
    w0 = oracle.dequant("aqlm_2x8", N, K, codes, scales, only0)
    w1 = oracle.dequant("aqlm_2x8", N, K, codes, scales, only1)
    w = oracle.dequant("aqlm_2x8", N, K, codes, scales, cb)
    lut0 = cb[0].astype(np.float64)
    expect0 = lut0[codes[:, :, 0]].reshape(N, K) * scales.astype(np.float64)[:, None]
    assert np.array_equal(w0, expect0)
    lut1 = cb[1].astype(np.float64)
    expect1 = lut1[codes[:, :, 1]].reshape(N, K) * scales.astype(np.float64)[:, None]
    assert np.array_equal(w1, expect1)
    assert np.allclose(w, w0 + w1, rtol=0, atol=1e-15)
    plain = oracle.dequant("aqlm_2x8", N, K, codes, np.ones(N, np.float16), cb)
    assert np.array_equal(w, plain * scales.astype(np.float64)[:, None])


def test_aqlm_group_order():
    """Pin: group g of row n covers k = 8g..8g+7, codes[n][g] = (code0, code1)."""
    N, K = 2, 24
    cb = np.zeros((2, 256, 8), dtype=np.float16)
    for e in range(256):
        cb[0, e, :] = e                       # codebook 0 carries the code
        cb[1, e, :] = np.arange(8) / 8.0      # codebook 1 carries the lane
    codes = np.zeros((N, K // 8, 2), dtype=np.uint8)
    codes[:, :, 0] = np.arange(N * (K // 8)).reshape(N, K // 8) + 1
    w = oracle.dequant("aqlm_2x8", N, K, codes, np.ones(N, np.float16), cb)
    for n in range(N):
        for g in range(K // 8):
            assert list(w[n, 8 * g:8 * g + 8]) == [codes[n, g, 0] + j / 8 for j in range(8)]


# ---------------------------------------------------------------- GEMV ---

FORMAT_CASES = ["q4_0", "cbk4", "cbk8", "pq2_0", "aqlm_2x8", "cbk4_row"]


def make_case(fmt, N, K, tag="pin", seed=0):
    """Canonical inputs for one format (host numpy), as the tests feed them."""
    g = inputs.rng(f"{tag}/{fmt}/{N}x{K}", seed)
    if fmt == "q4_0":
        return oracle.quantize_q4_0(inputs.w_fp32(g, N, K), N, K), None, None
    if fmt == "cbk4_row":
        cb = inputs.cbk_row_codebooks(g, N)
        return inputs.cbk_packed(g, N, K, 4, inputs.cbk_cell_probs(inputs.cbk_centroids(16))), None, cb
    if fmt in ("cbk4", "cbk8"):
        L = 16 if fmt == "cbk4" else 256
        cb = inputs.cbk_centroids(L)
        return inputs.cbk_packed(g, N, K, 4 if L == 16 else 8,
                                 inputs.cbk_cell_probs(cb)), None, cb
    if fmt == "pq2_0":
        return inputs.pq2_packed(g, N, K), None, None
    codes, scales, cb = inputs.aqlm_inputs(g, N, K)
    return codes, scales, cb


@pytest.mark.parametrize("fmt", FORMAT_CASES)
def test_gemv_equals_library_matmul_of_decoded_weights(fmt):
    """Pin: y = W x reduces to numpy's float64 matmul of the decoded matrix,
    the bound is sum |x*w|, and x = e_k returns column k exactly."""
    N, K = 37, 256
    packed, scales, cb = make_case(fmt, N, K)
    W = oracle.dequant(fmt, N, K, packed, scales, cb)
    x = inputs.x_fp16(inputs.rng("pin/x"), 3, K)
    y, b = oracle.gemv(fmt, N, K, packed, scales, cb, x)
    xd = x.astype(np.float64)
    assert np.allclose(y, xd @ W.T, rtol=1e-12, atol=1e-15)
    assert np.allclose(b, np.abs(xd) @ np.abs(W).T, rtol=1e-12, atol=1e-15)
    assert np.all(b >= np.abs(y))
    eye = np.zeros((4, K), dtype=np.float16)
    cols = [0, 1, K // 2 + 3, K - 1]
    for i, k in enumerate(cols):
        eye[i, k] = 1.0
    ye, _ = oracle.gemv(fmt, N, K, packed, scales, cb, eye)
    for i, k in enumerate(cols):
        assert np.array_equal(ye[i], W[:, k])


def test_gemv_exact_rational_sum_on_tiny_case():
    """Pin (brute force): on a tiny case the fp64 result equals the exact
    rational sum of x*w to within one rounding of the final value."""
    N, K = 3, 128
    packed, scales, cb = make_case("pq2_0", N, K, tag="tiny")
    W = oracle.dequant("pq2_0", N, K, packed)
    x = inputs.x_fp16(inputs.rng("tiny/x"), 2, K)
    y, _ = oracle.gemv("pq2_0", N, K, packed, None, None, x)
    for m in range(2):
        for n in range(N):
            exact = sum(Fraction(float(x[m, k])) * Fraction(float(W[n, k])) for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)


def test_gemv_row_subset_and_threads_agree():
    N, K = 50, 256
    packed, scales, cb = make_case("aqlm_2x8", N, K)
    x = inputs.x_fp16(inputs.rng("rows/x"), 2, K)
    y, b = oracle.gemv("aqlm_2x8", N, K, packed, scales, cb, x, nthreads=1)
    rows = [49, 0, 17, 17, 3]
    ys, bs = oracle.gemv("aqlm_2x8", N, K, packed, scales, cb, x, rows=rows, nthreads=4)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(bs, b[:, rows])


@pytest.mark.parametrize("fmt", ["cbk4", "aqlm_2x8"])
def test_gemv_residual_special_cases(fmt):
    """Pin: the residual form reduces to the residual itself for x = 0 and to
    the plain GEMV for a zero residual; row subsets take the residual's
    columns of the same rows."""
    N, K = 29, 256
    packed, scales, cb = make_case(fmt, N, K)
    g = inputs.rng("pin/residual")
    r = g.standard_normal((3, N))
    zero_x = np.zeros((3, K), dtype=np.float16)
    y0, b0 = oracle.gemv_residual(fmt, N, K, packed, scales, cb, zero_x, r)
    assert np.array_equal(y0, r) and np.array_equal(b0, np.zeros_like(r))
    x = inputs.x_fp16(g, 3, K)
    y, b = oracle.gemv(fmt, N, K, packed, scales, cb, x)
    yz, bz = oracle.gemv_residual(fmt, N, K, packed, scales, cb, x, np.zeros((3, N)))
    assert np.array_equal(yz, y) and np.array_equal(bz, b)
    rows = [5, 0, 28]
    ys, _ = oracle.gemv_residual(fmt, N, K, packed, scales, cb, x, r, rows=rows)
    yf, _ = oracle.gemv_residual(fmt, N, K, packed, scales, cb, x, r)
    assert np.array_equal(ys, yf[:, rows])


def test_residual_tolerance_rule():
    y_ref = np.array([1.0e6, 0.0, -3.0])
    bound = np.array([0.0, 0.0, 1.0])
    # one fp32 rounding of a large sum (an ulp of 1e6 in fp32 is 0.0625)
    assert oracle.within_tolerance_residual([1.0e6 + 0.0625, 0.0, -3.0 + 9e-4], y_ref, bound).all()
    assert not oracle.within_tolerance_residual([1.0e6 + 0.5, 0.0, -3.0], y_ref, bound).all()
    assert not oracle.within_tolerance_residual([1.0e6, 0.0, -3.0 - 2e-3], y_ref, bound).all()


def test_tolerance_rule():
    y_ref = np.array([1.0, -2.0, 0.0])
    bound = np.array([10.0, 2.0, 0.0])
    assert oracle.within_tolerance([1.0 + 9e-3, -2.0 - 1.9e-3, 9e-7], y_ref, bound).all()
    assert not oracle.within_tolerance([1.0 + 1.1e-2, -2.0, 0.0], y_ref, bound).all()
    assert not oracle.within_tolerance([1.0, -2.0, 2e-6], y_ref, bound).all()


# ------------------------------------------------------------- inputs ----

def test_cbk_centroids_and_cell_masses():
    """Pin: mid-rank N(0, 0.02) quantiles are symmetric and sorted, and the
    cell masses sum to one; drawn indices follow them (binomial 5 sigma)."""
    for L in (16, 256):
        c = inputs.cbk_centroids(L).astype(np.float64)
        assert np.all(np.diff(c) > 0)
        assert np.array_equal(c, -c[::-1])
        p = inputs.cbk_cell_probs(inputs.cbk_centroids(L))
        assert abs(p.sum() - 1) < 1e-12 and np.allclose(p, p[::-1])
    c16 = inputs.cbk_centroids(16)
    assert abs(float(c16[-1]) - 0.02 * 1.8627) < 2e-4          # Phi^-1(31/32)
    p = inputs.cbk_cell_probs(c16)
    packed = inputs.cbk_packed(inputs.rng("hist"), 512, 1024, 4, p)
    nib = np.concatenate([(packed & 15).ravel(), (packed >> 4).ravel()])
    cnt = np.bincount(nib, minlength=16)
    n = nib.size
    assert np.all(np.abs(cnt - n * p) <= 5 * np.sqrt(n * p * (1 - p)))


def test_pq2_code_frequencies_through_decode():
    packed = inputs.pq2_packed(inputs.rng("freq"), 64, 4096)
    w = oracle.dequant("pq2_0", 64, 4096, packed)
    d = np.repeat(packed.reshape(64, 32, 34)[:, :, 0:2].copy().view(np.float16)
                  .astype(np.float64).reshape(64, 32), 128, axis=1)
    ratio = np.where(d != 0, w / np.where(d != 0, d, 1), 0)
    n = ratio.size
    for v, p in ((-1, 0.3), (0, 0.4), (1, 0.3)):
        c = np.count_nonzero(ratio == v)
        assert abs(c - n * p) <= 5 * np.sqrt(n * p * (1 - p))
    assert np.count_nonzero(ratio == 2) == 0
