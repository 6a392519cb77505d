"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a temporary copy of ``oracle/oracle.c``
(on the CPU, never in the product path), builds it, and runs the pin suite
``tests/test_oracle.py`` against that build; the suite must fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "q4_0 nibbles swapped": [("int lo = qs[i] & 0x0f;", "int lo = qs[i] >> 4;"),
                             ("int hi = qs[i] >> 4;", "int hi = qs[i] & 0x0f;")],
    "q4_0 sign flipped": [("(double)(lo - 8) * d", "(double)(8 - lo) * d")],
    "q4_0 quantizer truncates": [("float r = roundf(v[i] / d);", "float r = truncf(v[i] / d);")],
    "q4_0 quantizer d sign": [("float d = amax / -8.0f;", "float d = amax / 8.0f;")],
    "pq2 fields read high-first": [("(qs[e / 4] >> (2 * (e % 4))) & 3",
                                    "(qs[e / 4] >> (6 - 2 * (e % 4))) & 3")],
    "pq2 code offset": [("w[b * 128 + e] = (double)(c - 1) * d;",
                         "w[b * 128 + e] = (double)(c - 2) * d;")],
    "pq2 byte index": [("qs[e / 4]", "qs[(e % 32)]")],
    "aqlm second codebook dropped": [("w[g * 8 + j] = s * (c0 + c1);", "w[g * 8 + j] = s * (c0);")],
    "aqlm codes swapped": [("int a = packed[(n * ng + g) * 2 + 0];",
                            "int a = packed[(n * ng + g) * 2 + 1];")],
    "aqlm scale dropped": [("w[g * 8 + j] = s * (c0 + c1);", "w[g * 8 + j] = (c0 + c1);")],
    "cbk4 nibble order": [("w[2 * j] = oracle_half_to_double(codebooks[row[j] & 0x0f]);",
                           "w[2 * j] = oracle_half_to_double(codebooks[row[j] >> 4]);")],
    "cbk8 index off by one bit": [("codebooks[row[k]]", "codebooks[row[k] ^ 1]")],
    "cbk4_row neighbour's codebook": [("const uint8_t* cb = (const uint8_t*)codebooks + n * 16 * 4;",
                                       "const uint8_t* cb = (const uint8_t*)codebooks + (n ^ 1) * 16 * 4;")],
    "cbk4_row nibble order": [("w[2 * j] = rdf32(cb, row[j] & 0x0f);", "w[2 * j] = rdf32(cb, row[j] >> 4);")],
    "int8 ties away from zero": [("float r = rintf(", "float r = roundf(")],
    "int8 scale over 128": [("float s = amax / 127.0f;", "float s = amax / 128.0f;")],
    "int8 block scale dropped": [("double da = d * (double)a[m * nb + b];", "double da = (double)a[m * nb + b];")],
    "int8 group scale of row 0": [("double da = d * (double)a[m * nb + b];", "double da = d * (double)a[b];")],
    "int8 codes of the next group": [("int t = (c - 1) * q[m * K + b * 128 + e];",
                                      "int t = (c - 1) * q[m * K + ((b + 1) % nb) * 128 + e];")],
    "aqlm_1x16 big-endian code": [("int code = rd16(packed + (n * ng + g) * 2);",
                                   "int code = (packed[(n * ng + g) * 2] << 8) | packed[(n * ng + g) * 2 + 1];")],
    "aqlm_1x16 scale dropped": [("w[g * 8 + j] = s * oracle_half_to_double(codebooks[code * 8 + j]);",
                                 "w[g * 8 + j] = oracle_half_to_double(codebooks[code * 8 + j]);")],
    "aqlm_1x16 entry stride": [("codebooks[code * 8 + j]", "codebooks[(code >> 1) * 8 + j]")],
    "hadamard parity of i | j": [("__builtin_popcount((unsigned)(i & j))", "__builtin_popcount((unsigned)(i | j))")],
    "hadamard signs ignored": [("double v = x[m * K + b0 + j] * (signs ? (double)signs[b0 + j] : 1.0);",
                                "double v = x[m * K + b0 + j];")],
    "butterfly difference reversed": [("v[i + h] = u - w;", "v[i + h] = w - u;")],
    "butterfly first stage skipped": [("for (int h = 1; h < B; h <<= 1)", "for (int h = 2; h < B; h <<= 1)")],
    "butterfly signs ignored": [("v[i] = x[m * K + b0 + i] * (signs ? (float)signs[b0 + i] : 1.0f);",
                                 "v[i] = x[m * K + b0 + i];")],
    "cbk8_row neighbour's codebook": [("const uint8_t* cb = (const uint8_t*)codebooks + n * 256 * 4;",
                                       "const uint8_t* cb = (const uint8_t*)codebooks + (n ^ 1) * 256 * 4;")],
    "cbk8_row index bit flipped": [("for (int64_t k = 0; k < K; ++k) w[k] = rdf32(cb, row[k]);",
                                    "for (int64_t k = 0; k < K; ++k) w[k] = rdf32(cb, row[k] ^ 1);")],
    "bound without abs": [("b += fabs(t);", "b += t;")],
    "x transposed against w": [("double t = xd[m * K + k] * w[k];",
                                "double t = xd[m * K + (K - 1 - k)] * w[k];")],
    "fp16 rounding truncates": [("double S = rint(ldexp(a, 10 - E));",
                                 "double S = floor(ldexp(a, 10 - E));")],
    "fp16 subnormal exponent": [("v = ldexp((double)mant, -24);", "v = ldexp((double)mant, -25);")],
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert old in src, f"mutation anchor not found: {old}"
        src = src.replace(old, new)
    c = tmp_path / "oracle_mut.c"
    lib = tmp_path / "liboracle_mut.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(c), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                          "-q", "-x", "-p", "no:cacheprovider"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"pins did not catch '{name}':\n{res.stdout[-2000:]}"
