"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function ``include/qgemv.h`` declares, and rejects bad
arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

from bit_weight_only_gb300 import build, qgemv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qgemv.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qgemv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("qgemv_create", "qgemv_create_stacked", "qgemv_run", "qgemv_destroy", "qgemv_dequant",
              "qgemv_last_error", "qgemv_packed_bytes", "qgemv_quantize_q4_0", "qgemv_status"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in qgemv.h but not exported"
    assert set(declared_functions()) <= set(qgemv._SIGNATURES)


def test_packed_bytes_matches_formats(lib):
    assert qgemv.qgemv_packed_bytes("q4_0", 4096, 4096) == 4096 * 128 * 18
    assert qgemv.qgemv_packed_bytes("pq2_0", 5120, 17408) == 5120 * 136 * 34
    assert qgemv.qgemv_packed_bytes("aqlm_2x8", 4096, 4096) == 4_194_304
    assert qgemv.qgemv_packed_bytes("cbk4", 7, 10) == 35
    assert qgemv.qgemv_packed_bytes("cbk8", 7, 9) == 63
    assert qgemv.qgemv_packed_bytes("q4_0", 7, 48) == 0
    assert qgemv.qgemv_packed_bytes(99, 7, 64) == 0
    assert qgemv.qgemv_packed_bytes(6, 7, 64) == 0   # reserved inside the library


@pytest.mark.parametrize("fmt, N, K", [("aqlm_1x16", 8192, 28672), ("aqlm_1x16", 3, 12), ("cbk4_row", 11008, 4096),
                                       ("cbk4_row", 5, 7), ("q4_0", 9, 96), ("pq2_0", 9, 384), ("cbk8", 3, 5),
                                       ("cbk8_row", 32000, 4096), ("cbk8_row", 3, 5)])
def test_packed_bytes_agree_with_the_oracle(lib, fmt, N, K):
    """The library's canonical sizes and the oracle's, written separately, agree."""
    import oracle
    assert qgemv.qgemv_packed_bytes(fmt, N, K) == oracle.packed_bytes(fmt, N, K)


def test_prepared_activation_sizes_and_host_checks(lib):
    assert qgemv.qgemv_xq_bytes(3, 5120) == 3 * 5120 + 8 * 3 * 40
    assert qgemv.qgemv_xq_bytes(0, 5120) == 0 and qgemv.qgemv_xq_bytes(1, 100) == 0
    # rejected on the host, before any launch
    assert lib.qgemv_prepare_x_int8(None, 1, 1024, None, 0, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_prepare_x_int8(16, 1, 1024, None, 512, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_prepare_x_int8(16, 1, 1280, None, 1024, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_prepare_x_int8(16, 1, 1024, 16, 0, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_prepare_x_int8(18, 1, 1024, None, 0, 16, None) == qgemv.QGEMV_ERR_ALIGN
    assert lib.qgemv_quantize_x_int8(16, 1, 200, 16, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_run_xq(None, 16, 1, 16, None, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_set_x_int8(None, 1) == qgemv.QGEMV_ERR_ARG


@pytest.mark.parametrize("args, fragment", [
    ((99, 8, 64, 1, None, None), "unknown format"),
    ((qgemv.Q4_0, 8, 48, 1, None, None), "invalid shape"),
    ((qgemv.Q4_0, 0, 64, 1, None, None), "invalid shape"),
    ((qgemv.PQ2_0, 8, 64, 1, None, None), "invalid shape"),
    ((qgemv.Q4_0, 8, 64, None, None, None), "packed is NULL"),
    ((qgemv.Q4_0, 8, 64, 1, 1, None), "takes no scales"),
    ((qgemv.AQLM_1X16, 8, 12, 1, 1, 1), "invalid shape"),
    ((qgemv.AQLM_1X16, 8, 64, 1, None, 1), "needs scales"),
    ((qgemv.CBK4_ROW, 8, 64, 1, None, None), "needs codebooks"),
    ((qgemv.CBK4_ROW, 8, 63, 1, None, 1), "invalid shape"),
    ((qgemv.CBK8_ROW, 8, 70000, 1, None, 1), "K up to 65536"),
    ((qgemv.CBK8_ROW, 8, 64, 1, None, None), "needs codebooks"),
    ((6, 8, 64, 1, None, None), "unknown format"),
])
def test_create_rejects_bad_arguments_on_host(lib, args, fragment):
    h = lib.qgemv_create(*args)
    assert not h
    assert fragment in qgemv.qgemv_last_error()
    assert qgemv.qgemv_last_error_code() == qgemv.QGEMV_ERR_ARG


def test_run_rejects_bad_handle_and_m(lib):
    assert lib.qgemv_run(None, 16, 1, 16, None) == qgemv.QGEMV_ERR_ARG
    bogus = ctypes.create_string_buffer(256)  # not a handle: magic check fails
    assert lib.qgemv_run(ctypes.addressof(bogus), 16, 1, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_dequant(None, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_status(None) == qgemv.QGEMV_ERR_ARG
    lib.qgemv_destroy(None)  # NULL is accepted


def test_stacked_create_rejects_bad_arguments_on_host(lib):
    rows = (ctypes.c_int64 * 2)(100, 200)
    assert not lib.qgemv_create_stacked(qgemv.CBK4, 2, rows, 256, 1, None, 1)
    assert "multiple of 128" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_stacked(qgemv.CBK4, 0, rows, 256, 1, None, 1)
    assert qgemv.qgemv_last_error_code() == qgemv.QGEMV_ERR_ARG
    ok_rows = (ctypes.c_int64 * 2)(2048, 2048)
    aqlm_rows = (ctypes.c_int64 * 2)(1024, 2048)  # AQLM 2x8 segments start on 2048-row blocks
    assert not lib.qgemv_create_stacked(qgemv.AQLM_2X8, 2, aqlm_rows, 256, 1, 1, 1)
    assert "multiple of 2048" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_stacked(99, 1, ok_rows, 256, 1, None, None)
    assert "unknown format" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_stacked(qgemv.AQLM_1X16, 2, ok_rows, 256, 1, 1, 1)
    assert "cannot be stacked" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_stacked(qgemv.CBK4_ROW, 2, ok_rows, 256, 1, None, 1)
    assert "cannot be stacked" in qgemv.qgemv_last_error()


def test_glu_create_rejects_bad_arguments_on_host(lib):
    assert not lib.qgemv_create_glu(qgemv.AQLM_2X8, 128, 256, 1, 1, None, None)
    assert "no fused" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_glu(qgemv.CBK4, 128, 256, 1, 1, 1, None)
    assert "needs both codebook" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_glu(qgemv.PQ2_0, 100, 256, 1, 1, None, None)
    assert "multiple of 64" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_glu(qgemv.Q4_0, 128, 48, 1, 1, None, None)
    assert not lib.qgemv_create_glu(qgemv.Q4_0, 128, 64, None, 1, None, None)
    assert not lib.qgemv_create_glu(qgemv.CBK4_ROW, 128, 64, 1, 1, None, None)
    assert "needs both codebook" in qgemv.qgemv_last_error()
    assert not lib.qgemv_create_glu(qgemv.PQ2_0, 128, 256, 1, 1, 1, None)
    assert qgemv.qgemv_last_error_code() == qgemv.QGEMV_ERR_ARG


def test_quantizer_rejects_bad_shape(lib):
    assert lib.qgemv_quantize_q4_0(16, 4, 48, 16, None) == qgemv.QGEMV_ERR_ARG
    assert lib.qgemv_quantize_q4_0(None, 4, 64, 16, None) == qgemv.QGEMV_ERR_ARG


def test_product_path_does_not_reference_the_oracle():
    """The CUDA package never imports, loads or links the oracle."""
    pkg = os.path.join(ROOT, "bit_weight_only_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f
