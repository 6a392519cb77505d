"""The host logic of bench.py that needs no GPU: the workloads' shapes are
valid for their formats, the canonical extra bytes of a stacked handle, and
the keying of the stored DRAM-traffic captures (a capture is stale exactly
when the code of its kernels changes, not when a comment does)."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bit_weight_only_gb300 import qgemv  # noqa: E402

FORMATS = {"q4_0", "cbk4", "cbk8", "pq2_0", "aqlm_2x8", "aqlm_1x16", "cbk4_row", "cbk8_row"}


@pytest.fixture(scope="module")
def lib():
    return qgemv.load()


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_workload_shapes_are_valid(lib, name):
    specs_fn, dominant, description = bench.WORKLOADS[name]
    specs = specs_fn()
    assert specs and description
    for fmt, call, N, K in specs:
        base = fmt[:-4] if fmt.endswith("_glu") else fmt
        assert base in FORMATS, (name, fmt)
        rows = list(N) if isinstance(N, (list, tuple)) else [N]
        for n in rows:
            assert qgemv.qgemv_packed_bytes(base, n, K) > 0, (name, call, n, K)
        if len(rows) > 1:  # stacked: every segment but the last on the format's tile rows
            tile = 2048 if base == "aqlm_2x8" else 128
            assert all(n % tile == 0 for n in rows[:-1]), (name, call, rows)
    assert dominant in {f for f, _, _, _ in specs}, name


def test_stacked_extra_bytes():
    """A stacked handle's codebooks and scales: a 32-byte CBK4 codebook per
    segment; for AQLM 2x8 an 8 KB codebook pair per segment and one fp16
    scale per row (the scales counted once, not per segment)."""
    assert bench.stacked_extra_bytes("cbk4", [4096, 4096, 4096]) == 3 * 32
    assert bench.stacked_extra_bytes("aqlm_2x8", [28672, 28672]) == 2 * 57344 + 2 * 8192
    assert bench.stacked_extra_bytes("aqlm_2x8", [2048]) == bench.canonical_extra_bytes("aqlm_2x8", 2048)
    fmt, _, segs, _ = bench.WORKLOADS["aqlm_70b_layer_stacked"][0]()[0]
    assert (fmt, segs) == ("aqlm_2x8", [28672, 28672])


def test_code_only_drops_comments_and_layout():
    a = "int x = 1; // one\n/* block\n comment */ int  y =\n 2;"
    b = "int x = 1;\nint y = 2;   // two"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only('const char* s = "// not a comment";') != bench._code_only("const char* s;")
    assert bench._code_only("a + b") != bench._code_only("a - b")


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    """Copy the sources, then: a comment edit keeps the hash, a code edit in a
    listed file changes it, an edit in an unlisted file does not."""
    csrc = os.path.join(ROOT, "bit_weight_only_gb300", "csrc")
    dst = tmp_path / "bit_weight_only_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in os.listdir(csrc):
        p = os.path.join(csrc, f)
        if os.path.isfile(p) and (f.endswith((".cu", ".cuh", ".h"))):
            (dst / f).write_text(open(p, encoding="utf-8").read(), encoding="utf-8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash("aqlm_1x16", 1)
    src = dst / "fmt_aqlm1x16.cu"
    text = src.read_text(encoding="utf-8")
    src.write_text("// a new comment line\n" + text, encoding="utf-8")
    assert bench.kernel_source_hash("aqlm_1x16", 1) == h0
    src.write_text(text.replace("constexpr int kWarps = 8;", "constexpr int kWarps = 4;"), encoding="utf-8")
    assert bench.kernel_source_hash("aqlm_1x16", 1) != h0
    src.write_text(text, encoding="utf-8")
    q0 = bench.kernel_source_hash("q4_0", 1)
    other = dst / "fmt_q4_0.cu"  # not among the 1x16 kernel's sources
    other.write_text(other.read_text(encoding="utf-8") + "\nint unused_symbol;\n", encoding="utf-8")
    assert bench.kernel_source_hash("aqlm_1x16", 1) == h0
    assert bench.kernel_source_hash("q4_0", 1) != q0
    # M > 1 adds the tensor-core kernels' sources
    m8 = bench.kernel_source_hash("aqlm_1x16", 8)
    assert m8 != h0
    mma = dst / "mma_kernel.cuh"
    mma.write_text(mma.read_text(encoding="utf-8") + "\nint another_unused_symbol;\n", encoding="utf-8")
    assert bench.kernel_source_hash("aqlm_1x16", 8) != m8
    assert bench.kernel_source_hash("aqlm_1x16", 1) == h0


def test_traffic_entries_name_known_workloads():
    t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert t
    for key, v in t.items():
        workload = key.split("/")[0]
        assert workload in bench.WORKLOADS, key
        assert v["format"] in FORMATS, key
        assert v["M"] >= 1 and v["dram_bytes_per_launch"] > 0 and v["launches"] >= 1, key
        assert len(v["kernel_source_hash"]) == 16 and v["commit"], key
        assert "--clock-control none" in v["how"], key
