"""bench.py's host helpers on CPU: the code-only source hash that ties the committed
DRAM traffic record to the kernel sources it was captured on, and the record lookup."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_text_ignores_comments_and_layout_only():
    a = "int f(int x) {  // doubles\n    return 2 * x; /* the\n  factor */\n}\n"
    b = "int f(int x) {\n\treturn 2 * x;\n}  // reflowed, re-commented\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench._code_text(a) == bench._code_text(b) == "int f(int x) { return 2 * x; }"
    assert bench._code_text(c) != bench._code_text(a)


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """A record is reported only while its kernel's sources hash to the recorded
    value (a record of other sources reads as null)."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    cur = bench.csrc_hash("norm_bwd")
    (prof / "traffic.tsv").write_text(
        "kernel\tworkload\tdram_bytes_per_launch\tcsrc_hash\n"
        f"norm_bwd\tw_now\t123\t{cur}\n"
        "norm_bwd\tw_old\t456\t000000000000\n")
    csrc = tmp_path / "mlp_block_backprop_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES["norm_bwd"]:
        src = os.path.join(ROOT, "mlp_block_backprop_gb300", "csrc", name)
        (csrc / name).write_text(open(src, encoding="utf-8").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w_now", "norm_bwd") == 123
    assert bench.recorded_traffic("w_old", "norm_bwd") is None
    assert bench.recorded_traffic("w_missing", "norm_bwd") is None
