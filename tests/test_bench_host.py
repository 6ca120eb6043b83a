"""Host logic of bench.py (no GPU): the kernel-source hash that keys the
committed ncu summaries ignores comments and whitespace but not code, and
a summary is looked up per state dtype."""
import os

import bench


def _write(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return p


def test_source_hash_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write(tmp_path, "a.cu", "int f(int x) {  // add one\n  return x + 1;\n}\n")
    h0 = bench.source_hash(["a.cu"])
    _write(tmp_path, "a.cu", "/* header */\nint f(int x) {\n\n  return x + 1;   // still one\n}\n")
    assert bench.source_hash(["a.cu"]) == h0
    _write(tmp_path, "a.cu", "int f(int x) {\n  return x + 2;\n}\n")
    assert bench.source_hash(["a.cu"]) != h0


def test_profiled_traffic_is_keyed_by_state_dtype_and_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    _write(tmp_path, "k.cu", "int g() { return 3; }\n")
    sha = bench.source_hash(["k.cu"])
    _write(tmp_path, "profiles/verify_w.md", f"traffic_bytes_per_launch: 100\nsource_sha: {sha}\n")
    assert bench.profiled_traffic("verify", "w", ["k.cu"]) == 100.0
    # no bf16 summary: a bf16 run reports no traffic rather than the fp32 one
    assert bench.profiled_traffic("verify", "w", ["k.cu"], "bf16") is None
    _write(tmp_path, "profiles/verify_w_bf16.md", f"traffic_bytes_per_launch: 50\nsource_sha: {sha}\n")
    assert bench.profiled_traffic("verify", "w", ["k.cu"], "bf16") == 50.0
    # a code change makes the summary stale
    _write(tmp_path, "k.cu", "int g() { return 4; }\n")
    assert bench.profiled_traffic("verify", "w", ["k.cu"]) is None

