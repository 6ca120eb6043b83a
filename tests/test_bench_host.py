"""Host logic of bench.py (no GPU): the kernel-source hash that keys the
committed ncu summaries ignores comments and whitespace but not code, a
summary is looked up per state dtype, `--gpus N` launches N ranks itself,
and the L2 rule picks a flush only for small timed units."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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



def test_gpus_flag_starts_that_many_ranks():
    # Without a torchrun environment, --gpus 2 re-launches bench.py under
    # torchrun with two ranks (gloo on the host for the oracle arm); rank 0
    # alone prints the line, which reports both ranks.
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"
    assert lines[0]["config"]["parallelism"].startswith("replicas x2")


def test_gpus_flag_must_match_world_size(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")
    assert bench.main(["--gpus", "4", "--impl", "reference", "--workload", "tiny"]) == 2
    assert "WORLD_SIZE=2" in capsys.readouterr().err


def test_l2_rule():
    l2 = 126 * 2 ** 20
    on, text = bench.l2_rule(40e6, l2)
    assert on and "flush" in text and "read" in text
    on, text = bench.l2_rule(13.4e9, l2)
    assert not on and text.startswith("no flush")
