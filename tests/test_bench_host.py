"""Host-side logic of bench.py, on the CPU: the algorithmic work behind the
roofline, the staleness check of the recorded DRAM traffic, and the JSON
line of the reference arm (the fp64 oracle timed on the host)."""
import glob
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_forward_algorithmic_work_of_the_long_workload():
    # q, k, v read and o written in bf16: 4·d·2 bytes per token-head; flops
    # 4·d'·d + 4·d' per token-head (d' = d for elu+1)
    flops, nbytes = bench._fwd_alg(W.LONG)
    token_heads = 1 * 16 * 65536
    assert nbytes == token_heads * 128 * 2 * 4 == 1073741824
    assert flops == token_heads * (4 * 128 * 128 + 4 * 128)


def test_performer_work_adds_the_two_projections():
    flops, nbytes = bench._fwd_alg(W.PERFORMER)
    w = W.PERFORMER
    th = w.B * w.H * w.n
    assert nbytes == th * w.d * 2 * 4
    assert flops == th * (4 * w.m * w.d + 4 * w.m + 4 * w.d * w.m)


def test_recorded_traffic_follows_its_sources(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = {"sources": ["k.cu"], "sources_sha": bench._source_sha(["k.cu"]),
             "dram_bytes_per_launch": 12345}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kern": entry}))
    assert bench._traffic("kern") == 12345
    assert bench._traffic("other") is None
    src.write_text("kernel v2\n")          # the kernel changed after the capture
    assert bench._traffic("kern") is None
    src.unlink()                           # or its source is gone
    assert bench._traffic("kern") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    assert {"forward_long", "decode_step"} <= set(t)
    for e in t.values():
        assert e["dram_bytes_per_launch"] > 0
        for s in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, s)), s


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, cwd=ROOT, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == W.LONG.name
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_profile_summaries_run_committed_files_only():
    # every command a summary under profiles/ prints is bench.py with one of
    # its own profile cases (no scratch scripts)
    src = open(os.path.join(ROOT, "bench.py")).read()
    m = re.search(r'"--profile-case",\s*choices=\[(.*?)\]', src, re.S)
    assert m, "bench.py defines --profile-case choices"
    choices = set(re.findall(r'"([a-z0-9-]+)"', m.group(1)))
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path, encoding="utf-8").read()
        for script in re.findall(r"python\s+(\S+\.py)", text):
            assert script == "bench.py", (path, script)
        for case in re.findall(r"--profile-case\s+([a-z0-9-]+)", text):
            assert case in choices, (path, case)
