"""The benchmark's host-side contract, checked on the CPU: the reference arm's one JSON line, the
metric string both arms share, and the rule that a recorded traffic figure is reported only for
the scan code and workload it was captured on."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_top_kv_fathom_gb300 import synth  # noqa: E402

CONTRACT_KEYS = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config"]


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in CONTRACT_KEYS:
        assert key in d, key
    assert d["impl"] == "reference"
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 1)
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["metric"] == bench.metric_name(synth.WORKLOADS["tiny"], 92)
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_metric_name_names_the_workload():
    w = synth.WORKLOADS["million"]
    m = bench.metric_name(w, 92)
    assert "n=%d" % w.n in m and "B=92" in m and "%d-layer" % w.layers in m
    assert m != bench.metric_name(w, 68)


def test_code_tokens_ignore_comments_and_layout():
    a = "int x = 1;  // the first\n\n   float  y;\n// a whole-line comment\n"
    b = "int x = 1;\nfloat y;"
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens("int x = 2;") != bench.code_tokens("int x = 1;")


def test_traffic_is_reported_only_for_the_recorded_source_and_workload(monkeypatch):
    rec = json.load(open(bench.TRAFFIC_RECORD))
    w = synth.WORKLOADS["million"]
    for res in ("host", "device"):
        r = rec[res]
        assert (r["n"], r["rows"]) == (w.n, w.kv_heads)
        monkeypatch.setattr(bench, "scan_source_hash", lambda: rec["scan_source_sha256"])
        assert bench.captured_traffic(res, w, r["budget"]) == r["bytes_per_launch"]
        assert bench.captured_traffic(res, w, r["budget"] + 1) is None  # another workload
        monkeypatch.setattr(bench, "scan_source_hash", lambda: "0" * 64)  # the kernel changed since
        assert bench.captured_traffic(res, w, r["budget"]) is None
