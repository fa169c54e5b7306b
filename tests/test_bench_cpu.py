"""Host-side checks of bench.py (no GPU): the byte model against the tensors a call moves, the
traffic record's tie to the kernel sources, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("name", ["tiny", "layer_r3277"])
def test_algorithmic_bytes_are_the_bytes_a_call_reads_and_writes(name):
    """The roofline's byte count equals the sizes of the call's inputs (q, k, v in their dtype,
    g, beta, cu_seqlens) plus its outputs (O in the input dtype, the fp32 final states)."""
    x = bench.make_inputs(name)
    e = 2 if x.dtype == "bf16" else 4
    inputs = (x.q.size + x.k.size + x.v.size) * e + (x.g.size + x.beta.size) * 4 + x.cu_seqlens.size * 4
    outputs = x.total_tokens * x.h_v * x.d_v * e + x.n_seqs * x.h_v * x.d_v * x.d_k * 4
    _, byts = bench.algorithmic(x)
    assert byts == inputs + outputs
    _, byts_state_only = bench.algorithmic(x, with_O=False)
    assert byts - byts_state_only == x.total_tokens * x.h_v * x.d_v * e


def test_recorded_traffic_is_dropped_when_the_sources_change(monkeypatch):
    got = bench.recorded_traffic("layer_r3277")
    assert got is None or got > 0
    monkeypatch.setattr(bench, "source_digest", lambda: "0" * 16)
    assert bench.recorded_traffic("layer_r3277") is None
    assert bench.recorded_traffic("no_such_workload") is None


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 1 and d["warmup"] == 1 and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "layer_r3277"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert np.isfinite(d["ms_per_step"]) and d["ms_per_step"] > 0
