"""Host-side logic of bench.py that needs no GPU.

- The reference arm (``--impl reference``): the CPU oracle timed on the host
  cores prints one JSON line with the contract's keys (``impl``, the metric
  and unit of the native arm, a ``cpu_baseline`` of kind ``oracle`` and an
  ``e2e`` with no host-device bytes); under torchrun only rank 0 prints.
- The ncu traffic figure is reported only while the kernel's sources are the
  ones the counters were taken on: the source digest ignores comments and
  blank space, and changes with any code token.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run_reference(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--ref-seconds", "1",
           "--steps", "2", "--warmup", "3", *args]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("workload", ["mamba2_bs256", "gdn_bs256"])
def test_reference_arm_line(workload):
    r = _run_reference(None, "--workload", workload)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == bench.WORKLOADS[workload]["desc"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert isinstance(cb["cores"], int) and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_code_digest_ignores_comments_only():
    src = "// kernel\nint f(int x) {\n  return x + 1;  // add one\n}\n/* block\n comment */\n"
    same = "int f(int x) {\n\n  return x + 1;\n}\n"
    changed = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_digest([src]) == bench.code_digest([same])
    assert bench.code_digest([src]) != bench.code_digest([changed])
    # the order of the files is part of the digest
    assert bench.code_digest([src, changed]) != bench.code_digest([changed, src])


def test_traffic_reported_only_for_the_profiled_sources(monkeypatch):
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    with open(path) as f:
        rec = json.load(f)
    k = "mamba2_replay"
    assert rec[k]["workload"] == "mamba2_bs256"
    # the committed record matches the committed sources
    assert bench._kernel_traffic(k, "mamba2_bs256") == rec[k]["dram_bytes_per_launch"]
    # another workload, or a changed kernel, gives no figure
    assert bench._kernel_traffic(k, "gdn_bs256") is None
    monkeypatch.setattr(bench, "source_hash", lambda kernel: "0" * 64)
    assert bench._kernel_traffic(k, "mamba2_bs256") is None
