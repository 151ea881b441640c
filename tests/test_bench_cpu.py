"""Host-side parts of bench.py: the workload config, the hash-gated traffic
record and the reference arm's JSON line (the CPU oracle; no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from compressed_composable_kv_gb300 import synth as S  # noqa: E402


@pytest.mark.parametrize("name", sorted(S.WORKLOADS))
def test_workload_config_names_the_workload_and_its_sizes(name):
    w = S.WORKLOADS[name]
    c = bench.workload_config(w, 2)
    assert c["workload"] == name and "model" not in c
    assert c["batch"] == w.batch and len(c["composed_slots"]) == w.batch
    assert c["question_tokens"] == w.q_len and c["decode_steps"] == w.decode_steps
    assert c["parallelism"] == "replicas x2"
    assert all(s >= 1 for s in c["composed_slots"])
    assert all(t >= s for t, s in zip(c["original_tokens"], c["composed_slots"]))


def test_default_workload_sizes():
    """The largest workload that fits one GPU: 4 sequences, each 32 documents
    of 4096 tokens at k = 4, i.e. 32 768 slots of 131 072 tokens."""
    c = bench.workload_config(S.WORKLOADS[bench.DEFAULT_WORKLOAD], 1)
    assert c["composed_slots"] == [32768] * 4 and c["original_tokens"] == [131072] * 4


def test_traffic_record_applies_only_to_the_captured_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "a.cu").write_text("kernel A\n")
    (tmp_path / "b.h").write_text("header B\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.sources_sha("a.cu,b.h")
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment\n\nother_kernel a.cu 0000000000000000 1.0\n"
        f"decode_kernel a.cu,b.h {sha} 4105.1\n")
    assert bench.profiled_traffic("decode_kernel") == 4105.1
    assert bench.profiled_traffic("missing_kernel") is None
    assert bench.profiled_traffic("other_kernel") is None      # hash does not match
    (tmp_path / "b.h").write_text("header B, edited\n")
    assert bench.profiled_traffic("decode_kernel") is None     # a source changed since the capture
    (tmp_path / "profiles" / "traffic.txt").unlink()
    assert bench.profiled_traffic("decode_kernel") is None


def test_committed_traffic_record_parses():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert any(r[0] == "decode_tc_kernel" for r in rows)
    for r in rows:
        for src in r[1].split(","):
            assert os.path.exists(os.path.join(ROOT, src)), src
        assert len(r[2]) == 16 and float(r[3]) > 0


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the oracle on the host and prints one
    JSON line with the keys the contract asks for."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tok/s"
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0)) and d["cpu_baseline"]["sample"]
    # the step time is the work the step ran, not the extrapolated request
    assert 0 < d["ms_per_step"] < 60e3 and d["extrapolated_request_s"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
