"""Host-side logic of bench.py that needs no GPU: the DRAM-traffic and
instruction records are read only while the kernel sources match their
digest, the bytes per parameter of each step kind, the oracle sample sizes,
the reference arm's JSON line for every step kind, and the timed oracle
itself (each step kind on a small sample)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("kind", sorted(bench.TRAFFIC_RECORDS))
def test_records_match_the_committed_sources(kind):
    """A record that matches the kernel sources holds per-parameter traffic
    near the algorithmic bytes (reads exact, writes at most one L2's worth
    short).  A stale record (sources changed since the capture) is reported
    as null by the benchmark and skipped here until it is retaken."""
    if not os.path.exists(os.path.join(ROOT, "profiles", bench.TRAFFIC_RECORDS[kind][0])):
        pytest.fail(f"{kind}: traffic record missing")
    rec = bench.recorded_traffic(kind)
    if rec is None:
        pytest.skip(f"{kind}: the kernel sources changed since the traffic was captured")
    for n_d, bytes_per_param in rec.items():
        algorithmic = bench.step_bytes_per_param(kind, n_d)
        assert 0.95 * algorithmic <= bytes_per_param <= algorithmic + 0.01, (kind, n_d, bytes_per_param)


def test_records_go_stale_with_the_sources(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_digest", lambda kind="adam": "0000000000000000")
    assert bench.recorded_traffic("adam") is None
    assert bench.recorded_traffic("adam8") is None
    assert bench.recorded_instructions("adam8") is None


def test_instruction_record_and_issue_peak():
    instr = bench.recorded_instructions("adam8")
    if instr is None:
        pytest.skip("adam8: the kernel sources changed since the instructions were counted")
    assert 60 < instr[4] < 200
    assert abs(bench.ISSUE_PEAK_TINSTR_S - 152 * 4 * 32 * 2.07e9) < 1


def test_bytes_per_param_and_samples():
    assert bench.step_bytes_per_param("adam", 4) == 34
    assert bench.step_bytes_per_param("sgd", 64) == 146
    assert bench.step_bytes_per_param("adam8", 16) == 46 + 16 / 2048
    assert bench.oracle_sample("adam8", 10 ** 9) == 1_000_000
    assert bench.oracle_sample("adam", 10 ** 9) == 4_000_000
    assert bench.oracle_sample("sgd", 1000) == 1000


@pytest.mark.parametrize("optimizer", ["adam", "sgd", "adam8"])
def test_oracle_throughput_each_kind(optimizer):
    from zero_partitioned_mixed_partition_gb300 import synth
    g, steps, seconds, threads = bench.oracle_throughput(synth.WORKLOADS["tiny"], 20_000, 0.0, 3, optimizer)
    assert g > 0 and steps == 1 and threads == 3


@pytest.mark.parametrize("optimizer", ["adam", "adam8"])
def test_reference_arm_line(optimizer):
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the contract's keys and the step kind's bytes per parameter."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--optimizer", optimizer,
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["bytes_per_param"] == round(bench.step_bytes_per_param(optimizer, 4), 4)
    assert optimizer in line["cpu_baseline"]["sample"]


def test_step_api_names():
    """The config of every line names the C-ABI entry point one timed step calls."""
    import argparse
    def ns(**kw):
        base = dict(optimizer="adam", clip=0.0, api="async")
        base.update(kw)
        return argparse.Namespace(**base)
    assert bench.step_api_name(ns()) == "zero_shard_step_async"
    assert bench.step_api_name(ns(api="sync")) == "zero_shard_step"
    assert bench.step_api_name(ns(api="noalloc")) == "zero_shard_step_noalloc"
    assert bench.step_api_name(ns(clip=1.0)) == "zero_shard_step_clipped_async"
    assert bench.step_api_name(ns(optimizer="sgd")) == "zero_shard_step_sgd_async"
    assert bench.step_api_name(ns(optimizer="adam8")) == "zero_shard_step_adam8_async"
