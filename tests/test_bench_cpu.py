"""Host-side checks of bench.py's contract that need no GPU: the reference
arm (the oracle timed on host cores) prints the JSON line the contract asks
for, and a committed ncu DRAM-traffic record is reported only while the
kernel sources it was taken on are unchanged."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_line_on_the_tiny_layer():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny" and d["config"]["tokens"] == 16
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["value"] == pytest.approx(16 / (d["ms_per_step"] * 1e-3))
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == len(os.sched_getaffinity(0)) and cb["value"] == d["value"]
    assert "whole layer" in cb["sample"] and cb["fraction_of_job_step"] == 1.0
    bits = d["config"]["committed_bits"]
    assert len(bits) == 8 and set(d["config"]) >= {"workload", "tokens", "hidden", "intermediate", "experts",
                                                     "top_k", "parent_bits", "seed_bits", "parallelism"}
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_steps_are_timed_passes(monkeypatch):
    d = bench.oracle_reference_steps("tiny", 4, 1)
    assert len(d["step_s"]) == 4 and all(t > 0 for t in d["step_s"])
    assert d["frac"] == 1.0 and "whole layer" in d["sample"]
    # when K + W whole passes would not fit the budget, each step covers a
    # fraction of every block's rows and says so
    monkeypatch.setattr(bench, "REF_BUDGET_S", 1e-6)
    d = bench.oracle_reference_steps("tiny", 2, 0)
    assert 0 < d["frac"] < 1 and "first" in d["sample"]


def test_cpu_baseline_is_a_whole_layer_pass():
    d = bench.oracle_baseline("tiny", passes=1)
    assert d["value"] > 0 and d["cores"] == len(os.sched_getaffinity(0))
    assert d["value"] == pytest.approx(16 / d["layer_s"])


def test_traffic_record_follows_the_kernel_sources(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    kernel, recs = next(iter(records.items()))
    rec = recs[0]
    csrc = os.path.join(ROOT, "any_precision_bit_pw_gb300", "csrc")
    current = bench.source_digest([os.path.join(csrc, name) for name in rec["source_files"]])
    got = bench.measured_traffic(kernel, rec["workload"], rec["tokens"])
    if current == rec["source_sha256"]:
        assert got == float(rec["dram_bytes_per_launch"])
    else:
        assert got is None
    # a source change (here: a different digest) voids the record
    monkeypatch.setattr(bench, "source_digest", lambda paths: "0" * 64)
    assert bench.measured_traffic(kernel, rec["workload"], rec["tokens"]) is None


def test_source_digest_ignores_comments(tmp_path):
    a, b = tmp_path / "a.cuh", tmp_path / "b.cuh"
    a.write_text("int f(int x) {\n  return x + 1;  // one\n}\n")
    b.write_text("/* header */\nint f(int x) {\n\n  return x + 1;\n}\n")
    assert bench.source_digest([str(a)]) == bench.source_digest([str(b)])
    b.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.source_digest([str(a)]) != bench.source_digest([str(b)])


def test_pw_arm_without_a_gpu_fails_at_once():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3"], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "needs a GPU" in r.stderr
    assert not r.stdout.strip()


def test_kernel_routes_follows_the_library_rule():
    """bench.py brackets the fused launch alone when the library routes in a
    launch of its own: batches of at most 32 tokens over at most 8 experts
    with at most 4 slots per token, on the decode path, route in-kernel."""
    import bench
    assert bench.kernel_routes(32, 2, 8)            # the 8x7B decode default
    assert not bench.kernel_routes(33, 2, 8)        # more tokens than one warp routes
    assert not bench.kernel_routes(128, 2, 8)
    assert not bench.kernel_routes(32, 8, 64)       # 60 routed + 4 shared experts
    assert not bench.kernel_routes(32, 9, 129)
    assert not bench.kernel_routes(32, 5, 8)
    assert not bench.kernel_routes(4096, 2, 8)      # prefill path


def test_bits_option_commits_every_block_at_that_bitwidth():
    import bench
    from any_precision_bit_pw_gb300 import synth
    wl = bench.get_workload("mixtral8x7b_uniform_sweep", 8, 3)
    assert wl.tokens == 8 and set(synth.committed_bits(wl)) == {3}
    assert "--bits" in bench._child_cmd("mixtral8x7b_uniform_sweep", 8, 3)
    assert bench.get_workload("mixtral8x7b_decode_mixed").tokens == 32
