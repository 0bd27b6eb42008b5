"""bench.py's JSON contract on the CPU: the reference arm (the fp64 oracle timed on the host
cores) prints one line with the contract's keys, and the GPU arm refuses to run without a
GPU instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=300):
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                          timeout=timeout)


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--workload", "tiny_bf16", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_bf16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU refusal")
def test_gpu_arm_refuses_without_gpu():
    r = _bench("--workload", "tiny_bf16", "--steps", "1", "--warmup", "0", timeout=120)
    assert r.returncode != 0
    assert "needs a CUDA GPU" in (r.stdout + r.stderr)
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_traffic_records_are_hash_locked(monkeypatch):
    """The DRAM traffic a bench line reports comes from profiles/traffic.json, and only while
    the kernel's sources hash to the profiled build: every record names an existing profile
    summary that carries its hash, and a changed source hash turns the figure off."""
    sys.path.insert(0, ROOT)
    import bench

    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)["entries"]
    assert entries
    for e in entries:
        assert e["kernel"] in bench.PARTITION_SOURCES
        summary = os.path.join(ROOT, e["from"].split(" ")[0])
        assert os.path.exists(summary), e["from"]
        with open(summary) as f:
            assert e["source_hash"] in f.read(), summary
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"]
        monkeypatch.setattr(bench, "source_hash", lambda kernel, h=e["source_hash"]: h)
        assert bench.recorded_traffic(e["kernel"], e["workload"]) == e["dram_bytes_per_launch"]
        monkeypatch.setattr(bench, "source_hash", lambda kernel: "0" * 16)
        assert bench.recorded_traffic(e["kernel"], e["workload"]) is None
