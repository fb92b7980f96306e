"""The benchmark's reference arm (the fp64 oracle on the host cores) prints
one JSON line with the fields of the benchmark contract (CPU only)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "llama60m_block", "--steps", "1", "--warmup", "1", "--cpu-tokens", "16"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["config"]["workload"] == "llama60m_block"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["vs_baseline"] is None and line["higher_is_better"] is True
    # the same sample definition as the cpu_baseline leg, and the config the
    # GPU arm prints for the same arguments (cuda_graph included)
    assert "16 tokens per step" in line["cpu_baseline"]["sample"]
    sys.path.insert(0, ROOT)
    import bench
    import synth
    wl = synth.WORKLOADS["llama60m_block"]

    class A:  # the arguments above, with the defaults of the other options
        mode, weight, optimizer, gpus, graph, concurrent = "cayley", "dense", "none", 1, "auto", "on"
    assert line["config"] == bench.workload_config(wl, wl.block_sizes[0], A)
    assert line["config"]["cuda_graph"] is True
