"""The benchmark's output contract, on CPU: the engine line carries every key the harness reads
(formatted from a synthetic measurement), and the reference arm (the CPU oracle) prints its
line on a real, bounded run."""
import json
import subprocess
import sys
import types

import pytest

ROOT = __import__("os").path.dirname(__import__("os").path.dirname(__import__("os").path.abspath(__file__)))

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "e2e", "roofline", "gpu_launches", "clocks")


def test_engine_line_has_the_contract_keys(capsys):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    cfg = synth.get_config("dense-2.3b-fp16")
    res = {"ms": 1000.0, "steps": 1024, "n_launch": 2, "step_pct": {"p50_us": 1.0, "p99_us": 2.0},
           "weight_bytes": 4686090240, "achieved_gbs": 3800.0, "per_launch_bytes": 2.4e12, "launch_ms": 500.0,
           "peak": 6757.9, "peak_kind": "measured", "e2e": 800.0, "n_e2e": 1024,
           "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}, "ctas": 152,
           "image_bytes": 1, "launches": 2, "ablation": None,
           "cpu": {"value": 4.2, "unit": "tokens/s", "cores": 16, "kind": "oracle", "sample": "x"}}
    bench.emit_engine(types.SimpleNamespace(warmup=16, layers=0), cfg, res, 1)
    line = json.loads(capsys.readouterr().out.strip())
    for k in REQUIRED:
        assert k in line, k
    assert line["value"] == pytest.approx(1024.0)  # 1024 steps in 1 s
    assert line["config"]["workload"].startswith("dense-2.3b-fp16")
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert set(line["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert line["roofline"]["frac"] == pytest.approx(3800.0 / 6757.9, rel=1e-3)
    assert line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.slow
def test_reference_arm_prints_its_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                          "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] == 3
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
