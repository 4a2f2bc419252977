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


def _engine_res(**kw):
    res = {"ms": 1000.0, "runs_ms": [1010.0, 1000.0, 990.0], "steps": 1024, "n_launch": 2,
           "step_pct": {"p50_us": 1.0, "p99_us": 2.0},
           "weight_bytes": 4686090240, "achieved_gbs": 3800.0, "per_launch_bytes": 2.4e12, "launch_ms": 500.0,
           "peak": 6757.9, "peak_kind": "measured", "read_gbs": 7000.0, "e2e": 800.0, "n_e2e": 1024,
           "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}, "ctas": 152,
           "image_bytes": 1, "launches": 2, "ablation": None,
           "cpu": {"value": 4.2, "unit": "tokens/s", "cores": 16, "kind": "oracle", "sample": "x"}}
    res.update(kw)
    return res


@pytest.mark.parametrize("workload,window,prompt", [("dense-2.3b-fp16-long-t0.7", 512, 3584),
                                                    ("dense-8b-bf16", 256, 1024),
                                                    ("moe-32x1408-top4-e4m3", 512, 256)])
def test_other_workload_lines_name_their_run(capsys, monkeypatch, workload, window, prompt):
    """--workload lines describe the run they time: shape, prompt, contexts, sampling, stored types."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    monkeypatch.setattr(bench, "WORKLOAD", workload)
    monkeypatch.setattr(bench, "WINDOW", bench.WORKLOADS[workload]["window"])
    cfg = synth.get_config(workload)
    bench.emit_engine(types.SimpleNamespace(warmup=16, layers=0), cfg, _engine_res(steps=window, n_launch=1), 1)
    line = json.loads(capsys.readouterr().out.strip())
    for k in REQUIRED:
        assert k in line, k
    assert line["metric"] == bench.WORKLOADS[workload]["metric"]
    assert line["config"]["prompt"] == prompt
    assert line["config"]["contexts"] == f"{prompt + 1}..{prompt + window}"
    assert line["config"]["workload"].startswith(workload) and f"prompt {prompt}" in line["config"]["workload"]
    assert cfg["kv_dtype"] in line["dtype"] and "f32 accumulation" in line["dtype"]
    if workload.endswith("t0.7"):
        assert line["config"]["temperature"] == 0.7 and "sampling" in line["config"]["workload"]
    if workload.startswith("moe"):
        assert "e4m3 experts" in line["dtype"] and "top-4" in line["config"]["workload"]
    assert line["roofline"]["frac_of_read_probe"] == pytest.approx(3800.0 / 7000.0, rel=1e-3)


def test_engine_line_has_the_contract_keys(capsys):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    cfg = synth.get_config("dense-2.3b-fp16")
    res = {"ms": 1000.0, "runs_ms": [1000.0, 1001.0, 999.0], "steps": 1024, "n_launch": 2,
           "step_pct": {"p50_us": 1.0, "p99_us": 2.0},
           "weight_bytes": 4686090240, "achieved_gbs": 3800.0, "per_launch_bytes": 2.4e12, "launch_ms": 500.0,
           "peak": 6757.9, "peak_kind": "measured", "read_gbs": 7000.0, "e2e": 800.0, "n_e2e": 1024,
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
    assert line["dtype"] == "f16 weights, f16 KV cache, f32 accumulation and activations"
    assert len(line["config"]["runs_tokens_per_s"]) == 3


@pytest.mark.slow
def test_reference_arm_prints_its_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                          "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] == 3
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_batch_line_has_the_contract_keys(capsys):
    """--batch N: value counts the tokens of all requests; the roofline is the batched kernel's."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    cfg = synth.get_config("dense-2.3b-fp16")
    res = {"ms": 1000.0, "steps": 512, "nb": 3, "n_launch": 1, "step_pct": {"p50_us": 1.0, "p99_us": 2.0},
           "weight_bytes": 4686090240, "achieved_gbs": 2100.0, "per_launch_bytes": 2.46e12, "launch_ms": 1000.0,
           "peak": 6757.9, "peak_kind": "measured", "e2e": 1300.0, "n_e2e": 512,
           "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10}, "ctas": 152,
           "launches": 1}
    bench.emit_batch(types.SimpleNamespace(warmup=8, layers=0), cfg, res, 1)
    line = json.loads(capsys.readouterr().out.strip())
    for k in REQUIRED:
        assert k in line, k
    assert line["value"] == pytest.approx(3 * 512.0)
    assert line["config"]["batch"] == 3 and line["higher_is_better"] is True
    assert line["roofline"]["kernel"] == "adp::decode_batch_kernel"
    assert line["e2e"]["d2h_bytes_per_step"] == 16


def test_prefill_line_has_the_contract_keys(capsys):
    """--prefill: time to first token (lower is better), roofline of the tensor-core GEMM."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    cfg = synth.get_config("dense-2.3b-fp16-long-t0.7")
    res = {"dev_ms": 31.0, "host_ms": 31.5, "step_ms": 4700.0, "P": 3584, "gemm_ms": 0.333,
           "gemm_flops": 2.0 * 3583 * 19456 * 2560, "gemm_shape": (3583, 19456, 2560),
           "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 4}, "ctas": 152,
           "n_layers": 25}
    bench.emit_prefill(types.SimpleNamespace(warmup=3, steps=5, layers=0), cfg, res, 1)
    line = json.loads(capsys.readouterr().out.strip())
    for k in REQUIRED:
        assert k in line, k
    assert line["higher_is_better"] is False and line["unit"] == "ms" and line["value"] == pytest.approx(31.0)
    assert line["roofline"]["bound"] == "tensor" and line["roofline"]["unit"] == "TFLOP/s"
    assert line["roofline"]["achieved"] == pytest.approx(2.0 * 3583 * 19456 * 2560 / 0.333e-3 / 1e12, rel=1e-3)
    assert line["gpu_launches"] == 1 + 7 * 25 + 1
