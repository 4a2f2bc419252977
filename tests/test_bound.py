"""The bound calculator against the numbers the pages print (tests/golden/pages_numbers.txt)."""
import os

import pytest

import synth
from autoregressive_decode_persistent_gb300 import bound

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    out = {}
    with open(os.path.join(HERE, "golden", "pages_numbers.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()[:2]
                out[k] = float(v)
    return out


G = _golden()


def test_bandwidth_bound_matches_pages():
    # 2B params at 2 bytes each on the two 8-GPU nodes -> the printed 7,700..8,400 tokens/s
    lo = bound.page_bound(G["node_bandwidth_TBps_8xH200"] * 1e12, G["model_params_billion"] * 1e9, 2)
    hi = bound.page_bound(G["node_bandwidth_TBps_8xMI300X"] * 1e12, G["model_params_billion"] * 1e9, 2)
    assert lo == pytest.approx(7675.0)
    assert hi == pytest.approx(8400.0)
    assert round(lo, -2) == G["bound_tokens_per_s_low"]
    assert round(hi, -2) == G["bound_tokens_per_s_high"]
    # the fp16 model is the printed 4 GB
    assert 2 * G["model_params_billion"] == G["fp16_model_gigabytes"]


def test_launch_overhead_model_matches_pages():
    t = bound.launch_overhead_per_token_s(G["launch_overhead_us"] * 1e-6, int(G["kernels_per_layer"]),
                                          int(G["layers"]))
    assert t * 1e6 == pytest.approx(G["launch_overhead_us_per_token"])
    assert round(1.0 / t, -1) == G["launch_cap_tokens_per_s"]


def test_time_budget_matches_pages():
    per_tok = bound.per_token_budget_s(G["fast_tokens_per_s"]) * 1e6
    assert int(per_tok) == G["budget_us_per_token"]
    assert round(per_tok / G["layers"], 1) == G["budget_us_per_layer"]


def test_agent_example_matches_pages():
    slow = bound.generation_time_s(G["agent_tokens"], G["slow_tokens_per_s"])
    fast = bound.generation_time_s(G["agent_tokens"], G["fast_tokens_per_s"])
    assert round(slow / 60) == G["slow_minutes"]
    assert fast < G["fast_seconds_below"]


def test_fp8_moe_projection_matches_pages():
    # 5.1B active parameters at 1 byte each is the printed 5.1 GB
    assert G["moe_active_params_billion"] * 1 == G["moe_fp8_gigabytes"]


def test_bytes_per_token_of_workloads():
    c = synth.get_config("dense-2.3b-fp16")
    # closed form: 25 layers x (2 d^2 + 2 d*hkv*hd + 3 d*ff + 2 d) + V d + 2 d, at 2 bytes
    d, L, ff, V = 2560, 25, 9728, 32000
    params = L * (2 * d * d + 2 * d * 512 + 3 * d * ff + 2 * d) + V * d + 2 * d
    assert bound.weight_bytes_per_token(c) == 2 * params == 4_686_090_240
    # total parameter count of the model (tied embedding counted once) is the pages' 2.3B class
    assert synth.configs.n_params(c) == 2_343_042_560
    assert bound.kv_read_bytes(c, 1) == 2 * 25 * 4 * 128 * 2
    # the pages' bound applied to this model's own byte count on one 8 TB/s GPU
    tok_s = bound.roofline_tokens_per_s(c, 768.5, 8e12)
    assert tok_s == pytest.approx(8e12 / (4_686_090_240 + 51_200 + 51_200 * 768.5))
    c8 = synth.get_config("dense-8b-bf16")
    assert bound.weight_bytes_per_token(c8) == 15_009_857_536
    cm = synth.get_config("moe-32x1408-top4-e4m3")
    assert bound.weight_bytes_per_token(cm) == 1_470_078_976


def test_mean_bytes_per_token_is_average_of_steps():
    c = synth.get_config("tiny")
    steps = [bound.bytes_per_token(c, 17 + i) for i in range(64)]
    assert bound.mean_bytes_per_token(c, 17, 64) == pytest.approx(sum(steps) / len(steps))


def test_batched_step_bytes():
    """A batched step reads the weights once and each request's own KV prefix: with one request it
    is the single-request step; each extra request adds exactly its KV read and write."""
    c = synth.get_config("dense-2.3b-fp16")
    assert bound.batch_step_bytes(c, [700]) == bound.bytes_per_token(c, 700)
    two = bound.batch_step_bytes(c, [513, 1024])
    assert two == bound.bytes_per_token(c, 513) + bound.bytes_per_token(c, 1024) - bound.weight_bytes_per_token(c)
    # KV row of the 2.3B model: 25 layers x 4 KV heads x 128 dims x 2 (K, V) x 2 bytes = 51,200
    assert bound.batch_step_bytes(c, [10, 10]) - bound.batch_step_bytes(c, [10, 9]) == 51_200
    steps = [bound.batch_step_bytes(c, [513 + i] * 3) for i in range(512)]
    assert bound.mean_batch_step_bytes(c, 3, 513, 512) == pytest.approx(sum(steps) / len(steps))
