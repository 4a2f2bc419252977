"""Full-size workloads on the GPU, in the launch configuration the benchmark times (persistent
kernel, one CTA per SM), against the CPU oracle on sampled steps.

Each case loads a synthetic KV prefix of the workload's prompt length into both the engine and
the oracle (the cache is the whole decode state; its contents are seeded N(0,1) values in the KV
dtype), then decodes a few steps teacher-forced on the oracle's tokens: bit-exact against the
oracle's contract mode (logits, tokens, every new KV row, MoE routing) and within the stated
tolerances against its plain fp32 mode."""
import numpy as np
import pytest

import synth
from oracle import EXACT, PLAIN

from gpu_common import assert_logits_within_tolerance, engine_forced, oracle_forced, oracle_free_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    import torch
    assert torch.cuda.is_available()
    from autoregressive_decode_persistent_gb300 import build
    build.build()


@pytest.mark.parametrize("name,prefix,steps,temperature", [
    ("dense-2.3b-fp16", 512, 6, 0.0),
    ("dense-2.3b-fp16-long-t0.7", 3584, 4, 0.7),
    ("dense-8b-bf16", 1024, 3, 0.0),
    ("moe-32x1408-top4-e4m3", 256, 5, 0.0),
    ("dense-2.3b-e4m3", 512, 5, 0.0),
    ("dense-2.3b-nvfp4", 512, 5, 0.0),
])
def test_full_size_workload(built, name, prefix, steps, temperature):
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    cfg = synth.get_config(name)
    W = synth.model_weights(cfg)
    kvp = synth.kv_prefix(cfg, prefix)
    first = synth.prompt(cfg, 1)
    us = synth.sampling_uniforms(steps, first=prefix) if temperature > 0 else None
    toks, ref_e, next_e, experts_e, om = oracle_free_run(cfg, W, first, steps - 1, EXACT, temperature, us, kvp)
    model = DecodeModel(cfg, W)
    got, next_g, k, v, experts_g = engine_forced(model, toks, temperature, us, kvp,
                                                 read_experts=bool(cfg["n_experts"]))
    model.close()
    n = prefix + len(toks)
    assert next_g == next_e
    assert np.array_equal(got.view(np.uint32), ref_e.view(np.uint32))
    assert np.array_equal(k[:, :, prefix:n], om.kc[:, :, prefix:n])
    assert np.array_equal(v[:, :, prefix:n], om.vc[:, :, prefix:n])
    assert np.array_equal(k[:, :, :prefix], kvp[0]) and np.array_equal(v[:, :, :prefix], kvp[1])
    if cfg["n_experts"]:
        for i in range(len(toks)):
            assert np.array_equal(experts_g[i], experts_e[i])
    ref_p, _, _ = oracle_forced(cfg, W, toks, PLAIN, temperature, us, kvp)
    assert_logits_within_tolerance(got, ref_p)


def test_full_size_prefill_path(built):
    """The prompt path at full size: adp_prefill of 16 tokens then 2 decode steps, against the
    oracle run step by step from an empty cache."""
    import torch
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    from oracle import OracleModel
    cfg = synth.get_config("dense-2.3b-fp16")
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg, 16)
    om = OracleModel(cfg, W)
    out = None
    for t in prompt:
        out = om.step(int(t), EXACT)
    model = DecodeModel(cfg, W)
    kv = model.new_kv()
    lg = torch.empty(cfg["vocab"], device=model.device)
    nxt = kv.prefill(prompt, logits=lg)
    assert nxt == out["next"]
    assert np.array_equal(lg.cpu().numpy().view(np.uint32), out["logits"].view(np.uint32))
    for _ in range(2):
        ref = om.step(nxt, EXACT)
        nxt = kv.step(nxt, logits=lg)
        assert nxt == ref["next"]
        assert np.array_equal(lg.cpu().numpy().view(np.uint32), ref["logits"].view(np.uint32))
    k, v = kv.read()
    assert np.array_equal(k, om.kc[:, :, :18]) and np.array_equal(v, om.vc[:, :, :18])


def test_full_size_batch(built):
    """The 2.3B fp16 workload decoded as a batch of as many requests as the model can batch,
    each with its own KV prefix (lengths 512, 700, 1000), teacher-forced for 3 steps: per request
    bit-exact against the oracle's contract mode and within tolerance of its plain mode."""
    import torch
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    cfg = synth.get_config("dense-2.3b-fp16")
    W = synth.model_weights(cfg)
    model = DecodeModel(cfg, W)
    nb = model.max_batch
    assert nb >= 2
    prefixes = [512, 700, 1000, 300][:nb]
    steps = 3
    firsts = synth.batch_prompts(cfg, [1] * nb)
    runs, kvps, kvs = [], [], []
    for r in range(nb):
        kvp = synth.kv_prefix(cfg, prefixes[r], seed=synth.SEED_KV + 50 + r)
        kvps.append(kvp)
        runs.append(oracle_free_run(cfg, W, firsts[r], steps - 1, EXACT, 0.0, None, kvp))
        kv = model.new_kv()
        kv.load(*kvp)
        kvs.append(kv)
    lg = torch.empty((nb, cfg["vocab"]), device=model.device)
    got = []
    for i in range(steps):
        nxt = model.step_batch(kvs, [runs[r][0][i] for r in range(nb)], logits=lg)
        got.append(lg.cpu().numpy().copy())
        for r in range(nb):
            assert nxt[r] == runs[r][2][i], (r, i)
            assert np.array_equal(got[i][r].view(np.uint32), runs[r][1][i].view(np.uint32)), (r, i)
    for r in range(nb):
        k, v = kvs[r].read()
        om, P = runs[r][4], prefixes[r]
        assert np.array_equal(k[:, :, P:P + steps], om.kc[:, :, P:P + steps])
        assert np.array_equal(v[:, :, P:P + steps], om.vc[:, :, P:P + steps])
        ref_p, _, _ = oracle_forced(cfg, W, runs[r][0], PLAIN, 0.0, None, kvps[r])
        assert_logits_within_tolerance(np.stack([g[r] for g in got]), ref_p)
    model.close()
