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
    ("dense-8b-e4m3", 1024, 3, 0.0),
    ("dense-8b-nvfp4", 1024, 2, 0.0),
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
    oracle run step by step from an empty cache: bit-exact against its contract mode, within the
    stated tolerances of its plain mode."""
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
    got = [lg.cpu().numpy().copy()]
    toks = [int(t) for t in prompt]
    assert np.array_equal(got[0].view(np.uint32), out["logits"].view(np.uint32))
    for _ in range(2):
        ref = om.step(nxt, EXACT)
        toks.append(nxt)
        nxt = kv.step(nxt, logits=lg)
        assert nxt == ref["next"]
        got.append(lg.cpu().numpy().copy())
        assert np.array_equal(got[-1].view(np.uint32), ref["logits"].view(np.uint32))
    k, v = kv.read()
    assert np.array_equal(k, om.kc[:, :, :18]) and np.array_equal(v, om.vc[:, :, :18])
    ref_p, _, _ = oracle_forced(cfg, W, toks, PLAIN)
    assert_logits_within_tolerance(np.stack([got[0]] + got[1:]), ref_p[15:])


@pytest.mark.parametrize("name", ["dense-2.3b-fp16", "dense-2.3b-nvfp4"])
def test_full_size_batch(built, name):
    """A 2.3B workload (fp16, and NVFP4 layer matrices) decoded as a batch of as many requests as
    the model can batch, each with its own KV prefix (lengths 512, 700, 1000), teacher-forced for 3
    steps: per request bit-exact against the oracle's contract mode and within tolerance of its
    plain mode."""
    import torch
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    cfg = synth.get_config(name)
    W = _weights(cfg)
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


_WEIGHTS = {}


def _weights(cfg):
    """Seeded weights of a full-size workload, generated once per test module and model."""
    key = (cfg["n_layers"], cfg["d_model"], cfg["weight_dtype"], cfg["index"])
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        _WEIGHTS[key] = synth.model_weights(cfg)
    return _WEIGHTS[key]


def _generate_case(cfg, prefix_kv, prefix_len, first, n, temperature=0.0, prefill=None):
    """adp_generate_async (the benchmarked launch: n chained steps in one persistent kernel) from a
    cache of prefix_len positions, against the oracle's contract-mode free run from the same cache:
    every chosen token and every new K/V row bit for bit.  The engine's cache is loaded from
    prefix_kv, or, with prefill = (tokens, expected next token), written by adp_prefill of those
    tokens (and then checked against prefix_kv bit for bit).  Returns the engine model and cache
    (at prefix_len + n positions) and the oracle's input and chosen tokens."""
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    W = _weights(cfg)
    us = synth.sampling_uniforms(n, first=prefix_len) if temperature > 0 else None
    toks, _, nexts, _, om = oracle_free_run(cfg, W, [first], n - 1, EXACT, temperature, us, prefix_kv)
    model = DecodeModel(cfg, W)
    kv = model.new_kv()
    if prefill is not None:
        assert kv.prefill(prefill[0]) == prefill[1]
        k, v = kv.read()
        assert np.array_equal(k, prefix_kv[0]) and np.array_equal(v, prefix_kv[1])
    else:
        kv.load(*prefix_kv)
    assert len(kv) == prefix_len
    out = torch.empty(n, dtype=torch.int32, device=model.device)
    dev_u = torch.tensor(us, dtype=torch.float32, device=model.device) if us is not None else None
    kv.generate_async(first, n, out, temperature, dev_u)
    adp.adp_sync(model.handle)
    assert out.cpu().tolist() == nexts
    m = prefix_len + n
    k, v = kv.read()
    assert len(kv) == m
    assert np.array_equal(k[:, :, prefix_len:m], om.kc[:, :, prefix_len:m])
    assert np.array_equal(v[:, :, prefix_len:m], om.vc[:, :, prefix_len:m])
    return model, kv, toks, nexts


def test_full_size_generate_async_after_a_512_position_prefix(built):
    """The benchmarked path itself: dense-2.3b-fp16, 16 chained steps in one launch after a
    512-position cache; then one more step's logits against the plain oracle on the same tokens."""
    import torch
    cfg = synth.get_config("dense-2.3b-fp16")
    kvp = synth.kv_prefix(cfg, 512)
    first = int(synth.prompt(cfg, 1)[0])
    model, kv, toks, nexts = _generate_case(cfg, kvp, 512, first, 16)
    lg = torch.empty(cfg["vocab"], device=model.device)
    kv.step(nexts[-1], logits=lg)
    model.close()
    ref_p, _, _ = oracle_forced(cfg, _weights(cfg), toks + [nexts[-1]], PLAIN, kv_prefix=kvp)
    assert_logits_within_tolerance(lg.cpu().numpy()[None], ref_p[-1:])


def test_full_size_generate_async_on_a_prefilled_prompt(built):
    """The same path on a cache that adp_prefill wrote from a real prompt (the first 23 tokens of
    the workload's prompt stream, through the decode kernel) rather than a synthetic prefix: the
    oracle prefills the same tokens itself, then both generate 8 chained steps from the 24th."""
    from oracle import OracleModel
    cfg = synth.get_config("dense-2.3b-fp16")
    prompt = [int(t) for t in synth.prompt(cfg, 24)]
    om = OracleModel(cfg, _weights(cfg))
    out = om.prefill(prompt[:-1], EXACT)
    kvp = (om.kc[:, :, :23].copy(), om.vc[:, :, :23].copy())  # the oracle's own prefill
    model, _, _, _ = _generate_case(cfg, kvp, 23, prompt[-1], 8, prefill=(prompt[:-1], out["next"]))
    model.close()


@pytest.mark.parametrize("name,prefix,steps,temperature", [
    ("dense-2.3b-fp16-long-t0.7", 4092, 4, 0.7),   # contexts 4093..4096 = max_ctx
    ("dense-8b-bf16", 1277, 3, 0.0),               # contexts 1278..1280, the workload's last
])
def test_full_size_run_to_the_last_context(built, name, prefix, steps, temperature):
    """Full-size runs that end at the workload's last context (for the long-context workload that is
    max_ctx: the attention partial buffers' last block is used): the chained launch bit-exact against
    the contract; the same steps through adp_decode_step within tolerance of the plain oracle; one
    step more at max_ctx is refused with ADP_ERR_CONTEXT_OVERFLOW."""
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config(name)
    kvp = synth.kv_prefix(cfg, prefix)
    first = int(synth.prompt(cfg, 1)[0])
    model, kv, toks, nexts = _generate_case(cfg, kvp, prefix, first, steps, temperature)
    if prefix + steps == cfg["max_ctx"]:
        with pytest.raises(adp.AdpError) as e:
            kv.step(nexts[-1])
        assert e.value.code == adp.ADP_ERR_CONTEXT_OVERFLOW
    us = synth.sampling_uniforms(steps, first=prefix) if temperature > 0 else None
    got, next_g, _, _, _ = engine_forced(model, toks, temperature, us, kvp)
    model.close()
    assert next_g == nexts
    ref_p, _, _ = oracle_forced(cfg, _weights(cfg), toks, PLAIN, temperature, us, kvp)
    assert_logits_within_tolerance(got, ref_p)
