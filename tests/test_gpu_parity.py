"""Engine (CUDA, through the C ABI) against the CPU oracle, teacher-forced on the oracle's tokens.

Bit-exact against the oracle's EXACT mode (same arithmetic contract): logits, chosen tokens
and every KV-cache row in storage dtype. Within the stated tolerances against the PLAIN
(textbook fp32) mode: logits max-abs <= 2e-2, relative L2 <= 5e-3, argmax equal whenever the
oracle's top-2 margin exceeds 0.05."""
import numpy as np
import pytest

import synth
from oracle import EXACT, PLAIN

from gpu_common import (assert_logits_within_tolerance, engine_forced, oracle_forced, oracle_free_run)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "a CUDA GPU is required"
    from autoregressive_decode_persistent_gb300 import build
    build.build()
    return torch


def _model(cfg, W, mode=0):
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    m = DecodeModel(cfg, W)
    m.set_kernel_mode(mode)
    return m


def _check_case(cfg, prompt_len, n_decode, mode=0, temperature=0.0, kv_prefix_len=0, plain=True):
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg, prompt_len)
    us = synth.sampling_uniforms(prompt_len + n_decode) if temperature > 0 else None
    kvp = synth.kv_prefix(cfg, kv_prefix_len) if kv_prefix_len else None
    toks, ref_e, next_e, experts_e, om = oracle_free_run(cfg, W, prompt, n_decode, EXACT, temperature, us, kvp)
    model = _model(cfg, W, mode)
    got, next_g, k, v, experts_g = engine_forced(model, toks, temperature, us, kvp,
                                                 read_experts=bool(cfg["n_experts"]))
    n = kv_prefix_len + len(toks)
    # bit-exact against the contract
    assert next_g == next_e
    assert np.array_equal(got.view(np.uint32), ref_e.view(np.uint32))
    assert np.array_equal(k, om.kc[:, :, :n]) and np.array_equal(v, om.vc[:, :, :n])
    if cfg["n_experts"]:
        for i in range(len(toks)):
            assert np.array_equal(experts_g[i], experts_e[i])
    if plain:
        ref_p, _, _ = oracle_forced(cfg, W, toks, PLAIN, temperature, us, kvp)
        assert_logits_within_tolerance(got, ref_p)
    model.close()
    return got, k, v


def test_tiny_full_run_bit_exact(torch_cuda):
    cfg = synth.get_config("tiny")
    _check_case(cfg, cfg["prompt_len"], cfg["decode_steps"])


@pytest.mark.parametrize("mode", [1, 2])
def test_tiny_multikernel_modes_bit_identical_to_persistent(torch_cuda, mode):
    cfg = synth.get_config("tiny")
    a = _check_case(cfg, 8, 24, mode=0)
    b = _check_case(cfg, 8, 24, mode=mode)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_tiny_temperature_sampling_bit_exact(torch_cuda):
    cfg = synth.get_config("tiny")
    _check_case(cfg, 16, 48, temperature=0.7)


@pytest.mark.parametrize("name", ["dense-2.3b-fp16", "dense-8b-bf16", "moe-32x1408-top4-e4m3", "dense-2.3b-e4m3",
                                  "dense-2.3b-nvfp4", "dense-8b-e4m3", "dense-8b-nvfp4"])
def test_shrunk_workloads_bit_exact(torch_cuda, name):
    cfg = synth.shrink(synth.get_config(name))
    _check_case(cfg, 8, 40)


def test_nvfp4_rows_split_into_several_chunks(torch_cuda):
    """NVFP4 at the 2.3B model's widths (one layer, small vocabulary): the FFN down projection's
    9728-long rows stream as several K-chunks with a ragged last one, each tile carrying its rows'
    codes and then their block scales."""
    cfg = synth.shrink(synth.get_config("dense-2.3b-nvfp4"), n_layers=1, d_model=2560, d_ff=9728)
    _check_case(cfg, 6, 10)


def test_nvfp4_widths_must_be_multiples_of_128(torch_cuda):
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.shrink(synth.get_config("dense-2.3b-nvfp4"))
    W = synth.model_weights(cfg)
    bad = dict(cfg, d_ff=704)
    with pytest.raises(adp.AdpError) as e:
        _model(bad, synth.model_weights(bad))
    assert e.value.code == adp.ADP_ERR_UNSUPPORTED_CONFIG
    W["layers"][0]["wq_bscale"] = None
    with pytest.raises(adp.AdpError) as e:
        _model(cfg, W)
    assert e.value.code == adp.ADP_ERR_INVALID_ARG


def test_mha_and_single_kv_head_variants(torch_cuda):
    _check_case(synth.shrink(synth.get_config("tiny"), n_kv_heads=4, n_heads=4), 8, 20)
    _check_case(synth.shrink(synth.get_config("tiny"), n_kv_heads=1, n_heads=6), 40, 60)


def test_head_dim_128_ragged_ffn(torch_cuda):
    cfg = synth.shrink(synth.get_config("tiny"), head_dim=128, n_heads=4, n_kv_heads=2, d_model=384, d_ff=1000)
    _check_case(cfg, 5, 30)


def test_prefill_matches_step_by_step(torch_cuda):
    import torch
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg)
    model = _model(cfg, W)
    kv1 = model.new_kv()
    lg1 = torch.empty(cfg["vocab"], device=model.device)
    n1 = kv1.prefill(prompt, logits=lg1)
    kv2 = model.new_kv()
    lg2 = torch.empty(cfg["vocab"], device=model.device)
    for t in prompt:
        n2 = kv2.step(int(t), logits=lg2)
    assert n1 == n2 and torch.equal(lg1, lg2)
    assert all(np.array_equal(a, b) for a, b in zip(kv1.read(), kv2.read()))
    assert len(kv1) == len(prompt)


def test_generate_async_matches_steps(torch_cuda):
    import torch
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    model = _model(cfg, W)
    prompt = synth.prompt(cfg)
    kv1 = model.new_kv()
    t = kv1.prefill(prompt)
    out = torch.empty(40, dtype=torch.int32, device=model.device)
    kv1.generate_async(t, 40, out)
    from autoregressive_decode_persistent_gb300 import adp
    adp.adp_sync(model.handle)
    kv2 = model.new_kv()
    t2 = kv2.prefill(prompt)
    steps = []
    for _ in range(40):
        t2 = kv2.step(t2)
        steps.append(t2)
    assert out.cpu().tolist() == steps
    assert all(np.array_equal(a, b) for a, b in zip(kv1.read(), kv2.read()))


def test_kv_checkpoint_round_trip(torch_cuda):
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    model = _model(cfg, W)
    prompt = synth.prompt(cfg)
    kv = model.new_kv()
    t = kv.prefill(prompt)
    k, v = kv.read()
    cont = [kv.step(t)]
    kv2 = model.new_kv()
    kv2.load(k, v)
    assert kv2.step(t) == cont[0]
    assert all(np.array_equal(a, b) for a, b in zip(kv.read(), kv2.read()))


def test_context_overflow_is_an_error(torch_cuda):
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.shrink(synth.get_config("tiny"), max_ctx=4)
    model = _model(cfg, synth.model_weights(cfg))
    kv = model.new_kv()
    for t in range(4):
        kv.step(t)
    with pytest.raises(adp.AdpError) as e:
        kv.step(1)
    assert e.value.code == adp.ADP_ERR_CONTEXT_OVERFLOW


def test_dependency_timeout_is_reported_and_recoverable(torch_cuda):
    """One CTA withholds its outputs of one phase: every CTA waiting for them gives up after 1 ms
    and the step returns ADP_ERR_BARRIER_TIMEOUT (no hang, no fault); the error is sticky until
    adp_reset, after which the model computes correctly again."""
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    model = _model(cfg, W)
    kv = model.new_kv()
    adp.adp_debug_set_wait_limit(model.handle, 1_000_000)
    adp.adp_debug_skip_publication(model.handle, 3, 2)  # CTA 3, the Wo phase of layer 0
    with pytest.raises(adp.AdpError) as e:
        kv.step(5)
    assert e.value.code == adp.ADP_ERR_BARRIER_TIMEOUT
    with pytest.raises(adp.AdpError) as e2:
        kv.step(5)
    assert e2.value.code == adp.ADP_ERR_BARRIER_TIMEOUT
    adp.adp_reset(model.handle)
    adp.adp_debug_set_wait_limit(model.handle, 200_000_000)
    kv.reset()
    lg = torch.empty(cfg["vocab"], device=model.device)
    kv.step(5, logits=lg)
    model2 = _model(cfg, W)
    kv2 = model2.new_kv()
    lg2 = torch.empty(cfg["vocab"], device=model2.device)
    kv2.step(5, logits=lg2)
    assert torch.equal(lg, lg2)


def test_moe_forced_experts_match_oracle(torch_cuda):
    cfg = synth.shrink(synth.get_config("moe-32x1408-top4-e4m3"))
    W = synth.model_weights(cfg)
    from oracle import OracleModel
    from autoregressive_decode_persistent_gb300 import adp
    import torch
    rng = np.random.default_rng(0)
    force = np.stack([rng.permutation(cfg["n_experts"])[: cfg["top_k"]] for _ in range(cfg["n_layers"])]).astype(
        np.int32)
    om = OracleModel(cfg, W)
    om_p = OracleModel(cfg, W)
    model = _model(cfg, W)
    adp.adp_debug_force_experts(model.handle, force)
    kv = model.new_kv()
    lg = torch.empty(cfg["vocab"], device=model.device)
    for t in synth.prompt(cfg, 6):
        ref = om.step(int(t), EXACT, force=force)
        ref_p = om_p.step(int(t), PLAIN, force=force)
        nxt = kv.step(int(t), logits=lg)
        assert nxt == ref["next"]
        got = lg.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref["logits"].view(np.uint32))
        assert_logits_within_tolerance(got[None], ref_p["logits"][None].astype(np.float64))


@pytest.mark.parametrize("name,temperature", [("tiny", 0.7), ("moe-32x1408-top4-e4m3", 0.0),
                                              ("dense-8b-bf16", 0.0), ("dense-2.3b-e4m3", 0.0),
                                              ("dense-2.3b-nvfp4", 0.7)])
def test_in_kernel_multi_step_generation_matches_oracle(torch_cuda, name, temperature):
    """adp_generate_async runs n decode steps in one persistent launch, each step taking the token
    the previous one chose (and, at T > 0, the next uniform): the tokens and the whole KV cache
    equal the oracle's free run in contract mode.  One more step on that cache (through
    adp_decode_step) gives logits within the stated tolerances of the plain oracle run on the same
    tokens."""
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config(name) if name == "tiny" else synth.shrink(synth.get_config(name))
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg, 6)
    n = 30
    us = synth.sampling_uniforms(len(prompt) + n) if temperature > 0 else None
    toks, _, nexts, _, om = oracle_free_run(cfg, W, prompt, n, EXACT, temperature, us)
    model = _model(cfg, W)
    kv = model.new_kv()
    t0 = kv.prefill(prompt[:-1]) if len(prompt) > 1 else None
    assert t0 == nexts[len(prompt) - 2] or temperature > 0
    out = torch.empty(n + 1, dtype=torch.int32, device=model.device)
    dev_u = torch.tensor(us[len(prompt) - 1:], dtype=torch.float32, device=model.device) if us is not None else None
    kv.generate_async(int(prompt[-1]), n + 1, out, temperature, dev_u)
    adp.adp_sync(model.handle)
    assert out.cpu().tolist() == nexts[len(prompt) - 1:len(prompt) + n]
    k, v = kv.read()
    m = len(prompt) + n
    assert np.array_equal(k[:, :, :m], om.kc[:, :, :m]) and np.array_equal(v[:, :, :m], om.vc[:, :, :m])
    lg = torch.empty(cfg["vocab"], device=model.device)
    kv.step(nexts[-1], logits=lg)
    ref_p, _, _ = oracle_forced(cfg, W, toks + [nexts[-1]], PLAIN)
    assert_logits_within_tolerance(lg.cpu().numpy()[None], ref_p[-1:])
    model.close()


def test_epoch_counter_restarts_before_it_would_wrap(torch_cuda):
    """Started two steps short of 2^32 epochs, the engine zeroes its exchange buffers and restarts
    the counter before the step that would run past it: tokens and logits equal a fresh model's,
    for single steps and for a multi-step launch."""
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    a, b = _model(cfg, W), _model(cfg, W)
    kva, kvb = a.new_kv(), b.new_kv()
    nph = 2 * 5 + 2  # tiny: five phases per layer, then the LM head and sampling
    # restart at the third single step; right away; before the multi-step launch
    for base in (2**32 - 4 * nph, 2**32 - 7, 2**32 - 10 * nph):
        adp.adp_debug_set_epoch_base(a.handle, base)
        kva.reset()
        kvb.reset()
        lga = torch.empty(cfg["vocab"], device=a.device)
        lgb = torch.empty(cfg["vocab"], device=b.device)
        ta = tb = 3
        for _ in range(4):
            ta = kva.step(ta, logits=lga)
            tb = kvb.step(tb, logits=lgb)
            assert ta == tb and torch.equal(lga, lgb)
        oa = torch.empty(12, dtype=torch.int32, device=a.device)
        ob = torch.empty(12, dtype=torch.int32, device=b.device)
        kva.generate_async(ta, 12, oa)
        kvb.generate_async(tb, 12, ob)
        adp.adp_sync(a.handle)
        adp.adp_sync(b.handle)
        assert oa.cpu().tolist() == ob.cpu().tolist()
    a.close()
    b.close()


def test_model_destroyed_before_its_caches(torch_cuda):
    """A model may go before its caches: they are orphaned, accept only adp_kv_destroy, and
    reject every other call."""
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config("tiny")
    model = _model(cfg, synth.model_weights(cfg))
    kv = model.new_kv()
    kv.step(3)
    h = kv.handle
    model.close()
    with pytest.raises(adp.AdpError) as e:
        adp.adp_kv_reset(h)
    assert e.value.code == adp.ADP_ERR_INVALID_ARG
    kv.close()


@pytest.mark.parametrize("name", ["tiny", "dense-2.3b-nvfp4", "moe-32x1408-top4-e4m3"])
def test_host_plan_is_the_models_plan(torch_cuda, name):
    """adp_plan on the host, for this GPU's SM count, gives the weight image and phase list the
    created model streams."""
    from autoregressive_decode_persistent_gb300 import adp
    from autoregressive_decode_persistent_gb300.model import make_config
    cfg = synth.get_config(name) if name == "tiny" else synth.shrink(synth.get_config(name))
    model = _model(cfg, synth.model_weights(cfg), mode=1)
    ph, img = adp.adp_plan(make_config(cfg), model.num_ctas)
    assert img == model.image_bytes
    assert len(ph) - 1 == model.launches_per_step  # one launch per phase but the last (sampling)
    model.close()
