"""Small-batch decode (adp_decode_batch, adp_generate_batch_async) against the CPU oracle.

A batch is nb independent requests, each with its own prompt, KV cache and position; the oracle
runs each request alone.  Per request the engine's batched step follows the same arithmetic
contract as the single-request step, so the bar is the single-request one: logits, chosen tokens
and KV rows bit-exact against the oracle's EXACT mode, and the logits within the stated
tolerances of its PLAIN mode.  Prompt lengths are ragged and cross attention-block boundaries
(32 positions), so the requests' attention item counts differ within a step."""
import numpy as np
import pytest

import synth
from oracle import EXACT, PLAIN, OracleModel

from gpu_common import assert_logits_within_tolerance, oracle_free_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "a CUDA GPU is required"
    from autoregressive_decode_persistent_gb300 import build
    build.build()
    return torch


def _model(cfg, W):
    from autoregressive_decode_persistent_gb300.model import DecodeModel
    return DecodeModel(cfg, W)


def _check_batch(cfg, lengths, n_decode, temperatures=None, plain=True):
    """Oracle free run per request; the engine prefills each request alone (single-request
    path), then decodes all of them together, teacher-forced on the oracle's tokens."""
    import torch
    nb = len(lengths)
    W = synth.model_weights(cfg)
    prompts = synth.batch_prompts(cfg, lengths)
    temps = temperatures or [0.0] * nb
    runs = []
    for r in range(nb):
        us = synth.batch_uniforms(lengths[r] + n_decode, r) if temps[r] > 0 else None
        runs.append(oracle_free_run(cfg, W, prompts[r], n_decode, EXACT, temps[r], us) + (us,))
    model = _model(cfg, W)
    assert model.max_batch >= nb
    kvs = [model.new_kv() for _ in range(nb)]
    for r in range(nb):
        if lengths[r] > 1:
            kvs[r].prefill(prompts[r][:-1])
    lg = torch.empty((nb, cfg["vocab"]), dtype=torch.float32, device=model.device)
    for i in range(n_decode + 1):
        toks, us = [], []
        for r in range(nb):
            k = lengths[r] - 1 + i
            toks.append(runs[r][0][k])
            us.append(float(runs[r][5][k]) if runs[r][5] is not None else 0.0)
        nxt = model.step_batch(kvs, toks, temps if temperatures else None, us, lg)
        got = lg.cpu().numpy()
        for r in range(nb):
            k = lengths[r] - 1 + i
            toks_r, logits_r, nexts_r = runs[r][0], runs[r][1], runs[r][2]
            assert nxt[r] == nexts_r[k], (r, i)
            assert np.array_equal(got[r].view(np.uint32), logits_r[k].view(np.uint32)), (r, i)
    for r in range(nb):
        om = runs[r][4]
        n = lengths[r] + n_decode
        k, v = kvs[r].read()
        assert len(kvs[r]) == n
        assert np.array_equal(k, om.kc[:, :, :n]) and np.array_equal(v, om.vc[:, :, :n]), r
    if plain:
        # the last batched step of every request against the textbook fp32 oracle
        for r in range(nb):
            toks_r = runs[r][0]
            us = runs[r][5]
            pm = OracleModel(cfg, W)
            out = None
            for j, t in enumerate(toks_r):
                out = pm.step(int(t), PLAIN, temperature=temps[r], u=float(us[j]) if us is not None else 0.0)
            assert_logits_within_tolerance(lg.cpu().numpy()[r:r + 1], out["logits"][None].astype(np.float64))
    for kv in kvs:
        kv.close()
    model.close()


@pytest.mark.parametrize("lengths", [[5, 12], [33, 1, 20], [40, 7, 32, 17]])
def test_tiny_batches_bit_exact(torch_cuda, lengths):
    _check_batch(synth.get_config("tiny"), lengths, 12)


def test_tiny_batch_mixes_greedy_and_sampled_requests(torch_cuda):
    _check_batch(synth.get_config("tiny"), [9, 30, 3], 16, temperatures=[0.7, 0.0, 0.7])


@pytest.mark.parametrize("name", ["dense-2.3b-fp16", "dense-8b-bf16", "dense-2.3b-e4m3", "dense-2.3b-nvfp4",
                                  "dense-8b-nvfp4"])
def test_shrunk_workloads_batch_bit_exact(torch_cuda, name):
    cfg = synth.shrink(synth.get_config(name))
    _check_batch(cfg, [8, 35], 10)


def test_single_request_batch_equals_decode_step(torch_cuda):
    """nb = 1 through the batched kernel gives the single-request kernel's logits and KV rows."""
    import torch
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    model = _model(cfg, W)
    prompt = synth.prompt(cfg, 10)
    a, b = model.new_kv(), model.new_kv()
    ta = a.prefill(prompt)
    tb = b.prefill(prompt)
    la = torch.empty(cfg["vocab"], device=model.device)
    lb = torch.empty((1, cfg["vocab"]), device=model.device)
    for _ in range(8):
        ta = a.step(ta, logits=la)
        tb = model.step_batch([b], [tb], logits=lb)[0]
        assert ta == tb and torch.equal(la, lb[0])
    assert all(np.array_equal(x, y) for x, y in zip(a.read(), b.read()))
    model.close()


@pytest.mark.parametrize("name", ["tiny", "dense-8b-bf16"])
def test_generate_batch_in_one_launch_matches_oracle(torch_cuda, name):
    """n batched steps in one persistent launch, each request feeding itself its chosen token:
    the tokens [n][nb] and every cache equal the oracle's free runs."""
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config(name) if name == "tiny" else synth.shrink(synth.get_config(name))
    W = synth.model_weights(cfg)
    lengths = [6, 34, 13]
    nb, n = len(lengths), 24
    prompts = synth.batch_prompts(cfg, lengths)
    runs = [oracle_free_run(cfg, W, prompts[r], n, EXACT) for r in range(nb)]
    model = _model(cfg, W)
    kvs = [model.new_kv() for _ in range(nb)]
    for r in range(nb):
        kvs[r].prefill(prompts[r][:-1])
    out = torch.empty((n + 1, nb), dtype=torch.int32, device=model.device)
    model.generate_batch_async(kvs, [int(p[-1]) for p in prompts], n + 1, out)
    adp.adp_sync(model.handle)
    got = out.cpu().numpy()
    for r in range(nb):
        L = lengths[r]
        assert got[:, r].tolist() == runs[r][2][L - 1:L + n], r
        k, v = kvs[r].read()
        om = runs[r][4]
        m = L + n
        assert np.array_equal(k[:, :, :m], om.kc[:, :, :m]) and np.array_equal(v[:, :, :m], om.vc[:, :, :m]), r
    model.close()


def test_batched_and_single_steps_interleave(torch_cuda):
    """Single-request steps and batched steps on the same model share one epoch counter; taking
    turns they stay bit-identical to a model that only runs single steps."""
    import torch
    cfg = synth.get_config("tiny")
    W = synth.model_weights(cfg)
    a, b = _model(cfg, W), _model(cfg, W)
    pa = synth.batch_prompts(cfg, [7, 21])
    kva = [a.new_kv() for _ in pa]
    kvb = [b.new_kv() for _ in pa]
    ta = [kva[r].prefill(pa[r]) for r in range(2)]
    tb = [kvb[r].prefill(pa[r]) for r in range(2)]
    for i in range(6):
        if i % 2:
            ta = a.step_batch(kva, ta)
        else:
            ta = [kva[r].step(ta[r]) for r in range(2)]
        tb = [kvb[r].step(tb[r]) for r in range(2)]
        assert ta == tb
    for r in range(2):
        assert all(np.array_equal(x, y) for x, y in zip(kva[r].read(), kvb[r].read()))
    a.close()
    b.close()


def test_batch_rejections(torch_cuda):
    from autoregressive_decode_persistent_gb300 import adp
    cfg = synth.get_config("tiny")
    model = _model(cfg, synth.model_weights(cfg))
    nbmax = model.max_batch
    assert nbmax == 4
    kvs = [model.new_kv() for _ in range(nbmax + 1)]
    with pytest.raises(adp.AdpError) as e:
        model.step_batch(kvs, [1] * len(kvs))
    assert e.value.code == adp.ADP_ERR_UNSUPPORTED_CONFIG
    with pytest.raises(adp.AdpError) as e:
        model.step_batch([kvs[0], kvs[0]], [1, 2])  # one cache twice
    assert e.value.code == adp.ADP_ERR_INVALID_ARG
    with pytest.raises(adp.AdpError) as e:
        model.step_batch(kvs[:2], [1, cfg["vocab"]])
    assert e.value.code == adp.ADP_ERR_INVALID_ARG
    assert all(len(k) == 0 for k in kvs)
    small = synth.shrink(cfg, max_ctx=3)
    m2 = _model(small, synth.model_weights(small))
    k2 = [m2.new_kv(), m2.new_kv()]
    for _ in range(3):
        m2.step_batch(k2, [1, 2])
    with pytest.raises(adp.AdpError) as e:
        m2.step_batch(k2, [1, 2])
    assert e.value.code == adp.ADP_ERR_CONTEXT_OVERFLOW
    moe = synth.shrink(synth.get_config("moe-32x1408-top4-e4m3"))
    m3 = _model(moe, synth.model_weights(moe))
    assert m3.max_batch == 0
    with pytest.raises(adp.AdpError) as e:
        m3.step_batch([m3.new_kv()], [1])
    assert e.value.code == adp.ADP_ERR_UNSUPPORTED_CONFIG
    for m in (model, m2, m3):
        m.close()
